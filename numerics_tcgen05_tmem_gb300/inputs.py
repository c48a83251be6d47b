"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and quantises them to bfloat16; it
holds none of the attention arithmetic.  Both the CPU oracle tests and the
CUDA path take their inputs from here, so the two see the same bits.

Every tensor is returned as a CPU ``torch.bfloat16`` tensor in the
contiguous ``[B, H, N, d]`` layout.  Values are drawn in float32 with a
``numpy.random.Generator`` (PCG64) seeded per workload and rounded to
bfloat16 (round-to-nearest-even) by ``torch``'s CPU conversion.

The workloads follow the shapes and value distributions the stability pages
discuss: a tiny dyadic case with planted tied row maxima (the failure
trigger of "Why Low-Precision Transformer Training Fails", as summarised on
the page "為什么BF16的FlashAttention會把訓練「炸掉」？"), GPT-2 small/medium
attention shapes, an attention-sink case with repeated keys, a LLaMA-7B
shaped long sequence and a 16k-token stress case.  No dataset item is used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BASE_SEED = 20261202


@dataclass
class Workload:
    """A seeded attention problem: inputs plus the call parameters."""

    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    causal: bool
    scale: float
    stable: int
    beta: float
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return tuple(self.q.shape)


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def tiny_ties(seed_offset: int = 0, B: int = 1, H: int = 2, N: int = 128, d: int = 64,
              stable: int = 1, beta: float = 1.25) -> Workload:
    """Dyadic inputs with planted repeated row maxima.

    Q, K, V are uniform on {k/8 : k in [-16, 16]}, so every product q*k is a
    multiple of 1/64 and every FP32 partial sum of a dot product is exact.
    About 10% of the key rows of each head are copies of other key rows, so
    rows whose maximum falls on a copied key see the maximum more than once.
    Three planted rows make both signs certain:
      * key rows 1 and 2 are copies of key row 0;
      * query row 1 (sees keys 0, 1) is sign-adjusted so its tied maximum is
        <= -1 in raw units (scaled <= -1/8): the negative-maximum case;
      * query row 2 (sees keys 0, 1, 2) is sign-adjusted so its tied
        maximum is >= +1 in raw units: the positive case.
    dO is N(0, 1) rounded to bf16.
    """
    rng = np.random.default_rng(BASE_SEED + 0 + 1000 * seed_offset)
    grid = lambda shape: (rng.integers(-16, 17, size=shape).astype(np.float32) / 8.0)
    q = grid((B, H, N, d))
    k = grid((B, H, N, d))
    v = grid((B, H, N, d))
    n_dup = max(1, int(round(0.10 * N))) if N > 3 else 0
    for b in range(B):
        for h in range(H):
            if n_dup:
                dst = rng.choice(np.arange(3, N), size=min(n_dup, N - 3), replace=False) if N > 3 else []
                for t in dst:
                    src = int(rng.integers(0, N - 1))
                    if src >= t:
                        src += 1
                    k[b, h, t] = k[b, h, src]
            if N >= 3:
                # make sure key row 0 is not all zero, so planted dot products can be made nonzero
                if not np.any(k[b, h, 0]):
                    k[b, h, 0, 0] = 1.0
                k[b, h, 1] = k[b, h, 0]
                k[b, h, 2] = k[b, h, 0]
                for row, sign in ((1, -1.0), (2, +1.0)):
                    dot = float(np.dot(q[b, h, row].astype(np.float64), k[b, h, 0].astype(np.float64)))
                    if dot == 0.0 or abs(dot) < 1.0:
                        # push the dot product away from zero along key 0's largest channel
                        c = int(np.argmax(np.abs(k[b, h, 0])))
                        q[b, h, row, c] = np.float32(2.0 * np.sign(k[b, h, 0, c]))
                        dot = float(np.dot(q[b, h, row].astype(np.float64), k[b, h, 0].astype(np.float64)))
                    if abs(dot) < 1.0:
                        q[b, h, row] = k[b, h, 0]
                        dot = float(np.dot(q[b, h, row].astype(np.float64), k[b, h, 0].astype(np.float64)))
                    if np.sign(dot) != sign:
                        q[b, h, row] = -q[b, h, row]
    do = _normal(rng, (B, H, N, d))
    return Workload("tiny_ties", _bf16(q), _bf16(k), _bf16(v), _bf16(do), True, 1.0 / 8.0,
                    stable, beta, {"B": B, "H": H, "N": N, "d": d})


def gpt2_small(B: int = 8, H: int = 12, N: int = 1024, d: int = 64, stable: int = 1,
               beta: float = 1.25) -> Workload:
    """GPT-2-small attention: Q, K ~ N(0,1)*sqrt(3) so the scaled logit std is 3."""
    rng = np.random.default_rng(BASE_SEED + 1)
    s = 1.0 / math.sqrt(d)
    sig = math.sqrt(3.0)
    q = _normal(rng, (B, H, N, d), sig)
    k = _normal(rng, (B, H, N, d), sig)
    v = _normal(rng, (B, H, N, d))
    do = _normal(rng, (B, H, N, d))
    return Workload("gpt2_small", _bf16(q), _bf16(k), _bf16(v), _bf16(do), True, s, stable, beta,
                    {"B": B, "H": H, "N": N, "d": d, "logit_std": 3.0})


def gpt2_medium_sink(B: int = 16, H: int = 16, N: int = 1024, d: int = 64, stable: int = 1,
                     beta: float = 1.25, sink_frac: float = 0.05, bias: float = 4.0) -> Workload:
    """GPT-2-medium attention with an attention sink.

    Channel 0 is reserved: every query has q[..., 0] = 1 and key 0 plus its
    copies get k[..., 0] = bias / scale (other keys 0), so their logit carries
    an exact +bias.  Key 0 (all channels) is copied to sink_frac of the
    positions, so each query sees the sink key several times with bit-identical
    logits: a repeated row maximum.
    """
    rng = np.random.default_rng(BASE_SEED + 2)
    s = 1.0 / math.sqrt(d)
    q = _normal(rng, (B, H, N, d))
    k = _normal(rng, (B, H, N, d))
    v = _normal(rng, (B, H, N, d))
    do = _normal(rng, (B, H, N, d))
    n_copy = int(round(sink_frac * N))
    q[..., 0] = 1.0
    k[..., 0] = 0.0
    for b in range(B):
        pos = rng.choice(np.arange(1, N), size=min(n_copy, N - 1), replace=False) if N > 1 else []
        for h in range(H):
            k[b, h, 0, 0] = np.float32(bias / s)
            for p in pos:
                k[b, h, p] = k[b, h, 0]
    return Workload("gpt2_medium_sink", _bf16(q), _bf16(k), _bf16(v), _bf16(do), True, s, stable, beta,
                    {"B": B, "H": H, "N": N, "d": d, "sink_copies": n_copy, "bias": bias})


def llama7b_long(B: int = 1, H: int = 32, N: int = 8192, d: int = 128, stable: int = 1,
                 beta: float = 1.25, heads=None) -> Workload:
    """LLaMA-7B shaped attention: Q, K, V ~ N(0,1)/sqrt(2), one outlier channel x8.

    "1% outlier channels" of d=128 rounds to one channel; the same seeded
    channel index is scaled by 8 in Q, K and V.  ``heads`` draws only the
    listed heads (the same values those heads get in the full draw), so the
    oracle can check a subset of a large problem.
    """
    rng = np.random.default_rng(BASE_SEED + 3)
    s = 1.0 / math.sqrt(d)
    ch = int(rng.integers(0, d))
    return _per_head_draw("llama7b_long", rng, B, H, N, d, True, s, stable, beta, heads,
                          qk_std=1.0 / math.sqrt(2.0), v_std=1.0 / math.sqrt(2.0), outlier=(ch, 8.0))


def extreme_16k(B: int = 1, H: int = 16, N: int = 16384, d: int = 128, causal: bool = True,
                stable: int = 1, beta: float = 1.25, heads=None) -> Workload:
    """16k tokens, Q, K ~ N(0,1)*sqrt(5) (scaled logit std 5); V, dO ~ N(0,1)."""
    rng = np.random.default_rng(BASE_SEED + 4)
    s = 1.0 / math.sqrt(d)
    return _per_head_draw("extreme_16k" + ("" if causal else "_noncausal"), rng, B, H, N, d, causal, s,
                          stable, beta, heads, qk_std=math.sqrt(5.0), v_std=1.0, outlier=None)


def _per_head_draw(name, rng, B, H, N, d, causal, s, stable, beta, heads, qk_std, v_std, outlier):
    """Draw each (b, h) from its own child seed so any subset of heads is reproducible."""
    sel = [(b, h) for b in range(B) for h in range(H)]
    if heads is not None:
        sel = [sel[i] for i in heads]
    seeds = rng.integers(0, 2**63 - 1, size=B * H)
    shape = (len(sel), N, d)
    q = np.empty(shape, np.float32)
    k = np.empty(shape, np.float32)
    v = np.empty(shape, np.float32)
    do = np.empty(shape, np.float32)
    for t, (b, h) in enumerate(sel):
        r = np.random.default_rng(int(seeds[b * H + h]))
        q[t] = _normal(r, (N, d), qk_std)
        k[t] = _normal(r, (N, d), qk_std)
        v[t] = _normal(r, (N, d), v_std)
        do[t] = _normal(r, (N, d))
        if outlier is not None:
            c, f = outlier
            q[t, :, c] *= f
            k[t, :, c] *= f
            v[t, :, c] *= f
    if heads is None:
        shp = (B, H, N, d)
    else:
        shp = (1, len(sel), N, d)
    meta = {"B": B, "H": H, "N": N, "d": d, "heads": None if heads is None else list(heads)}
    if outlier is not None:
        meta["outlier_channel"] = outlier[0]
    return Workload(name, _bf16(q.reshape(shp)), _bf16(k.reshape(shp)), _bf16(v.reshape(shp)),
                    _bf16(do.reshape(shp)), causal, s, stable, beta, meta)


def random_case(B: int, H: int, N: int, d: int, causal: bool, seed: int, std: float = 1.0,
                stable: int = 1, beta: float = 1.25, scale=None) -> Workload:
    """Plain N(0, std) Q, K, V, dO for edge-case shapes (ragged N, tiny N)."""
    rng = np.random.default_rng(BASE_SEED + 100 + seed)
    s = 1.0 / math.sqrt(d) if scale is None else scale
    q = _normal(rng, (B, H, N, d), std)
    k = _normal(rng, (B, H, N, d), std)
    v = _normal(rng, (B, H, N, d))
    do = _normal(rng, (B, H, N, d))
    return Workload(f"random_B{B}H{H}N{N}d{d}{'c' if causal else 'n'}", _bf16(q), _bf16(k), _bf16(v),
                    _bf16(do), causal, s, stable, beta, {"B": B, "H": H, "N": N, "d": d})


def tiny_tail_rows(N: int = 32768, d: int = 64, H: int = 1, tail_score: float = -178.0) -> Workload:
    """Rows whose softmax denominator is one exact 1.0 plus N - 1 tiny terms.

    Every query row is e_0 (1 in channel 0); key 0 is the zero vector (raw score 0, the
    row's unique maximum) and every other key is tail_score * e_0, so each row sees one
    score 0 and N - 1 scores tail_score.  At d = 64 (scale 1/8) the tiny terms are
    exp(-22.25) ~ 2^-32: a 128-key block of them sums to less than half an FP32 ulp of 1,
    the case that separates a compensated cross-block row sum from a plain one.
    Non-causal; V and dO are N(0, 1), seeded.
    """
    rng = np.random.default_rng(BASE_SEED + 5)
    q = np.zeros((1, H, N, d), dtype=np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, H, N, d), dtype=np.float32)
    k[:, :, 1:, 0] = tail_score
    v = _normal(rng, (1, H, N, d))
    do = _normal(rng, (1, H, N, d))
    return Workload(f"tiny_tail_N{N}d{d}", _bf16(q), _bf16(k), _bf16(v), _bf16(do), False, 1.0 / math.sqrt(d), 1,
                    1.25, {"B": 1, "H": H, "N": N, "d": d})


WORKLOADS = {
    "tiny_ties": tiny_ties,
    "gpt2_small": gpt2_small,
    "gpt2_medium_sink": gpt2_medium_sink,
    "llama7b_long": llama7b_long,
    "extreme_16k": extreme_16k,
}
