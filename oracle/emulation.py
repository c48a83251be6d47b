"""CPU emulation of the blocked (online-softmax) forward -- TEST INFRASTRUCTURE ONLY.

Mirrors the arithmetic contract of a tiled FlashAttention forward, not its
instructions: FP32 scores, FP32 running statistics, unnormalised
probabilities rounded to BF16 (round-to-nearest-even) for the P~V product,
FP32 accumulation of O, and a final O = diag(l)^-1 O rounded to BF16.  It
shares no code with the CUDA path; only ``tests/`` and ``bench.py``'s CPU
baseline may use it.

Sources (page title, section):
  * ijyty.com/news/896914 (BF16 FlashAttention stability) §2.1: per key block
        m = max(m_prev, rowmax(S)),  P~ = exp(S - m),
        l = exp(m_prev - m) l_prev + rowsum(P~),
        O = diag(exp(m_prev - m)) O_prev + P~ V,  finally O = diag(l)^-1 O;
    §2.2 / §3.1: a repeated row maximum gives P~ entries of exactly 1.0,
    and BF16 rounds to nearest even; §4.1 the stabilised shift rule;
    §4.2 the rule applied inside the block loop.
  * "Flash Attention低精度训练稳定性优化实践" (jsqmd.com) §3.2: QK^T
    accumulated in FP32, softmax kept in FP32, the product with V in BF16.

Readings where the pages are silent:
  * Blocked tie count (the pages apply the rule to "S" inside the block loop
    but never say how counts combine across blocks): each row keeps a
    running (rm, rs) over all visible columns seen so far.  Per block,
    bm = max of its visible entries and bc = how many equal bm; the merge is
        rm' = max(rm, bm),  rs' = [rm == rm'] rs + [bm == rm'] bc,
    starting from (-inf, 0).  After each block the shift is the rule applied
    to (rm', rs').  The final (rm, rs, branch) then equals the rule applied
    to the whole row, whatever the block width.  With this reading the
    shift may decrease from one block to the next, so the correction factor
    exp(scale (m_prev - m)) can exceed 1.
  * ``stable == 2`` is the other, block-local reading of §4.2:
    m_j = max(m_{j-1}, rule(rowmax S_j, count in S_j)); it depends on the
    block width.
  * l accumulates the FP32 P~ (before the BF16 cast): the softmax stays in
    FP32 and only the product with V is cast.  Across blocks it is a Kahan
    (compensated) sum by default, the summation the same page (§7.2) recommends
    for the softmax denominator of large models.
  * FP8 forward (same page, §6.1: the shift carries over to FP8 with dynamic
    scaling): P~ is multiplied by 2^8 and rounded to E4M3 (nearest, ties to
    even) for the P~V product; l still sums the FP32 P~.
  * exp is evaluated in FP64 and rounded to FP32 (the GPU's exp is not
    reproduced bit for bit; results are compared within tolerances, and the
    exact-1.0 counts only where the margin to the BF16 rounding boundary is
    far larger than any exp error).

Parity status: pinned in ``tests/test_emulation_pins.py`` -- in FP64 mode the
blocked recurrence equals the one-shot oracle for every block width; the
running tie state equals the whole-row state; plain mode produces exact-1.0
entries at repeated maxima and stable mode removes them; on rows whose block
sums fall below half an ulp of l, the uncompensated FP32 row sum drifts by the
lost sums while the compensated one stays at the FP64 closed form.
"""
from __future__ import annotations

import numpy as np

from .attention import BRANCH_BETA, BRANCH_RM, BRANCH_ZERO, _f64, visible
from .fp8 import P_SCALE_LOG2, decode_e4m3, encode_e4m3

BF16_ONE_BITS = 0x3F80


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to the nearest BF16 (ties to even); returns FP32 holding BF16 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    out = r.view(np.float32).copy()
    nan = np.isnan(x)
    out[nan] = np.nan
    return out


def _rule32(rm, rs, beta32, stable):
    """The stabilised shift in FP32 (beta * rm rounded to FP32)."""
    if not stable:
        return rm.copy(), np.zeros(rm.shape, dtype=np.int8)
    repeated = rs > 1
    pos = repeated & (rm > 0)
    neg = repeated & (rm < 0)
    m = np.where(pos, (beta32 * rm).astype(rm.dtype), np.where(neg, rm.dtype.type(0), rm))
    br = np.where(pos, BRANCH_BETA, np.where(neg, BRANCH_ZERO, BRANCH_RM)).astype(np.int8)
    return m.astype(rm.dtype), br


def blocked_forward(q, k, v, scale: float, causal: bool, stable: int = 0, beta: float = 1.25,
                    block_n: int = 128, precision: str = "bf16", compensated: bool = True):
    """Blocked online-softmax forward over key blocks of width ``block_n``.

    precision="bf16": FP32 state, P~ rounded to BF16 for P~V, O rounded to BF16.
    precision="fp8": the same, but P~ * 2^8 is rounded to E4M3 for P~V (the FP8
    forward; pass the dequantised Q, K, V).
    precision="fp64": the same recurrence with every value in FP64 and no
    rounding (used to pin the recurrence against the one-shot definition).
    compensated: in FP32, the row sum l = alpha l + rowsum(P~) is accumulated across
    blocks with Kahan's compensated summation (ijyty.com §7.2 recommends it for the
    softmax denominator of large models): a compensation c carries the low-order part
    each update loses, scaled by alpha with the sum, and the final row sum is l - c.
    With compensated=False the update is the plain FP32 recurrence.

    Returns dict(o, lse, rm, rs, branch, m, ones) per [B, H, N]; ``ones`` is
    the number of visible P~ entries of a row whose rounded value (BF16, or
    E4M3 of P~ * 2^8 divided by 2^8) is exactly 1.0 (counted per block, as the
    blocks are processed).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    if precision not in ("bf16", "fp8", "fp64"):
        raise ValueError(precision)
    low = precision != "fp64"
    ft = np.float32 if low else np.float64
    beta_t = ft(beta)
    res = {key: np.zeros((B, H, N), dtype=ft) for key in ("lse", "rm", "m")}
    res["o"] = np.zeros((B, H, N, dv), dtype=ft)
    res["rs"] = np.zeros((B, H, N), dtype=np.int64)
    res["branch"] = np.zeros((B, H, N), dtype=np.int8)
    res["ones"] = np.zeros((B, H, N), dtype=np.int64)
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            rm = np.full(N, -np.inf, dtype=ft)
            rs = np.zeros(N, dtype=np.int64)
            m = np.full(N, -np.inf, dtype=ft)
            l = np.zeros(N, dtype=ft)
            lc = np.zeros(N, dtype=ft)          # Kahan compensation of l (FP32 paths)
            acc = np.zeros((N, dv), dtype=ft)
            ones = np.zeros(N, dtype=np.int64)
            br = np.zeros(N, dtype=np.int8)
            for j0 in range(0, N, block_n):
                cols = np.arange(j0, min(N, j0 + block_n))
                vis = visible(rows, N, causal)[:, cols]
                s = (q[b, h] @ k[b, h, cols].T).astype(ft)          # FP32 scores
                sm = np.where(vis, s, ft(-np.inf))
                bm = sm.max(axis=1)
                bc = ((sm == bm[:, None]) & vis).sum(axis=1)
                bc = np.where(np.isneginf(bm), 0, bc)
                if stable == 2:
                    mb, brb = _rule32(bm, bc, beta_t, 1)
                    m_new = np.maximum(m, mb)
                    br = np.where(mb >= m, brb, br)  # branch of the block that set the shift
                    rm_new = np.maximum(rm, bm)
                    rs = np.where(rm == rm_new, rs, 0) + np.where(bm == rm_new, bc, 0)
                    rm = rm_new
                else:
                    rm_new = np.maximum(rm, bm)
                    rs = np.where(rm == rm_new, rs, 0) + np.where(bm == rm_new, bc, 0)
                    rm = rm_new
                    m_new, br = _rule32(rm, rs, beta_t, stable)
                with np.errstate(invalid="ignore"):
                    alpha = np.where(np.isneginf(m), 0.0,
                                     np.exp(scale * (m.astype(np.float64) - m_new.astype(np.float64)))).astype(ft)
                live = ~np.isneginf(m_new)
                e64 = np.where(vis & live[:, None],
                               np.exp(scale * (s.astype(np.float64) - np.where(live, m_new, 0.0)[:, None].astype(np.float64))),
                               0.0)
                p = e64.astype(ft)
                if low:
                    if precision == "bf16":
                        pb = round_bf16(p)
                    else:
                        ps = np.float32(2.0 ** P_SCALE_LOG2)
                        pb = (decode_e4m3(encode_e4m3((p * ps).astype(np.float32))) / float(ps)).astype(np.float32)
                    ones += ((pb == np.float32(1.0)) & vis).sum(axis=1)
                    rowsum = p.sum(axis=1, dtype=np.float32)
                    ls = (alpha * l).astype(ft)
                    if compensated:
                        y = (rowsum - (alpha * lc).astype(ft)).astype(ft)
                        t = (ls + y).astype(ft)
                        lc = ((t - ls).astype(ft) - y).astype(ft)
                        l = t
                    else:
                        l = (ls + rowsum).astype(ft)
                    pv = (pb.astype(np.float64) @ v[b, h, cols]).astype(ft)
                    acc = (alpha[:, None] * acc).astype(ft) + pv
                else:
                    ones += ((p == 1.0) & vis).sum(axis=1)
                    l = alpha * l + p.sum(axis=1)
                    acc = alpha[:, None] * acc + p @ v[b, h, cols]
                m = m_new
            if low:
                l = (l - lc).astype(ft)
            o = acc / l[:, None]
            if low:
                o = round_bf16(o.astype(np.float32))
                lse = (ft(scale) * m).astype(ft) + np.log(l.astype(np.float64)).astype(ft)
            else:
                lse = scale * m + np.log(l)
            res["o"][b, h] = o
            res["lse"][b, h] = lse
            res["rm"][b, h] = rm
            res["rs"][b, h] = rs
            res["branch"][b, h] = br
            res["m"][b, h] = m
            res["ones"][b, h] = ones
    return res
