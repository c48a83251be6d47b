"""GPU parity of the FP8 path (fa_quantize_fp8, fa_fwd_fp8 through the C ABI) against the oracle.

The E4M3 inputs of every forward test come from the oracle's quantiser (or are exactly
representable dyadic values with unit scales); the GPU quantiser is checked separately,
byte for byte, against the same oracle quantiser.

Tolerances: the GPU rounds P~ * 2^8 to E4M3 (3 mantissa bits) for the P~V product, so O
differs from the FP64 attention of the dequantised inputs by the E4M3 rounding of P~: a
relative error up to 2^-4 per entry, averaged over the keys.  Against the oracle O must be
within 6e-2 (relative Frobenius); against the FP8 blocked emulation, which makes the same
rounding, within 1e-2.  The LSE sums the unrounded FP32 P~ and keeps the BF16 path's 1e-3.
"""
import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from oracle import emulation as E
from oracle import fp8 as F
from tests._parity import assert_lse, f64, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

FP8_REL_TOL = 6e-2
FP8_EMU_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_quantized(w):
    """Oracle quantisation of a workload's Q, K, V: codes (numpy uint8) and descales."""
    out, ds = [], []
    for t in (w.q, w.k, w.v):
        c, s = F.quantize_per_tensor(t.float().numpy())
        out.append(c)
        ds.append(s)
    return out, np.array(ds, dtype=np.float32)


def run_fp8(codes, ds, w, stable, beta=1.25, stats=True):
    q8, k8, v8 = (torch.from_numpy(np.ascontiguousarray(c)).cuda() for c in codes)
    d = torch.from_numpy(ds).cuda()
    out = binding.forward_fp8(q8, k8, v8, d, causal=w.causal, scale=w.scale, stable=stable, beta=beta, stats=stats)
    binding.device_status()
    return out


def dequantized(codes, ds):
    return [F.dequantize(c, s) for c, s in zip(codes, ds)]


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("n", [1, 15, 16, 17, 1000, 3 * 4097, 1 << 20])
def test_quantize_bit_exact(n):
    g = torch.Generator().manual_seed(n)
    x = (torch.randn(n, generator=g) * 3.0).to(torch.bfloat16)
    if n > 20:
        x[7] = 0.0
        x[11] = -1e-40          # a BF16 subnormal
        x[13] = 2.0 ** -126
    want, wds = F.quantize_per_tensor(x.float().numpy())
    x8, ds = binding.quantize_fp8(x.cuda())
    binding.device_status()
    assert ds.item() == float(wds) and ds.cpu().numpy().view(np.uint32)[0] == np.float32(wds).view(np.uint32)
    np.testing.assert_array_equal(x8.cpu().numpy(), want)


def test_quantize_zero_and_constant_tensors():
    z = torch.zeros(4096, dtype=torch.bfloat16)
    x8, ds = binding.quantize_fp8(z.cuda())
    assert ds.item() == 1.0 and not x8.any().item()
    c = torch.full((333,), -2.5, dtype=torch.bfloat16)
    x8, ds = binding.quantize_fp8(c.cuda())
    binding.device_status()
    assert ds.item() == np.float32(2.5) / np.float32(448)
    assert torch.all(x8.cpu() == 0xFE)          # every element is -amax -> -448


def test_quantize_full_size_tensors():
    w = inputs.llama7b_long()
    for t in (w.q, w.v):
        want, wds = F.quantize_per_tensor(t.float().numpy())
        x8, ds = binding.quantize_fp8(t.cuda())
        binding.device_status()
        assert ds.item() == float(wds)
        assert np.array_equal(x8.cpu().numpy(), want)


# ----------------------------------------------------------------- forward

@pytest.mark.parametrize("N", [300, 2048, 2560])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("stable", [0, 1, 2])
def test_tiny_ties_exact_statistics(stable, d, N):
    # k/8 with |k| <= 16 is exact in E4M3 and the dot products are exact in FP32, so with
    # unit scales the row maximum, ties, branch and the exact-1.0 counts are decidable
    # (N = 2048: 16 key blocks, with ties first reached late in the row; at d = 64 rows of up
    # to 2048 keys run one query tile per CTA, longer ones two)
    w = inputs.tiny_ties(d=d, N=N, H=2)
    vals = [t.double().numpy() for t in (w.q, w.k, w.v)]
    codes = [F.encode_e4m3(x) for x in vals]
    assert all(np.array_equal(F.decode_e4m3(c), x) for c, x in zip(codes, vals))
    ones3 = np.ones(3, dtype=np.float32)
    o, lse, st = run_fp8(codes, ones3, w, stable)
    ref = F.forward_fp8(*codes, ones3, w.scale, w.causal, stable=1 if stable == 2 else stable, beta=w.beta)
    em = E.blocked_forward(*vals, w.scale, w.causal, stable=stable, beta=w.beta, block_n=128, precision="fp8")
    assert rel_fro(o, ref["o"]) <= FP8_REL_TOL
    assert rel_fro(o, em["o"]) <= FP8_EMU_TOL
    assert_lse(lse, ref["lse"])
    np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
    np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), em["branch"])
    np.testing.assert_array_equal(st["row_ones"].cpu().numpy(), em["ones"])
    if stable == 0:
        rep = ref["rs"] > 1
        assert np.all(st["row_ones"].cpu().numpy()[rep] >= ref["rs"][rep])
    # the statistics-free kernel decides the same shifts on these tie-heavy rows: identical O
    # and LSE
    o2, lse2 = run_fp8(codes, ones3, w, stable, stats=False)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("N", [1, 100, 128, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_shapes(N, d, causal):
    w = inputs.random_case(2, 2, N, d, causal, seed=N * 13 + d + 5, std=1.5)
    codes, ds = oracle_quantized(w)
    o, lse = run_fp8(codes, ds, w, 1, stats=False)
    deq = dequantized(codes, ds)
    ref = F.forward_fp8(*codes, ds, w.scale, causal, stable=1, beta=w.beta)
    em = E.blocked_forward(*deq, w.scale, causal, stable=1, beta=w.beta, precision="fp8")
    assert rel_fro(o, ref["o"]) <= FP8_REL_TOL
    assert rel_fro(o, em["o"]) <= FP8_EMU_TOL
    assert_lse(lse, ref["lse"])


def test_stats_and_plain_paths_agree():
    w = inputs.random_case(1, 4, 640, 128, True, seed=99, std=1.0)
    codes, ds = oracle_quantized(w)
    for stable in (0, 1, 2):
        o1, l1 = run_fp8(codes, ds, w, stable, stats=False)
        o2, l2, _ = run_fp8(codes, ds, w, stable, stats=True)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sink_ties_take_the_beta_branch():
    # exact +4-logit sink ties survive quantisation (identical key rows stay identical)
    w = inputs.gpt2_medium_sink(B=2, H=2, N=512, d=128)
    codes, ds = oracle_quantized(w)
    o, lse, st = run_fp8(codes, ds, w, 1)
    ref = F.forward_fp8(*codes, ds, w.scale, True, stable=1, beta=1.25)
    assert rel_fro(o, ref["o"]) <= FP8_REL_TOL
    assert_lse(lse, ref["lse"])
    got_br = st["row_branch"].cpu().numpy()
    assert np.mean(got_br == ref["branch"]) > 0.999
    assert (ref["branch"] == 1).sum() > 100


def test_llama7b_full_size_sampled_heads():
    w = inputs.llama7b_long()
    codes, ds = oracle_quantized(w)
    o, lse = run_fp8(codes, ds, w, 1, stats=False)
    heads = [0, 31]
    sub = [c[:, heads] for c in codes]
    ref = F.forward_fp8(*sub, ds, w.scale, True, stable=1, beta=w.beta)
    assert rel_fro(o[:, heads], ref["o"]) <= FP8_REL_TOL
    assert_lse(lse[:, heads], ref["lse"])


def test_nonfinite_descale_is_reported():
    w = inputs.random_case(1, 1, 256, 128, True, seed=5)
    codes, ds = oracle_quantized(w)
    bad = ds.copy()
    bad[2] = np.float32(np.nan)
    q8, k8, v8 = (torch.from_numpy(c).cuda() for c in codes)
    o = torch.empty(q8.shape, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(q8.shape[:3], device="cuda", dtype=torch.float32)
    assert binding.fa_fwd_fp8(q8, k8, v8, torch.from_numpy(bad).cuda(), o, lse, True, w.scale, 1, 1.25) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_WARN_NONFINITE
    assert binding.fa_fwd_fp8(q8, k8, v8, torch.from_numpy(ds).cuda(), o, lse, True, w.scale, 1, 1.25) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_OK


@pytest.mark.parametrize("beta", [1.1, 1.5])
def test_sink_other_betas(beta):
    w = inputs.gpt2_medium_sink(B=1, H=2, N=640, d=128)
    codes, ds = oracle_quantized(w)
    o, lse, st = run_fp8(codes, ds, w, 1, beta=beta)
    ref = F.forward_fp8(*codes, ds, w.scale, True, stable=1, beta=beta)
    assert rel_fro(o, ref["o"]) <= FP8_REL_TOL
    assert_lse(lse, ref["lse"])
    assert np.mean(st["row_branch"].cpu().numpy() == ref["branch"]) > 0.999


def test_extreme_16k_noncausal_sampled_head():
    w = inputs.extreme_16k(causal=False)
    codes, ds = oracle_quantized(w)
    o, lse = run_fp8(codes, ds, w, 1, stats=False)
    sub = [c[:, [7]] for c in codes]
    ref = F.forward_fp8(*sub, ds, w.scale, False, stable=1, beta=w.beta)
    assert rel_fro(o[:, [7]], ref["o"]) <= FP8_REL_TOL
    assert_lse(lse[:, [7]], ref["lse"])


def test_gpt2_small_full():
    # the d = 64 workload in full: E4M3 rows of 64 bytes (64-byte swizzle) and the S ring
    w = inputs.gpt2_small()
    codes, ds = oracle_quantized(w)
    o, lse = run_fp8(codes, ds, w, 1, stats=False)
    ref = F.forward_fp8(*codes, ds, w.scale, True, stable=1, beta=w.beta)
    assert rel_fro(o, ref["o"]) <= FP8_REL_TOL
    assert_lse(lse, ref["lse"])
