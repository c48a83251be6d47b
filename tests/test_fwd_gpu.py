"""GPU parity of the forward (fa_fwd through the C ABI) against the FP64 oracle."""
import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from oracle import attention as A
from oracle import emulation as E
from tests._parity import assert_close_bf16, assert_lse, f64, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_fwd(w, stable, beta=1.25, stats=True):
    q, k, v, _ = to_dev(w)
    out = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=stable, beta=beta, stats=stats)
    binding.device_status()
    return out


@pytest.mark.parametrize("stable", [0, 1])
def test_tiny_ties_bit_exact_stats(stable):
    w = inputs.tiny_ties()
    o, lse, st = run_fwd(w, stable)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=stable, beta=w.beta)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    # dyadic inputs: every FP32 score is exact, so all rows are decidable
    np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
    np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), ref["branch"])
    # exact-1.0 P~ counts equal the BF16 blocked emulation's (128-key blocks)
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=stable, beta=w.beta, block_n=128)
    np.testing.assert_array_equal(st["row_ones"].cpu().numpy(), em["ones"])
    if stable:
        sel = (ref["rs"] > 1) & (ref["rm"] != 0) & (w.scale * np.abs(ref["m"] - ref["rm"]) >= 2.0 ** -7)
        assert sel.sum() > 0 and np.all(st["row_ones"].cpu().numpy()[sel] == 0)
    else:
        rep = ref["rs"] > 1
        assert np.all(st["row_ones"].cpu().numpy()[rep] >= ref["rs"][rep])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("stable", [0, 1])
def test_long_dyadic_rows_exact_statistics(stable, causal, d):
    # 16 key blocks of exact (dyadic) scores with copied key rows: a few hundred rows have a
    # repeated maximum, many of them first reached late in the row.  There the kernel
    # counts ties only in the 32-column chunks that can hold a row's new maximum; the raw
    # maxima, tie counts and branches must still equal the oracle's exactly, and the
    # exact-1.0 counts the BF16 emulation's.
    w0 = inputs.tiny_ties(N=2048, H=2, d=d)
    w = inputs.Workload(w0.name, w0.q, w0.k, w0.v, w0.do, causal, w0.scale, stable, w0.beta)
    o, lse, st = run_fwd(w, stable)
    ref = A.forward(w.q, w.k, w.v, w.scale, causal, stable=stable, beta=w.beta)
    assert (ref["rs"] > 1).sum() > 100
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
    np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), ref["branch"])
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, causal, stable=stable, beta=w.beta, block_n=128)
    np.testing.assert_array_equal(st["row_ones"].cpu().numpy(), em["ones"])
    # the statistics-free kernel decides the same shifts: identical O and LSE
    o2, lse2 = run_fwd(w, stable, stats=False)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("stable", [0, 1])
def test_full_length_dyadic_rows_exact_statistics(stable):
    # the target length (8192 tokens, d = 128, causal) with exact (dyadic) scores and copied
    # key rows: repeated maxima of both signs all along the row; every row is decidable, so
    # the raw maxima, tie counts and branches must equal the oracle's bit for bit and the
    # exact-1.0 counts the BF16 emulation's
    w = inputs.tiny_ties(N=8192, H=2, d=128)
    w = inputs.Workload(w.name, w.q, w.k, w.v, w.do, True, w.scale, stable, w.beta)
    o, lse, st = run_fwd(w, stable)
    ref = A.forward(w.q, w.k, w.v, w.scale, True, stable=stable, beta=w.beta)
    assert (ref["rs"] > 1).sum() > 500
    if stable:
        assert (ref["branch"] == 1).sum() > 500 and (ref["branch"] == 2).sum() >= 1
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
    np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), ref["branch"])
    em = E.blocked_forward(w.q[:, :1], w.k[:, :1], w.v[:, :1], w.scale, True, stable=stable, beta=w.beta,
                           block_n=128)
    np.testing.assert_array_equal(st["row_ones"][:, :1].cpu().numpy(), em["ones"])
    o2, lse2 = run_fwd(w, stable, stats=False)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("N", [2048, 2049, 4096])
@pytest.mark.parametrize("stable", [0, 1, 2])
def test_d64_both_cta_shapes_exact_statistics(N, stable):
    # At d = 64 the forward runs one query tile per CTA (two CTAs per SM) for rows of up to
    # 2048 keys and two tiles per CTA (with a third S buffer) beyond: both shapes must give
    # the oracle's statistics bit for bit on exact (dyadic) scores, causal and not.
    for causal in (True, False):
        w0 = inputs.tiny_ties(N=N, H=2, d=64)
        w = inputs.Workload(w0.name, w0.q, w0.k, w0.v, w0.do, causal, w0.scale, stable, w0.beta)
        o, lse, st = run_fwd(w, stable)
        ref = A.forward(w.q, w.k, w.v, w.scale, causal, stable=1 if stable == 2 else stable, beta=w.beta)
        em = E.blocked_forward(w.q, w.k, w.v, w.scale, causal, stable=stable, beta=w.beta, block_n=128)
        assert_close_bf16("o", o, ref["o"])
        assert_lse(lse, ref["lse"])
        np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
        np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
        np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), em["branch"])
        np.testing.assert_array_equal(st["row_ones"].cpu().numpy(), em["ones"])
        o2, lse2 = run_fwd(w, stable, stats=False)
        assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("stable", [0, 1])
def test_gpt2_small_full(stable):
    w = inputs.gpt2_small()
    o, lse, st = run_fwd(w, stable)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=stable, beta=w.beta)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    # ties/branches on decidable rows of two heads
    for b, h in ((0, 0), (7, 11)):
        dec, bound = A.decidable_rows(w.q, w.k, True, b, h)
        np.testing.assert_array_equal(st["row_ties"][b, h].cpu().numpy()[dec], ref["rs"][b, h][dec])
        np.testing.assert_array_equal(st["row_branch"][b, h].cpu().numpy()[dec], ref["branch"][b, h][dec])
        assert np.all(np.abs(f64(st["row_max_raw"][b, h]) - ref["rm"][b, h]) <= bound * 2 + 1e-6)


def test_sink_plain_and_betas():
    w = inputs.gpt2_medium_sink()
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=0)
    for stable, beta in ((0, 1.25), (1, 1.1), (1, 1.25), (1, 1.5)):
        o, lse, st = run_fwd(w, stable, beta)
        assert_close_bf16(f"o stable={stable} beta={beta}", o, ref["o"])
        assert_lse(lse, ref["lse"])
        _, br = A.shift_rule(ref["rm"], ref["rs"], beta, stable)
        got_rs, got_br = st["row_ties"].cpu().numpy(), st["row_branch"].cpu().numpy()
        # sink ties come from bit-identical key rows; check all rows of a few heads for decidability
        for b, h in ((0, 0), (15, 15)):
            dec, _ = A.decidable_rows(w.q, w.k, True, b, h)
            assert dec.mean() > 0.99
            np.testing.assert_array_equal(got_rs[b, h][dec], ref["rs"][b, h][dec])
            np.testing.assert_array_equal(got_br[b, h][dec], br[b, h][dec])
        # over all heads, mismatches may only occur on rows whose top-2 gap is tiny
        agree = np.mean(got_br == br)
        assert agree > 0.999, agree


@pytest.mark.parametrize("N", [1, 17, 100, 128, 129, 255, 256, 257, 300, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_shapes(N, d, causal):
    w = inputs.random_case(2, 3, N, d, causal, seed=N * 7 + d, std=1.5)
    o, lse, st = run_fwd(w, 1)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=w.beta)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])


def test_no_stats_pointer_path_matches():
    w = inputs.gpt2_small(B=2, H=4, N=512)
    o1, l1 = run_fwd(w, 1, stats=False)
    o2, l2, _ = run_fwd(w, 1, stats=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_nan_key_reaches_every_output_row():
    # a NaN key column poisons every row's scores: the shift ignores it (max skips NaN) but
    # its exponential is NaN, so every row of O and the LSE turn NaN and the call reports it
    w = inputs.random_case(1, 1, 512, 64, False, seed=8)
    q, k, v, _ = to_dev(w)
    k[0, 0, 130, 0] = float("nan")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    assert binding.fa_fwd(q, k, v, o, lse, False, w.scale, 1, 1.25) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_WARN_NONFINITE
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()


def _check_sampled_heads(w, ws, heads, stable, o, lse, st):
    """O, LSE against the oracle on the sampled heads; tie counts and shift branches
    bit-exact on every decidable row (at least 99 % of the rows), the raw row maximum within
    its FP32 error bound there."""
    ref = A.forward(ws.q, ws.k, ws.v, w.scale, w.causal, stable=stable, beta=w.beta)
    assert_close_bf16("o", o[:, heads], ref["o"])
    assert_lse(lse[:, heads], ref["lse"])
    for i, h in enumerate(heads):
        dec, bound = A.decidable_rows(ws.q, ws.k, w.causal, 0, i)
        assert dec.mean() >= 0.99, dec.mean()
        np.testing.assert_array_equal(st["row_ties"][0, h].cpu().numpy()[dec], ref["rs"][0, i][dec])
        np.testing.assert_array_equal(st["row_branch"][0, h].cpu().numpy()[dec], ref["branch"][0, i][dec])
        err = np.abs(f64(st["row_max_raw"][0, h]) - ref["rm"][0, i])
        assert np.all(err[dec] <= 2 * bound[dec]), float(np.max(err[dec] - 2 * bound[dec]))


@pytest.mark.parametrize("stable", [0, 1])
def test_llama7b_full_size_sampled_heads(stable):
    # full 8192-token, 32-head problem on the GPU, plain and stabilised; the oracle checks two
    # heads in full, and the statistics-free kernel (the one the benchmark times) must give
    # the same O and LSE bit for bit
    w = inputs.llama7b_long()
    o, lse, st = run_fwd(w, stable)
    heads = [0, 31]
    ws = inputs.llama7b_long(heads=heads)
    assert torch.equal(ws.q[0, 0], w.q[0, 0]) and torch.equal(ws.q[0, 1], w.q[0, 31])
    _check_sampled_heads(w, ws, heads, stable, o, lse, st)
    o2, lse2 = run_fwd(w, stable, stats=False)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("stable", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_extreme_16k_sampled_head(causal, stable):
    w = inputs.extreme_16k(causal=causal)
    o, lse, st = run_fwd(w, stable)
    heads = [5]
    ws = inputs.extreme_16k(causal=causal, heads=heads)
    _check_sampled_heads(w, ws, heads, stable, o, lse, st)
    o2, lse2 = run_fwd(w, stable, stats=False)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_invalid_arguments_rejected_on_device():
    w = inputs.tiny_ties()
    q, k, v, _ = to_dev(w)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device)
    assert binding.fa_fwd(q, k, v, o, lse, True, -1.0, 1, 1.25) == binding.FA_ERR_INVALID_ARG
    assert binding.fa_fwd(q, k, v, o, lse, True, 0.125, 1, 0.5) == binding.FA_ERR_INVALID_ARG
    assert binding.fa_fwd(q, k, v, o, lse, True, 0.125, 3, 1.25) == binding.FA_ERR_INVALID_ARG
    assert binding.fa_device_status() == binding.FA_OK


@pytest.mark.parametrize("N", [128, 300, 1024])
def test_block_local_variant_matches_emulation(N):
    # stable = 2: each 128-key block applies the rule to its own (max, count); on dyadic
    # inputs the per-row state, the branch of the block that set the shift and the
    # exact-1.0 counts equal the BF16 emulation's
    w = inputs.tiny_ties(N=N, H=2)
    o, lse, st = run_fwd(w, 2)
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=2, beta=w.beta, block_n=128)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=0)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    np.testing.assert_array_equal(st["row_max_raw"].cpu().numpy().astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(st["row_ties"].cpu().numpy(), ref["rs"])
    np.testing.assert_array_equal(st["row_branch"].cpu().numpy(), em["branch"])
    np.testing.assert_array_equal(st["row_ones"].cpu().numpy(), em["ones"])


def test_block_local_variant_large_random():
    w = inputs.gpt2_medium_sink(B=2, H=4, N=1024)
    o, lse = run_fwd(w, 2, stats=False)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=0)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])


def test_zero_maximum_ties_keep_branch_zero():
    # A zero query row scores 0 against every key: its maximum 0 repeats, which matches
    # neither branch of the shift rule (rm > 0 or rm < 0), so m = 0, every visible P~ is
    # exactly 1.0 and the output is the mean of the visible values.
    w = inputs.random_case(1, 2, 200, 64, True, seed=77)
    q = w.q.clone()
    q[:, :, 5] = 0
    q[:, :, 150] = 0
    w = inputs.Workload("zero_rows", q, w.k, w.v, w.do, True, w.scale, 1, 1.25)
    o, lse, st = run_fwd(w, 1)
    ref = A.forward(w.q, w.k, w.v, w.scale, True, stable=1, beta=1.25)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, True, stable=1, beta=1.25, block_n=128)
    for row in (5, 150):
        assert np.all(ref["rm"][0, :, row] == 0) and np.all(ref["rs"][0, :, row] == row + 1)
        np.testing.assert_array_equal(st["row_branch"][0, :, row].cpu().numpy(), [0, 0])
        np.testing.assert_array_equal(st["row_ties"][0, :, row].cpu().numpy(), [row + 1] * 2)
        np.testing.assert_array_equal(st["row_ones"][0, :, row].cpu().numpy(), em["ones"][0, :, row])
        np.testing.assert_allclose(f64(o[0, :, row]), f64(w.v[0, :, :row + 1]).mean(axis=1), atol=1e-2)
    assert np.all(em["ones"][0, :, 5] == 6)


def test_row_minimum_statistic():
    w = inputs.tiny_ties(N=300)
    o, lse, st = run_fwd(w, 1)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=w.beta)
    # dyadic inputs: FP32 scores are exact
    np.testing.assert_array_equal(st["row_min_raw"].cpu().numpy().astype(np.float64), ref["rmin"])


def test_nonfinite_outputs_are_reported():
    # ijyty.com §7.1 / jsqmd.com §5 NaN monitor: an Inf in V reaches O; the call completes
    # and fa_device_status reports FA_WARN_NONFINITE once, then the word is clear again
    w = inputs.random_case(1, 2, 256, 64, True, seed=3)
    q, k, v, do = to_dev(w)
    v[0, 1, 7, 3] = float("inf")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)
    assert binding.fa_fwd(q, k, v, o, lse, True, w.scale, 1, 1.25) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_WARN_NONFINITE
    assert binding.fa_device_status() == binding.FA_OK
    # the finite head is unaffected
    ref = A.forward(w.q[:, :1], w.k[:, :1], w.v[:, :1], w.scale, True, stable=1)
    assert_close_bf16("o", o[:, :1], ref["o"])
    v[0, 1, 7, 3] = 0.0
    assert binding.fa_fwd(q, k, v, o, lse, True, w.scale, 1, 1.25) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_OK


def test_longest_sequence_sampled_head():
    # 32k tokens (the largest size tested): one head checked against the oracle in full
    w = inputs.random_case(1, 2, 32768, 128, True, seed=321, std=1.0)
    o, lse = run_fwd(w, 1, stats=False)
    sub = inputs.Workload("sub", w.q[:, 1:], w.k[:, 1:], w.v[:, 1:], w.do[:, 1:], True, w.scale, 1, 1.25)
    ref = A.forward(sub.q, sub.k, sub.v, w.scale, True, stable=1, beta=1.25, row_block=256)
    assert_close_bf16("o", o[:, 1:], ref["o"])
    assert_lse(lse[:, 1:], ref["lse"])


@pytest.mark.parametrize("beta", [1.0, 2.0])
def test_beta_at_and_beyond_the_recommended_range(beta):
    # beta = 1 makes the positive branch m = rm (the plain shift); beta = 2 moves it far
    w = inputs.gpt2_medium_sink(B=2, H=2, N=512)
    o, lse, st = run_fwd(w, 1, beta)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=beta)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    assert np.mean(st["row_branch"].cpu().numpy() == ref["branch"]) > 0.999


@pytest.mark.parametrize("scale", [0.01, 1.0])
def test_unusual_scales(scale):
    w = inputs.random_case(1, 2, 700, 128, True, seed=int(scale * 1000) + 3, std=1.0)
    w = inputs.Workload("scaled", w.q, w.k, w.v, w.do, True, scale, 1, 1.25)
    o, lse = run_fwd(w, 1, stats=False)
    ref = A.forward(w.q, w.k, w.v, scale, True, stable=1, beta=1.25)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])


@pytest.mark.parametrize("stable", [0, 1, 2])
def test_repeated_launches_without_stats(stable):
    # back-to-back launches of the plain-output kernels (their hand-offs run at full speed):
    # every launch completes without a timeout and gives the same bits as the first
    w = inputs.gpt2_small()
    q, k, v, _ = to_dev(w)
    first = None
    for _ in range(6):
        o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=stable, beta=w.beta)
        if first is None:
            first = (o, lse)
    binding.device_status()
    assert torch.equal(o, first[0]) and torch.equal(lse, first[1])
    ref = A.forward(w.q[:1], w.k[:1], w.v[:1], w.scale, True, stable=stable if stable < 2 else 0, beta=w.beta)
    assert_close_bf16("o", o[:1], ref["o"])


@pytest.mark.parametrize("stable", [0, 1])
def test_compensated_row_sum_on_rows_whose_blocks_fall_below_an_ulp(stable):
    # ijyty.com §7.2 (Kahan summation of the softmax denominator).  32768 keys in 256 blocks:
    # one score 0 (P~ = 1) and 32767 scores whose P~ is ~2^-32, so every block after the first
    # adds less than half an FP32 ulp of l.  A plain FP32 row sum drops all of them and misses
    # the LSE by the dropped mass, ~7e-6 (the emulation pins this on the CPU); the kernel's
    # compensated sum must stay within 1e-6 of the FP64 closed form
    # log(1 + (N - 1) exp(scale * tail)).
    N = 32768
    w = inputs.tiny_tail_rows(N=N)
    o, lse = run_fwd(w, stable, stats=False)
    tail = np.exp(w.scale * -178.0)
    exact = np.log1p((N - 1) * tail)
    assert (N // 128 - 1) * 128 * tail > 5e-6
    err = np.abs(f64(lse) - exact)
    assert err.max() <= 1e-6, err.max()
    # O is key 0's value row plus the tail's ~7e-6 share
    want = np.broadcast_to(f64(w.v[:, :, :1]), o.shape)
    assert_close_bf16("o", o, want)
