"""Pins of the blocked BF16 emulation (the oracle's second program)."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import emulation as E
from numerics_tcgen05_tmem_gb300 import inputs


def test_round_bf16_ties_to_even_and_matches_torch():
    one = np.float32(1.0)
    halfway = np.float32(1.0 + 2.0 ** -8)          # midway between 1 and 1 + 2^-7
    assert E.round_bf16(np.array([halfway]))[0] == one
    upper = np.float32(1.0 + 3 * 2.0 ** -8)         # midway between 1+2^-7 and 1+2^-6 -> even
    assert E.round_bf16(np.array([upper]))[0] == np.float32(1.0 + 2.0 ** -6)
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32) * 10
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(E.round_bf16(x), ref)


def test_exp_margin_near_one_clears_bf16_rounding():
    # On the dyadic grid the nearest non-tie score sits 2^-9 (scaled) below the
    # maximum.  exp(-2^-9) lies ~1.9e-6 above the BF16 midpoint 1 - 2^-9, so it
    # rounds to 1.0; two grid steps below (exp(-2^-8)) it does not.  Both sit
    # far from the midpoint compared with any FP32 exp error, so exact-1.0
    # counts are the same whichever correctly rounded exp is used.
    mid = 1.0 - 2.0 ** -9
    p1 = np.float32(np.exp(-2.0 ** -9))
    p2 = np.float32(np.exp(-2.0 ** -8))
    assert E.round_bf16(np.array([p1]))[0] == np.float32(1.0)
    assert E.round_bf16(np.array([p2]))[0] == np.float32(1.0 - 2.0 ** -8)
    assert float(p1) - mid > 1.5e-6 and mid - float(p2) > 1e-3


@pytest.mark.parametrize("block_n", [1, 3, 16, 128])
@pytest.mark.parametrize("stable", [0, 1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_fp64_recurrence_equals_one_shot(block_n, stable, causal):
    # ijyty.com §2.1: the online softmax over key blocks reaches the one-shot result
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 2, 45, 8)) * 2
    k = rng.standard_normal((1, 2, 45, 8)) * 2
    k[0, :, 10] = k[0, :, 3]
    v = rng.standard_normal((1, 2, 45, 8))
    ref = A.forward(q, k, v, 0.5, causal)
    em = E.blocked_forward(q, k, v, 0.5, causal, stable=stable, block_n=block_n, precision="fp64")
    np.testing.assert_allclose(em["o"], ref["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(em["lse"], ref["lse"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("block_n", [1, 7, 32, 128])
def test_running_tie_state_equals_whole_row(block_n):
    w = inputs.tiny_ties()
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1)
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, block_n=block_n)
    np.testing.assert_array_equal(em["rm"].astype(np.float64), ref["rm"])
    np.testing.assert_array_equal(em["rs"], ref["rs"])
    np.testing.assert_array_equal(em["branch"], ref["branch"])


def test_plain_mode_produces_exact_ones_at_repeated_maxima():
    # ijyty.com §2.2/§3.1: a repeated row maximum gives P~ entries of exactly 1.0
    w = inputs.tiny_ties()
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=0)
    rs, ones = em["rs"], em["ones"]
    assert np.all(ones[rs > 1] >= rs[rs > 1])
    assert np.all(ones >= 1)           # the maximum itself always gives exp(0) = 1
    assert np.sum(rs > 1) >= 5


def test_stable_mode_removes_exact_ones():
    # web578.cn "mechanism 2": with a repeated maximum the shift moves so the
    # exponent at the maximum is strictly below 1 -> no exact 1.0 after BF16 rounding
    w = inputs.tiny_ties()
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=1.25)
    rm, rs, m = em["rm"].astype(np.float64), em["rs"], em["m"].astype(np.float64)
    margin = w.scale * np.abs(m - rm)
    sel = (rs > 1) & (rm != 0) & (margin >= 2.0 ** -7)
    assert sel.sum() >= 4
    assert np.all(em["ones"][sel] == 0)
    # rows with a unique maximum keep their single exact 1.0
    assert np.all(em["ones"][rs == 1] >= 1)


def test_bf16_emulation_within_contract_tolerance():
    w = inputs.gpt2_small(B=1, H=2, N=300)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1)
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=1)
    rel = np.linalg.norm(em["o"] - ref["o"]) / np.linalg.norm(ref["o"])
    assert rel <= 1e-2
    assert np.max(np.abs(em["lse"] - ref["lse"])) <= 1e-3


def test_block_local_variant_with_one_block_is_the_whole_row_rule():
    # stable = 2 with a single key block: m = max(-inf, rule(bm, bc)) = rule(rm, rs)
    w = inputs.tiny_ties(N=128)
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=w.beta)
    em2 = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=2, beta=w.beta, block_n=128)
    em1 = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=w.beta, block_n=128)
    np.testing.assert_array_equal(em2["branch"], ref["branch"])
    np.testing.assert_array_equal(em2["m"], em1["m"])
    np.testing.assert_array_equal(em2["ones"], em1["ones"])


def test_block_local_shift_is_the_running_max_of_block_rules():
    # brute force on FP64 scores (exact for dyadic inputs): per block, the rule applied to
    # that block's own maximum and tie count; the row keeps the largest shift, and the branch
    # of the latest block whose shift is at least the previous one
    w = inputs.tiny_ties(N=300, H=2)
    q, k = w.q.double().numpy(), w.k.double().numpy()
    em = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=2, beta=w.beta, block_n=128)
    beta32 = np.float32(w.beta)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            s = q[b, h] @ k[b, h].T
            for i in range(q.shape[2]):
                m, br = -np.inf, 0
                for j0 in range(0, i + 1, 128):
                    blk = s[i, j0:min(i + 1, j0 + 128)]
                    bm = blk.max()
                    bc = int((blk == bm).sum())
                    if bc > 1 and bm > 0:
                        mb, brb = float(np.float32(beta32 * np.float32(bm))), 1
                    elif bc > 1 and bm < 0:
                        mb, brb = 0.0, 2
                    else:
                        mb, brb = bm, 0
                    if mb >= m:
                        br = brb
                    m = max(m, mb)
                assert em["m"][b, h, i] == np.float32(m), (b, h, i)
                assert em["branch"][b, h, i] == br, (b, h, i)
    assert (em["branch"] != 0).sum() > 0


def test_compensated_row_sum_keeps_the_blocks_an_fp32_sum_drops():
    # ijyty.com §7.2 (Kahan summation of the softmax denominator).  Each row sees one score 0
    # (its unique maximum: P~ = 1) and N - 1 scores whose exp is ~2^-32, so after the first
    # block every block adds less than half an FP32 ulp of l.  The plain FP32 recurrence
    # drops all of them; the compensated one keeps them.  The closed form of the LSE is
    # log(1 + (N - 1) exp(scale * tail)), and the one-shot FP64 oracle reaches it.
    N = 4096
    w = inputs.tiny_tail_rows(N=N)
    q = w.q
    exact = np.log1p((N - 1) * np.exp(w.scale * -178.0))
    ref = A.forward(q, w.k, w.v, w.scale, False)
    np.testing.assert_allclose(ref["lse"], exact, rtol=0, atol=1e-15)
    plain = E.blocked_forward(q, w.k, w.v, w.scale, False, block_n=128, compensated=False)
    kahan = E.blocked_forward(q, w.k, w.v, w.scale, False, block_n=128, compensated=True)
    tail = np.exp(w.scale * -178.0)
    lost = (N // 128 - 1) * 128 * tail                        # every block after the first
    assert np.all(np.abs(plain["lse"] - exact) > 0.9 * lost)
    # compensated: only the first block's own tiny terms (summed with the 1.0 inside the
    # block) and the FP32 rounding of the final l (half an ulp of 1) remain
    assert np.all(np.abs(kahan["lse"] - exact) <= 128 * tail + 2.0 ** -24)
    assert 128 * tail + 2.0 ** -24 < 0.15 * lost


def test_compensation_changes_nothing_when_no_block_is_dropped():
    # on ordinary rows the two recurrences agree to FP32 rounding
    w = inputs.gpt2_small(B=1, H=1, N=512)
    a = E.blocked_forward(w.q, w.k, w.v, w.scale, True, stable=1, compensated=False)
    b = E.blocked_forward(w.q, w.k, w.v, w.scale, True, stable=1, compensated=True)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=2e-6)
    np.testing.assert_array_equal(a["ones"], b["ones"])
