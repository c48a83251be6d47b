"""Pins of the FP64 oracle against facts the pages and the mathematics fix.

Each test would fail on a plausible mistake in the oracle (a dropped term, a
wrong sign or index, a transposed operand, an off-by-one causal mask).
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from numerics_tcgen05_tmem_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    # a softmax row is a probability distribution
    q, k = _rand((1, 1, 37, 8), 1), _rand((1, 1, 37, 8), 2)
    p = A.probabilities(q, k, 0.7, causal)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)


@pytest.mark.parametrize("ties", [2, 3, 5])
@pytest.mark.parametrize("stable", [0, 1])
def test_k_tied_maxima_give_one_over_k(ties, stable):
    # BF16 FlashAttention stability page §3.2: k equal maxima -> each gets 1/k
    N, d = 8, 2
    q = np.zeros((1, 1, N, d)); q[..., 0] = 1.0
    k = np.zeros((1, 1, N, d)); k[..., 0] = -400.0
    tied = [1, 4, 6, 0, 3][:ties]
    k[0, 0, tied, 0] = 5.0
    v = _rand((1, 1, N, 3), 3)
    out = A.forward(q, k, v, 1.0, False, stable=stable, beta=1.25)
    np.testing.assert_allclose(out["o"][0, 0, 0], v[0, 0, tied].mean(axis=0), rtol=0, atol=1e-12)
    assert abs(out["lse"][0, 0, 0] - (5.0 + math.log(ties))) <= 1e-12
    assert out["rs"][0, 0, 0] == ties and out["rm"][0, 0, 0] == 5.0
    assert out["branch"][0, 0, 0] == (1 if stable else 0)
    p = A.probabilities(q, k, 1.0, False)
    np.testing.assert_allclose(p[0, tied], 1.0 / ties, rtol=0, atol=1e-12)


def test_single_key():
    q, k, v = _rand((1, 2, 1, 4), 4), _rand((1, 2, 1, 4), 5), _rand((1, 2, 1, 4), 6)
    for causal in (False, True):
        out = A.forward(q, k, v, 0.3, causal)
        np.testing.assert_array_equal(out["o"], v)
        np.testing.assert_allclose(out["lse"][..., 0], 0.3 * np.sum(q * k, axis=-1)[..., 0], atol=1e-14)


def test_uniform_logits_causal_and_not():
    # q = 0: every visible key weighs the same.  Causal row i averages v_0..v_i and
    # has LSE = ln(i+1); a non-causal row averages all of v with LSE = ln N.
    N, d = 11, 4
    q = np.zeros((1, 1, N, d))
    k, v = _rand((1, 1, N, d), 7), _rand((1, 1, N, 5), 8)
    c = A.forward(q, k, v, 1.0, True)
    for i in range(N):
        np.testing.assert_allclose(c["o"][0, 0, i], v[0, 0, :i + 1].mean(axis=0), atol=1e-13)
        assert abs(c["lse"][0, 0, i] - math.log(i + 1)) <= 1e-13
    n = A.forward(q, k, v, 1.0, False)
    np.testing.assert_allclose(n["o"][0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (N, 5)), atol=1e-13)
    np.testing.assert_allclose(n["lse"][0, 0], math.log(N), atol=1e-13)


def test_lse_matches_direct_logsumexp_small():
    # the LSE of one row written out directly: ln sum_j exp(s q.k_j) over visible keys
    q, k, v = _rand((1, 1, 6, 3), 9), _rand((1, 1, 6, 3), 10), _rand((1, 1, 6, 3), 11)
    s = 0.9
    out = A.forward(q, k, v, s, True)
    i = 4
    direct = math.log(sum(math.exp(s * sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(3))) for j in range(i + 1)))
    assert abs(out["lse"][0, 0, i] - direct) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_translation_of_keys_keeps_output(causal):
    # adding the same vector u to every key adds q_i.u to every logit of row i:
    # the softmax (hence O) is unchanged and LSE moves by s q_i.u
    q, k, v = _rand((1, 2, 9, 5), 12), _rand((1, 2, 9, 5), 13), _rand((1, 2, 9, 5), 14)
    u = _rand((5,), 15)
    s = 0.6
    a = A.forward(q, k, v, s, causal)
    b = A.forward(q, k + u, v, s, causal)
    np.testing.assert_allclose(b["o"], a["o"], atol=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"] + s * (q @ u), atol=1e-12)


def test_key_permutation_equivariance_noncausal():
    q, k, v = _rand((1, 1, 10, 4), 16), _rand((1, 1, 10, 4), 17), _rand((1, 1, 10, 4), 18)
    perm = np.random.default_rng(19).permutation(10)
    a = A.forward(q, k, v, 0.5, False)
    b = A.forward(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    np.testing.assert_allclose(b["o"], a["o"], atol=1e-12)


def test_shift_rule_golden_cases():
    with open(os.path.join(GOLDEN, "shift_rule_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        row = np.array(c["row"])[None, :]
        vis = np.array(c["visible"], dtype=bool)[None, :]
        rm, rs = A.row_max_and_ties(row, vis)
        m, br = A.shift_rule(rm, rs, c["beta"], 1)
        assert rm[0] == c["rm"] and rs[0] == c["rs"], c
        assert br[0] == c["branch"], c
        assert abs(m[0] - c["m"]) <= 1e-12, c
        m0, br0 = A.shift_rule(rm, rs, c["beta"], 0)
        assert m0[0] == c["rm"] and br0[0] == 0


@pytest.mark.parametrize("make", [lambda: inputs.tiny_ties(), lambda: inputs.gpt2_medium_sink(B=1, H=2, N=256)])
def test_shift_invariance_plain_vs_stable(make):
    # BF16 FlashAttention stability page §3.2: the stabilised shift changes the
    # unnormalised P~ only; the normalised output and LSE are unchanged.
    w = make()
    plain = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=0)
    for beta in (1.1, 1.25, 1.5):
        st = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=beta)
        assert np.any(st["branch"] != 0)
        np.testing.assert_allclose(st["o"], plain["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(st["lse"], plain["lse"], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(st["rs"], plain["rs"])


def test_tiny_ties_has_both_signs_of_repeated_maximum():
    w = inputs.tiny_ties()
    st = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=1.25)
    br = st["branch"]
    assert np.sum(br == A.BRANCH_BETA) >= 2 and np.sum(br == A.BRANCH_ZERO) >= 2
    # planted rows: row 1 repeated negative maximum, row 2 repeated positive maximum
    assert np.all(br[0, :, 1] == A.BRANCH_ZERO) and np.all(br[0, :, 2] == A.BRANCH_BETA)
    assert np.all(st["rs"][0, :, 2] == 3)
    # planted margins clear the BF16 rounding of exp near 1 (scaled |rm| >= 1/8)
    assert np.all(w.scale * np.abs(st["rm"][0, :, 1]) >= 1 / 8)


def test_sink_case_has_many_ties():
    w = inputs.gpt2_medium_sink(B=1, H=2, N=1024)
    st = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1)
    frac = np.mean(st["rs"] > 1)
    assert frac > 0.8  # most rows see the sink key (and its copies) as their maximum


# ---------------------------------------------------------------- backward pins

def _loss(q, k, v, do, s, causal):
    return float(np.sum(do * A.forward(q, k, v, s, causal)["o"]))


@pytest.mark.parametrize("N,d", [(5, 4), (8, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(N, d, causal):
    q, k, v, do = (_rand((1, 1, N, d), 20 + i) for i in range(4))
    s = 1.0 / math.sqrt(d)
    f = A.forward(q, k, v, s, causal)
    g = A.backward(q, k, v, f["o"], f["lse"], do, s, causal)
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            args_m = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            num[idx] = (_loss(*args_p, do, s, causal) - _loss(*args_m, do, s, causal)) / (2 * h)
        rel = np.linalg.norm(g[name] - num) / np.linalg.norm(num)
        assert rel <= 1e-6, (name, rel)


def test_delta_identity_and_dk_sums_to_zero():
    # delta_i = rowsum(dO o O) equals sum_j P_ij dP_ij, and since each row of
    # dS sums to zero, sum_j dK_j = s sum_i q_i sum_j dS_ij = 0.
    N, d = 23, 6
    q, k, v, do = (_rand((1, 1, N, d), 30 + i) for i in range(4))
    s = 0.4
    for causal in (False, True):
        f = A.forward(q, k, v, s, causal)
        g = A.backward(q, k, v, f["o"], f["lse"], do, s, causal)
        p = A.probabilities(q, k, s, causal)
        dp = do[0, 0] @ v[0, 0].T
        np.testing.assert_allclose(g["delta"][0, 0], (p * dp).sum(axis=1), rtol=0, atol=1e-12)
        assert np.max(np.abs(g["dk"][0, 0].sum(axis=0))) <= 1e-12 * max(1.0, np.abs(g["dk"]).max())


def test_dv_closed_form_uniform_causal():
    # q = 0, causal: P_ij = 1/(i+1) for j <= i, so dV_j = sum_{i >= j} dO_i / (i+1)
    N, d = 9, 3
    q = np.zeros((1, 1, N, d))
    k, v, do = (_rand((1, 1, N, d), 40 + i) for i in range(3))
    f = A.forward(q, k, v, 1.0, True)
    g = A.backward(q, k, v, f["o"], f["lse"], do, 1.0, True)
    expect = np.array([sum(do[0, 0, i] / (i + 1) for i in range(j, N)) for j in range(N)])
    np.testing.assert_allclose(g["dv"][0, 0], expect, atol=1e-13)


def test_backward_independent_of_forward_shift():
    # the backward uses only O and LSE, so plain and stable forwards give the same gradients
    w = inputs.tiny_ties()
    res = []
    for st in (0, 1):
        f = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=st)
        res.append(A.backward(w.q, w.k, w.v, f["o"], f["lse"], w.do, w.scale, w.causal))
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(res[1][key], res[0][key], rtol=0, atol=1e-11)


# ---------------------------------------------------------------- decidability

def test_dyadic_rows_are_all_decidable():
    w = inputs.tiny_ties()
    for h in range(2):
        dec, _ = A.decidable_rows(w.q, w.k, True, 0, h)
        assert dec.all()


def test_near_tie_is_undecidable():
    # two different keys whose logits differ by far less than the FP32 error bound
    d = 64
    rng = np.random.default_rng(50)
    q = rng.standard_normal((1, 1, 2, d))
    k = rng.standard_normal((1, 1, 2, d))
    k[0, 0, 1] = k[0, 0, 0]
    k[0, 0, 1, 5] += 1e-9 / q[0, 0, 1, 5]
    dec, _ = A.decidable_rows(q, k, False)
    assert not dec[1]


def test_decidability_is_per_row_whatever_the_row_block():
    # the row blocking only bounds memory: one row at a time gives the same decisions
    w = inputs.gpt2_medium_sink(B=1, H=1, N=512)
    for causal in (True, False):
        d1, b1 = A.decidable_rows(w.q, w.k, causal, 0, 0, row_block=1)
        d2, b2 = A.decidable_rows(w.q, w.k, causal, 0, 0, row_block=200)
        np.testing.assert_array_equal(d1, d2)
        np.testing.assert_array_equal(b1, b2)


def test_row_minimum_over_visible_keys():
    # hand example: row 2 sees keys 0..2 (causal) with scores 3, -4, 7 -> min -4
    q = np.array([[[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]]])
    k = np.array([[[[3.0, 0.0], [0.0, -4.0], [4.0, 3.0]]]])
    v = np.zeros((1, 1, 3, 2))
    out = A.forward(q, k, v, 1.0, True)
    assert out["rmin"][0, 0, 2] == -4.0 and out["rm"][0, 0, 2] == 7.0
    assert out["rmin"][0, 0, 0] == 3.0        # only key 0 visible
    nc = A.forward(q, k, v, 1.0, False)       # non-causal: row 0 scores 3, 0, 4; row 1 scores 0, -4, 3
    assert nc["rmin"][0, 0, 0] == 0.0 and nc["rmin"][0, 0, 1] == -4.0
