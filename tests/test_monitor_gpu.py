"""The NaN/Inf monitor, per output (O, LSE, dQ, dK, dV).

The pages ask for a monitor of NaN and of the softmax input's range
(ijyty.com/news/896914 §7.1; "Flash Attention低精度训练稳定性优化实践" §5) and
describe an overflow check on the backward's gradients ("FlashAttention
训练时为什么会梯度爆炸？" §3.3).  Every epilogue counts the NaN/Inf entries it
stores, per output, into the device status record; fa_device_report_read returns
the counts and clears them.  Each test plants a non-finite value that reaches
exactly one output (or, for the LSE, the pair O and LSE), and checks that the
reported counts equal the non-finite entries of the returned tensors and that
every other count is zero.
"""
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from tests._parity import require_gpu, to_dev

pytestmark = pytest.mark.gpu

HUGE = 2.0e38  # finite in BF16 (largest finite is about 3.39e38); its products overflow FP32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _nonfinite(t):
    return int((~torch.isfinite(t.float())).sum().item())


def _report():
    rc, rep = binding.fa_device_report_read()
    return rc, rep["nonfinite"]


def _clean_report():
    rc, counts = _report()
    assert rc == binding.FA_OK and all(v == 0 for v in counts.values()), counts


def _fwd_bwd(q, k, v, do, causal, scale):
    o, lse = binding.forward(q, k, v, causal=causal, scale=scale, stable=1, beta=1.25)
    rc_f, counts_f = _report()
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    rc_b, counts_b = _report()
    return (o, lse, dq, dk, dv), (rc_f, counts_f), (rc_b, counts_b)


def test_inf_in_v_is_counted_in_o_only():
    w = inputs.random_case(1, 2, 256, 64, True, seed=3)
    q, k, v, do = to_dev(w)
    v[0, 1, 7, 3] = float("inf")
    _clean_report()
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, stable=1, beta=1.25)
    rc, counts = _report()
    assert rc == binding.FA_WARN_NONFINITE
    # Key 7 lies in the first 128-key block, which every row of head 1 multiplies with V as a
    # dense product: rows 0-6 (whose causal mask hides key 7) weigh it by P~ = 0, and
    # 0 * Inf = NaN.  So column 3 of all 256 rows of head 1 is not finite, and only that.
    assert counts["o"] == _nonfinite(o) == 256
    assert _nonfinite(o[0, 1, :, 3]) == 256 and _nonfinite(o[0, 0]) == 0
    assert counts["lse"] == 0 and _nonfinite(lse) == 0
    assert counts["dq"] == counts["dk"] == counts["dv"] == 0
    _clean_report()


def test_underflowing_row_sum_is_counted_in_lse_and_o():
    # Outside the stabilised shift's domain: a repeated positive maximum moves the shift to
    # beta * rm; when scale (beta - 1) rm exceeds the FP32 exponent range every P~ of the row
    # underflows, the row sum is 0, LSE = -inf and O = 0/0.  Only those rows are affected.
    w = inputs.random_case(1, 1, 256, 64, True, seed=9)
    q, k, v, do = to_dev(w)
    # row 40 of Q and keys 10, 11 share one huge direction: their scores are the row's
    # repeated maximum, rm = 64 * 4096 = 2^18, so scale (beta - 1) rm = 2^13 >> 126
    q[0, 0, 40] = 0
    q[0, 0, 40, :64] = 64.0
    k[0, 0, 10] = 0
    k[0, 0, 10, :64] = 64.0
    k[0, 0, 11] = k[0, 0, 10]
    _clean_report()
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, stable=1, beta=1.25)
    rc, counts = _report()
    assert rc == binding.FA_WARN_NONFINITE
    assert counts["lse"] == _nonfinite(lse) >= 1
    assert not torch.isfinite(lse[0, 0, 40])
    assert counts["o"] == _nonfinite(o) >= 1
    assert counts["dq"] == counts["dk"] == counts["dv"] == 0
    _clean_report()


def test_overflowing_dv_is_counted_in_dv_only():
    # dO channel c huge and V channel c zero: dP = dO V^T and delta = rowsum(dO o O) do not
    # see channel c (its products are exactly 0), but dV[:, c] = P^T dO[:, c] overflows
    w = inputs.random_case(1, 2, 384, 64, True, seed=11)
    q, k, v, do = to_dev(w)
    v[0, 0, :, 5] = 0
    do[0, 0, :, 5] = HUGE
    _clean_report()
    (o, lse, dq, dk, dv), (rc_f, cf), (rc_b, cb) = _fwd_bwd(q, k, v, do, True, w.scale)
    assert rc_f == binding.FA_OK
    assert rc_b == binding.FA_WARN_NONFINITE
    assert cb["dv"] == _nonfinite(dv) >= 1
    assert cb["dq"] == _nonfinite(dq) == 0 and cb["dk"] == _nonfinite(dk) == 0
    assert cb["o"] == cb["lse"] == 0
    _clean_report()


def test_overflowing_dk_is_counted_in_dk_only():
    # Q channel c huge and K channel c zero: the scores do not see channel c, but
    # dK[:, c] = scale dS^T Q[:, c] overflows; dQ = scale dS K has K[:, c] = 0.  scale = 1,
    # so the overflow shows in the stored value even if the FP32 sum were to saturate.
    w = inputs.random_case(1, 2, 384, 128, True, seed=12, scale=1.0)
    q, k, v, do = to_dev(w)
    k[0, 1, :, 17] = 0
    q[0, 1, :, 17] = HUGE
    _clean_report()
    (o, lse, dq, dk, dv), (rc_f, cf), (rc_b, cb) = _fwd_bwd(q, k, v, do, True, w.scale)
    assert rc_f == binding.FA_OK and _nonfinite(o) == 0 and _nonfinite(lse) == 0
    assert rc_b == binding.FA_WARN_NONFINITE
    assert cb["dk"] == _nonfinite(dk) >= 1
    assert cb["dq"] == _nonfinite(dq) == 0 and cb["dv"] == _nonfinite(dv) == 0
    _clean_report()


def test_overflowing_dq_is_counted_in_dq_only():
    # K channel c huge on every other key and Q channel c zero: the scores do not see
    # channel c, but dQ[:, c] = scale sum over those keys of dS K[:, c] overflows (the sum
    # over all keys of a row of dS is 0, over half of them it is not); dK sees Q[:, c] = 0
    w = inputs.random_case(1, 2, 384, 64, False, seed=13, scale=1.0)
    q, k, v, do = to_dev(w)
    q[0, 0, :, 9] = 0
    k[0, 0, ::2, 9] = HUGE
    _clean_report()
    (o, lse, dq, dk, dv), (rc_f, cf), (rc_b, cb) = _fwd_bwd(q, k, v, do, False, w.scale)
    assert rc_f == binding.FA_OK and _nonfinite(o) == 0
    assert rc_b == binding.FA_WARN_NONFINITE
    assert cb["dq"] == _nonfinite(dq) >= 1
    assert cb["dk"] == _nonfinite(dk) == 0 and cb["dv"] == _nonfinite(dv) == 0
    _clean_report()


def test_counts_accumulate_until_read():
    # two calls before one read: the counts add up, and one read clears them
    w = inputs.random_case(1, 1, 128, 64, False, seed=21)
    q, k, v, do = to_dev(w)
    v[0, 0, 0, 0] = float("nan")
    _clean_report()
    for _ in range(2):
        o, lse = binding.forward(q, k, v, causal=False, scale=w.scale, stable=0)
    rc, counts = _report()
    assert rc == binding.FA_WARN_NONFINITE
    assert counts["o"] == 2 * _nonfinite(o) == 2 * 128
    _clean_report()
