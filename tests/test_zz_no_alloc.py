"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers (a plugin inside a host application that owns the device-memory
budget, or a latency-critical path where cudaMalloc would synchronise the
device) cannot call cudaMalloc.  fa_bwd_noalloc runs the same backward with its
scratch in a fixed device array inside the library.  This test calls it through
the C ABI and checks its gradients against fa_bwd's (the entry point with a
caller-allocated workspace) on two calls in a row with different problems, so
leftovers of the first call in the shared scratch cannot leak into the second.

It lives in its own file, collected last, and passes both alone in a fresh
process and after the other tests.
"""
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from tests._parity import REL_TOL, rel_fro, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _grads_both_ways(w):
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=1, beta=1.25)
    ref = binding.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, want_delta=True)
    got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
           torch.empty(q.shape[:3], device=q.device, dtype=torch.float32)]
    rc = binding.fa_bwd_noalloc(q, k, v, o, lse, do, *got, w.causal, w.scale)
    assert rc == binding.FA_OK, binding.last_error()
    # its kernels report into the entry point's own status record (no timeout, no NaN)
    rc, rep = binding.fa_bwd_noalloc_status()
    assert rc == binding.FA_OK and rep["flags"] == 0, (binding.last_error(), rep)
    binding.device_status()
    return ref, got


def test_noalloc_matches_workspace_backward_on_two_calls_in_a_row():
    first = inputs.gpt2_small(B=2, H=6, N=1024, d=64)          # ~12.6 MB of scratch
    second = inputs.random_case(1, 3, 700, 128, False, seed=5)  # different size, d and mask
    for w in (first, second):
        ref, got = _grads_both_ways(w)
        for name, a, b in zip(("dq", "dk", "dv", "delta"), got, ref):
            err = rel_fro(a, b)
            assert err <= REL_TOL, f"{w.name} {name}: {err:.3e}"
        # the two paths run the same kernels: dK, dV and delta agree exactly
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]) and torch.equal(got[3], ref[3])


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H, N, d = 1, 16, 8192, 128   # needs ~67 MB of scratch > 32 MiB
    assert binding.fa_bwd_workspace_size(B, H, N, d) > binding.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((B, H, N, d), device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros((B, H, N), device="cuda", dtype=torch.float32)
    rc = binding.fa_bwd_noalloc(x, x, x, x, lse, x, x, x, x, None, True, 0.088)
    assert rc == binding.FA_ERR_INVALID_ARG
    assert "fa_bwd_noalloc holds at most" in binding.last_error()


def test_noalloc_status_reports_nonfinite_gradients_and_clears():
    # A NaN in dO reaches dQ, dK and dV.  The no-allocation entry point's own status record
    # reports it (with per-output counts equal to the non-finite entries written), a second
    # read finds it clear, and the library's allocated record is not touched.
    w = inputs.random_case(1, 2, 256, 64, True, seed=4)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    binding.device_status()
    do[0, 0, 200, 5] = float("nan")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert binding.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, None, True, w.scale) == binding.FA_OK
    rc, rep = binding.fa_bwd_noalloc_status()
    assert rc == binding.FA_WARN_NONFINITE
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert rep["nonfinite"][name] == int((~torch.isfinite(t.float())).sum().item()) > 0, (name, rep)
    assert rep["nonfinite"]["o"] == rep["nonfinite"]["lse"] == 0
    assert binding.fa_bwd_noalloc_status()[0] == binding.FA_OK
    assert binding.fa_device_report_read()[0] == binding.FA_OK
    do[0, 0, 200, 5] = 0.0
    assert binding.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, None, True, w.scale) == binding.FA_OK
    assert binding.fa_bwd_noalloc_status()[0] == binding.FA_OK
