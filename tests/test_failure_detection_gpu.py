"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait in the kernels gives up after a time limit, raises the CTA's
abort flag, records FA_ERR_TIMEOUT in the device status record and lets every warp
unwind (in-flight copies land, TMEM is freed).  A test build of the library
(FA_TEST_HOOKS, 100 ms limit) can make the MMA warp wait on a barrier that nothing
arrives on (forward and backward).  The call must report the timeout through
fa_device_status, and the same CUDA context must then compute correct results.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, build, inputs
from oracle import attention as A
from tests._parity import assert_close_bf16, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks_lib():
    require_gpu()
    path = build.build(testhooks=True)
    lib = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, vp, vp]
    lib.fa_fwd.restype = ci
    lib.fa_bwd_workspace_size.argtypes = [ci, ci, ci, ci]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp] * 10 + [ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = ci
    lib.fa_device_status.argtypes = [vp]
    lib.fa_device_status.restype = ci
    lib.fa_bwd_noalloc.argtypes = [vp] * 10 + [ci, ci, ci, ci, ci, cf, vp]
    lib.fa_bwd_noalloc.restype = ci
    lib.fa_bwd_noalloc_status.argtypes = [vp, ctypes.POINTER(binding.DeviceReport)]
    lib.fa_bwd_noalloc_status.restype = ci
    lib.fa_last_error.restype = ctypes.c_char_p
    return lib


def _fwd(lib, w, q, k, v, o, lse):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, H, N, d = q.shape
    return lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                      int(w.causal), w.scale, 1, w.beta, None, stream)


def test_wait_that_runs_out_reports_timeout_and_context_stays_usable(hooks_lib, monkeypatch):
    w = inputs.gpt2_small(B=1, H=4, N=512)
    q, k, v, _ = to_dev(w)
    o = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:3], device=q.device, dtype=torch.float32)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("FA_TEST_INJECT_STALL", "1")
    assert _fwd(hooks_lib, w, q, k, v, o, lse) == binding.FA_OK      # the launch itself is fine
    assert hooks_lib.fa_device_status(stream) == binding.FA_ERR_TIMEOUT
    assert b"timed out" in hooks_lib.fa_last_error()
    assert hooks_lib.fa_device_status(stream) == binding.FA_OK       # reading clears the word
    # same context, no injection: a normal, correct result
    monkeypatch.setenv("FA_TEST_INJECT_STALL", "0")
    assert _fwd(hooks_lib, w, q, k, v, o, lse) == binding.FA_OK
    assert hooks_lib.fa_device_status(stream) == binding.FA_OK
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=1, beta=w.beta)
    assert_close_bf16("o", o, ref["o"])
    # and the product library in the same process is unaffected
    o2, lse2 = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=1)
    binding.device_status()
    assert torch.equal(o2, o)


def test_backward_wait_that_runs_out_reports_timeout_and_context_stays_usable(hooks_lib, monkeypatch):
    w = inputs.gpt2_small(B=1, H=4, N=512)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=1)
    binding.device_status()
    B, H, N, d = q.shape
    ws = torch.empty(hooks_lib.fa_bwd_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def bwd():
        return hooks_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, B, H, N, d, int(w.causal), w.scale,
                                ws.data_ptr(), ws.numel(), stream)

    monkeypatch.setenv("FA_TEST_INJECT_STALL", "1")
    assert bwd() == binding.FA_OK
    assert hooks_lib.fa_device_status(stream) == binding.FA_ERR_TIMEOUT
    assert hooks_lib.fa_device_status(stream) == binding.FA_OK
    monkeypatch.setenv("FA_TEST_INJECT_STALL", "0")
    assert bwd() == binding.FA_OK
    assert hooks_lib.fa_device_status(stream) == binding.FA_OK
    f = A.forward(w.q, w.k, w.v, w.scale, w.causal)
    g = A.backward(w.q, w.k, w.v, f["o"], f["lse"], w.do, w.scale, w.causal)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close_bf16(name, got, g[name])


def test_noalloc_backward_timeout_is_readable_from_its_own_status(hooks_lib, monkeypatch):
    # fa_bwd_noalloc reports into a static status record of its own: a bounded wait that
    # runs out there is returned by fa_bwd_noalloc_status (and not by fa_device_status),
    # the read clears it, and the same context then computes correct gradients
    w = inputs.gpt2_small(B=1, H=4, N=512)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=1)
    binding.device_status()
    B, H, N, d = q.shape
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def bwd():
        return hooks_lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, B, H, N,
                                        d, int(w.causal), w.scale, stream)

    monkeypatch.setenv("FA_TEST_INJECT_STALL", "1")
    assert bwd() == binding.FA_OK
    rep = binding.DeviceReport()
    assert hooks_lib.fa_bwd_noalloc_status(stream, ctypes.byref(rep)) == binding.FA_ERR_TIMEOUT
    assert rep.flags & binding.FA_DEVFLAG_TIMEOUT
    assert hooks_lib.fa_device_status(stream) == binding.FA_OK
    assert hooks_lib.fa_bwd_noalloc_status(stream, None) == binding.FA_OK
    monkeypatch.setenv("FA_TEST_INJECT_STALL", "0")
    assert bwd() == binding.FA_OK
    assert hooks_lib.fa_bwd_noalloc_status(stream, None) == binding.FA_OK
    f = A.forward(w.q, w.k, w.v, w.scale, w.causal)
    g = A.backward(w.q, w.k, w.v, f["o"], f["lse"], w.do, w.scale, w.causal)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close_bf16(name, got, g[name])
