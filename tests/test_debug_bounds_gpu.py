"""The index-checking debug build over the ragged-shape suite.

compute-sanitizer is not available to this project, so the library has a debug
build (FA_DEBUG_BOUNDS) in which the kernels check their computed global,
shared-memory, tensor-memory and TMA indices before each access and record the
first violation (site and index) in the device status record instead of
trapping.  This test runs the forward, the backward and the FP8 forward of that
build over ragged and edge shapes, and asserts that no check fired and that the
results are those of the product library (bit for bit, except dQ, whose FP32
reduce-adds may land in another order).
"""
import ctypes

import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, build, inputs
from tests._parity import rel_fro, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    require_gpu()
    lib = ctypes.CDLL(build.build(debug_bounds=True))
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, vp, vp]
    lib.fa_fwd.restype = ci
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, vp, vp]
    lib.fa_fwd_fp8.restype = ci
    lib.fa_bwd_workspace_size.argtypes = [ci, ci, ci, ci]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp] * 10 + [ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = ci
    lib.fa_device_report_read.argtypes = [vp, ctypes.POINTER(binding.DeviceReport)]
    lib.fa_device_report_read.restype = ci
    lib.fa_last_error.restype = ctypes.c_char_p
    return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _assert_clean(lib):
    rep = binding.DeviceReport()
    rc = lib.fa_device_report_read(_stream(), ctypes.byref(rep))
    assert rc == binding.FA_OK and rep.flags == 0, (lib.fa_last_error(), rep.as_dict())


@pytest.mark.parametrize("N", [1, 17, 100, 128, 129, 255, 256, 257, 300, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_shapes_trip_no_index_check(dbg, N, d, causal):
    w = inputs.random_case(2, 3, N, d, causal, seed=N * 13 + d, std=1.3)
    q, k, v, do = to_dev(w)
    B, H = q.shape[:2]
    stable = 1 if N % 2 else 2 if N % 3 == 0 else 0
    o, lse = torch.empty_like(q), torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    assert dbg.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                      int(causal), w.scale, stable, 1.25, None, _stream()) == binding.FA_OK
    _assert_clean(dbg)
    o_ref, lse_ref = binding.forward(q, k, v, causal=causal, scale=w.scale, stable=stable, beta=1.25)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)

    ws = torch.empty(dbg.fa_bwd_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert dbg.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, B, H, N, d, int(causal), w.scale,
                      ws.data_ptr(), ws.numel(), _stream()) == binding.FA_OK
    _assert_clean(dbg)
    dq_ref, dk_ref, dv_ref = binding.backward(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    binding.device_status()
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    assert rel_fro(dq, dq_ref) <= 1e-3


@pytest.mark.parametrize("N", [1, 129, 300, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_fp8_forward_trips_no_index_check(dbg, N, d):
    w = inputs.random_case(1, 2, N, d, True, seed=N + d, std=1.0)
    q, k, v, _ = to_dev(w)
    (q8, dq8), (k8, dk8), (v8, dv8) = (binding.quantize_fp8(t) for t in (q, k, v))
    desc = torch.cat([dq8, dk8, dv8])
    B, H = q.shape[:2]
    o, lse = torch.empty_like(q), torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    assert dbg.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), desc.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, H, N, d, 1, w.scale, 1, 1.25, None, _stream()) == binding.FA_OK
    _assert_clean(dbg)
    o_ref, lse_ref = binding.forward_fp8(q8, k8, v8, desc, causal=True, scale=w.scale, stable=1, beta=1.25)
    binding.device_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_item_walk_trips_no_index_check(dbg, causal):
    # d = 64 with more (key tile, head) items than SMs: every CTA of the debug build walks
    # several items, so the index checks also cover the walk's later items
    w = inputs.random_case(4, 40, 700, 64, causal, seed=707 + causal, std=1.1)
    q, k, v, do = to_dev(w)
    B, H, N, d = q.shape
    assert B * H * ((N + 127) // 128) > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    o, lse = binding.forward(q, k, v, causal=causal, scale=w.scale, stable=1, beta=1.25)
    ws = torch.empty(dbg.fa_bwd_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert dbg.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, B, H, N, d, int(causal), w.scale,
                      ws.data_ptr(), ws.numel(), _stream()) == binding.FA_OK
    _assert_clean(dbg)
    dq_ref, dk_ref, dv_ref = binding.backward(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    binding.device_status()
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
    assert rel_fro(dq, dq_ref) <= 1e-3
