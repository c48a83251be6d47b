"""The backward's work-item walk (d = 64, up to 4096 tokens).

There the backward launches one CTA per SM and each CTA walks several (key tile,
head) items: the next item's K and V load into a second buffer, and its first
products run while the current item's dK and dV are written out.  Every
per-step barrier then runs its phases across item boundaries.  The test build
(FA_TEST_HOOKS) lets the grid be forced, from one CTA that walks every item to
one CTA per item, so each boundary case runs: items per CTA from 1 to all of
them, a last round that leaves some CTAs idle, ragged and single-tile rows.
dK and dV are summed inside one CTA in a fixed order, so they must be bit-identical
to the product library's; dQ is reduced across CTAs in no fixed order.
"""
import ctypes

import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, build, inputs
from oracle import attention as A
from tests._parity import assert_close_bf16, rel_fro, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks_lib():
    require_gpu()
    lib = ctypes.CDLL(build.build(testhooks=True))
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_bwd_workspace_size.argtypes = [ci, ci, ci, ci]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp] * 10 + [ci, ci, ci, ci, ci, cf, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = ci
    lib.fa_device_status.argtypes = [vp]
    lib.fa_device_status.restype = ci
    lib.fa_last_error.restype = ctypes.c_char_p
    return lib


def _bwd(lib, w, q, k, v, o, lse, do):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, H, N, d = q.shape
    ws = torch.empty(lib.fa_bwd_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None, B, H, N, d, int(w.causal), w.scale,
                    ws.data_ptr(), ws.numel(), stream)
    assert rc == binding.FA_OK, lib.fa_last_error()
    assert lib.fa_device_status(stream) == binding.FA_OK, lib.fa_last_error()
    return dq, dk, dv


CASES = [
    # (B, H, N, causal): items = B * H * ceil(N / 128)
    (1, 3, 1000, True),    # 24 items, causal: 8 .. 1 query tiles each
    (2, 3, 700, False),    # 36 items, ragged last tile
    (1, 5, 129, True),     # 10 items, one and two query tiles
    (3, 1, 128, False),    # 3 items of a single query tile
]


@pytest.mark.parametrize("B,H,N,causal", CASES)
@pytest.mark.parametrize("grid", [1, 2, 5, 7, 0])
def test_item_walk_matches_one_item_per_cta(hooks_lib, monkeypatch, B, H, N, causal, grid):
    w = inputs.random_case(B, H, N, 64, causal, seed=N * 7 + H, std=1.2)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=causal, scale=w.scale, stable=1)
    dq0, dk0, dv0 = binding.backward(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    binding.device_status()
    # grid 0: one CTA per item, the walk of length one
    items = B * H * ((N + 127) // 128)
    monkeypatch.setenv("FA_TEST_BWD_GRID", str(grid if grid else items))
    dq, dk, dv = _bwd(hooks_lib, w, q, k, v, o, lse, do)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    assert rel_fro(dq, dq0) <= 1e-3


def test_single_cta_walk_matches_oracle(hooks_lib, monkeypatch):
    # one CTA walks all 24 items; gradients against the FP64 oracle
    w = inputs.random_case(2, 3, 500, 64, True, seed=77, std=1.0)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, stable=1)
    binding.device_status()
    monkeypatch.setenv("FA_TEST_BWD_GRID", "1")
    dq, dk, dv = _bwd(hooks_lib, w, q, k, v, o, lse, do)
    f = A.forward(w.q, w.k, w.v, w.scale, True)
    ref = A.backward(w.q, w.k, w.v, f["o"], f["lse"], w.do, w.scale, True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close_bf16(name, got, ref[name])


def test_grid_override_is_ignored_at_d128(hooks_lib, monkeypatch):
    # d = 128 has one K/V buffer and always takes one CTA per item
    w = inputs.random_case(1, 2, 384, 128, True, seed=5, std=1.0)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, stable=1)
    dq0, dk0, dv0 = binding.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
    binding.device_status()
    monkeypatch.setenv("FA_TEST_BWD_GRID", "1")
    dq, dk, dv = _bwd(hooks_lib, w, q, k, v, o, lse, do)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    assert rel_fro(dq, dq0) <= 1e-3


def test_walk_at_full_gpt2_small_size_matches_one_item_per_cta(hooks_lib, monkeypatch):
    # 768 items: the product's own walk (one CTA per SM) against one CTA per item
    w = inputs.gpt2_small()
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale, stable=1)
    dq0, dk0, dv0 = binding.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
    binding.device_status()
    monkeypatch.setenv("FA_TEST_BWD_GRID", str(8 * 12 * 8))
    dq, dk, dv = _bwd(hooks_lib, w, q, k, v, o, lse, do)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    assert rel_fro(dq, dq0) <= 1e-3
