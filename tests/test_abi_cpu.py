"""The C-ABI library builds, loads without a GPU and exports what include/fa.h declares.

Only host-side logic runs here (argument validation, workspace sizing); no
kernel is launched.
"""
import ctypes
import os
import re

import pytest

from numerics_tcgen05_tmem_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(binding.EXPORTS) <= set(names), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_version_string(lib):
    assert b"sm_103a" in lib.fa_version()


def test_workspace_size(lib):
    # FP32 dQ accumulator [B,H,N,d], then delta and lse*log2(e) padded to 128-row tiles
    B, H, N, d = 2, 3, 1000, 128
    n_pad = 1024
    want = -(-(B * H * N * d * 4) // 256) * 256 + 2 * (-(-(B * H * n_pad * 4) // 256) * 256)
    assert lib.fa_bwd_workspace_size(B, H, N, d) == want
    assert lib.fa_bwd_workspace_size(1, 1, 1, 96) == 0
    assert lib.fa_bwd_workspace_size(0, 1, 1, 64) == 0


def _fwd(lib, q=None, k=None, v=None, o=None, lse=None, B=1, H=1, N=128, d=64, causal=1, scale=0.125,
         stable=1, beta=1.25):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stable, beta, None, None)


def test_invalid_arguments_fail_before_touching_the_gpu(lib):
    good = ctypes.c_void_p(1 << 20)     # aligned, never dereferenced: validation fails first
    assert _fwd(lib, None, good, good, good, good) == binding.FA_ERR_INVALID_ARG
    assert b"q is NULL" in lib.fa_last_error()
    assert _fwd(lib, ctypes.c_void_p((1 << 20) + 8), good, good, good, good) == binding.FA_ERR_INVALID_ARG
    assert b"aligned" in lib.fa_last_error()
    assert _fwd(lib, good, good, good, good, good, d=96) == binding.FA_ERR_UNSUPPORTED
    assert _fwd(lib, good, good, good, good, good, N=0) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, None) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, scale=float("nan")) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, scale=0.0) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, stable=3) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, stable=-1) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, beta=0.9) == binding.FA_ERR_INVALID_ARG
    assert _fwd(lib, good, good, good, good, good, beta=float("inf")) == binding.FA_ERR_INVALID_ARG


def test_backward_invalid_arguments(lib):
    good = ctypes.c_void_p(1 << 20)
    ws = lib.fa_bwd_workspace_size(1, 1, 128, 64)
    rc = lib.fa_bwd(good, good, good, good, good, good, good, good, None, None, 1, 1, 128, 64, 1, 0.125,
                    good, ws, None)
    assert rc == binding.FA_ERR_INVALID_ARG
    rc = lib.fa_bwd(good, good, good, good, good, good, good, good, good, None, 1, 1, 128, 64, 1, 0.125,
                    good, ws - 256, None)
    assert rc == binding.FA_ERR_INVALID_ARG
    assert b"workspace" in lib.fa_last_error()


def test_fp8_invalid_arguments(lib):
    good = ctypes.c_void_p(1 << 20)
    ds = ctypes.c_void_p(1 << 21)

    def fwd8(q=good, descale=ds, d=128, N=128, stable=1):
        return lib.fa_fwd_fp8(q, good, good, descale, good, good, 1, 1, N, d, 1, 0.125, stable, 1.25, None, None)

    assert fwd8(d=96) == binding.FA_ERR_UNSUPPORTED
    assert b"d=96" in lib.fa_last_error()
    assert fwd8(descale=None) == binding.FA_ERR_INVALID_ARG
    assert fwd8(descale=ctypes.c_void_p((1 << 21) + 2)) == binding.FA_ERR_INVALID_ARG
    assert fwd8(q=None) == binding.FA_ERR_INVALID_ARG
    assert fwd8(N=0) == binding.FA_ERR_INVALID_ARG
    assert fwd8(stable=5) == binding.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_fp8(None, 16, good, ds, None) == binding.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_fp8(good, 16, ctypes.c_void_p((1 << 20) + 4), ds, None) == binding.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_fp8(good, 16, good, None, None) == binding.FA_ERR_INVALID_ARG
    assert b"descale" in lib.fa_last_error()


def test_device_report_layout_matches_header():
    # fa_device_report: flags, bounds_site, bounds_value, nonfinite[5], reserved -> 64 bytes
    assert ctypes.sizeof(binding.DeviceReport) == 64
    assert binding.DeviceReport.nonfinite.offset == 16
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    for name, val in (("FA_OUT_O", 0), ("FA_OUT_LSE", 1), ("FA_OUT_DQ", 2), ("FA_OUT_DK", 3), ("FA_OUT_DV", 4)):
        assert re.search(rf"\b{name} = {val}\b", src), name
        assert getattr(binding, name) == val


def test_report_reader_rejects_null_output(lib):
    assert lib.fa_device_report_read(None, None) == binding.FA_ERR_INVALID_ARG
    assert b"out is NULL" in lib.fa_last_error()
