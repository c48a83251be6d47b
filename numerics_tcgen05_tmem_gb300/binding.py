"""Thin ctypes binding of ``libfa.so`` (see ``include/fa.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the stream.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_DEVICE_BOUNDS = 5
FA_WARN_NONFINITE = 6

# which output a non-finite count belongs to (fa_device_report.nonfinite[i])
FA_OUT_O, FA_OUT_LSE, FA_OUT_DQ, FA_OUT_DK, FA_OUT_DV = range(5)
OUTPUT_NAMES = ("o", "lse", "dq", "dk", "dv")
FA_DEVFLAG_TIMEOUT, FA_DEVFLAG_BOUNDS, FA_DEVFLAG_NONFINITE = 1, 2, 4

# every symbol include/fa.h declares
EXPORTS = ("fa_fwd", "fa_fwd_fp8", "fa_quantize_fp8", "fa_bwd", "fa_bwd_staged", "fa_bwd_noalloc",
           "fa_bwd_noalloc_status", "fa_bwd_workspace_size", "fa_device_status", "fa_device_report_read",
           "fa_last_error", "fa_version")

# size of the fixed device scratch behind fa_bwd_noalloc (FA_NOALLOC_SCRATCH_BYTES in fa.h)
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

FA_BWD_PREPROCESS, FA_BWD_MAIN, FA_BWD_DQ_CONVERT, FA_BWD_ALL = 1, 2, 4, 7


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"fa error {code}: {msg}")
        self.code = code


class RowStats(ctypes.Structure):
    _fields_ = [("row_max_raw", ctypes.c_void_p), ("row_ties", ctypes.c_void_p),
                ("row_branch", ctypes.c_void_p), ("row_ones", ctypes.c_void_p),
                ("row_min_raw", ctypes.c_void_p)]


class DeviceReport(ctypes.Structure):
    """fa_device_report: flags, the first failed index check and non-finite counts per output."""
    _fields_ = [("flags", ctypes.c_uint32), ("bounds_site", ctypes.c_uint32), ("bounds_value", ctypes.c_int64),
                ("nonfinite", ctypes.c_uint64 * 5), ("reserved", ctypes.c_uint64)]

    def as_dict(self):
        return {"flags": int(self.flags), "bounds_site": int(self.bounds_site),
                "bounds_value": int(self.bounds_value),
                "nonfinite": {n: int(self.nonfinite[i]) for i, n in enumerate(OUTPUT_NAMES)}}


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m numerics_tcgen05_tmem_gb300.build`")
    L = ctypes.CDLL(path)
    vp, ci, cf, cs = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, ctypes.POINTER(RowStats), vp]
    L.fa_fwd.restype = ci
    L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, cf, ctypes.POINTER(RowStats), vp]
    L.fa_fwd_fp8.restype = ci
    L.fa_quantize_fp8.argtypes = [vp, cs, vp, vp, vp]
    L.fa_quantize_fp8.restype = ci
    L.fa_bwd_workspace_size.argtypes = [ci, ci, ci, ci]
    L.fa_bwd_workspace_size.restype = cs
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, cs, vp]
    L.fa_bwd.restype = ci
    L.fa_bwd_staged.argtypes = L.fa_bwd.argtypes + [ci]
    L.fa_bwd_staged.restype = ci
    L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp]
    L.fa_bwd_noalloc.restype = ci
    L.fa_device_status.argtypes = [vp]
    L.fa_device_status.restype = ci
    L.fa_device_report_read.argtypes = [vp, ctypes.POINTER(DeviceReport)]
    L.fa_device_report_read.restype = ci
    L.fa_bwd_noalloc_status.argtypes = [vp, ctypes.POINTER(DeviceReport)]
    L.fa_bwd_noalloc_status.restype = ci
    L.fa_last_error.argtypes = []
    L.fa_last_error.restype = ctypes.c_char_p
    L.fa_version.argtypes = []
    L.fa_version.restype = ctypes.c_char_p
    _lib = L
    return L


def last_error() -> str:
    return load().fa_last_error().decode()


def _check(rc: int):
    if rc != FA_OK:
        raise FAError(rc, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_qkv(*ts):
    for t in ts:
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
            raise ValueError("expected contiguous CUDA bfloat16 tensors of shape [B, H, N, d]")
    if any(t.shape != ts[0].shape for t in ts):
        raise ValueError("q, k, v (and o, dO) must have the same shape")


# ----------------------------------------------------------------- raw C calls

def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stable: int, beta: float, stats=None, stream=None) -> int:
    B, H, N, d = q.shape
    st = _row_stats(stats)
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                         float(scale), int(stable), float(beta), ctypes.byref(st) if st is not None else None,
                         _stream(stream))


def _row_stats(stats):
    if stats is None:
        return None
    return RowStats(*(None if stats.get(n) is None else stats[n].data_ptr()
                      for n in ("row_max_raw", "row_ties", "row_branch", "row_ones", "row_min_raw")))


def fa_fwd_fp8(q8, k8, v8, descale, o, lse, causal: bool, scale: float, stable: int, beta: float, stats=None,
               stream=None) -> int:
    B, H, N, d = q8.shape
    st = _row_stats(stats)
    return load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(descale), _ptr(o), _ptr(lse), B, H, N, d,
                             int(bool(causal)), float(scale), int(stable), float(beta),
                             ctypes.byref(st) if st is not None else None, _stream(stream))


def fa_quantize_fp8(x, x8, descale, stream=None) -> int:
    return load().fa_quantize_fp8(_ptr(x), int(x.numel()), _ptr(x8), _ptr(descale), _stream(stream))


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, delta, causal: bool, scale: float, workspace, stream=None,
           stages: int = FA_BWD_ALL) -> int:
    B, H, N, d = q.shape
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(delta),
            B, H, N, d, int(bool(causal)), float(scale), _ptr(workspace), nbytes, _stream(stream))
    if stages == FA_BWD_ALL:
        return load().fa_bwd(*args)
    return load().fa_bwd_staged(*args, int(stages))


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, delta, causal: bool, scale: float, stream=None) -> int:
    """fa_bwd without a workspace: the library's fixed device scratch is used (nothing is allocated)."""
    B, H, N, d = q.shape
    return load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(delta), B, H, N, d, int(bool(causal)), float(scale),
                                 _stream(stream))


def fa_device_status(stream=None) -> int:
    return load().fa_device_status(_stream(stream))


def fa_device_report_read(stream=None):
    """(status code, report dict) of the library's device status record; reading clears it."""
    rep = DeviceReport()
    rc = load().fa_device_report_read(_stream(stream), ctypes.byref(rep))
    return rc, rep.as_dict()


def fa_bwd_noalloc_status(stream=None):
    """(status code, report dict) of fa_bwd_noalloc's own status record; reading clears it."""
    rep = DeviceReport()
    rc = load().fa_bwd_noalloc_status(_stream(stream), ctypes.byref(rep))
    return rc, rep.as_dict()


# ----------------------------------------------------------------- tensor-level helpers

def _stats_dict(B, H, N, device):
    return {"row_max_raw": torch.empty((B, H, N), device=device, dtype=torch.float32),
            "row_ties": torch.empty((B, H, N), device=device, dtype=torch.int32),
            "row_branch": torch.empty((B, H, N), device=device, dtype=torch.int8),
            "row_ones": torch.empty((B, H, N), device=device, dtype=torch.int32),
            "row_min_raw": torch.empty((B, H, N), device=device, dtype=torch.float32)}


def forward(q, k, v, causal: bool = True, scale=None, stable: int = 1, beta: float = 1.25, stats: bool = False,
            stream=None):
    """Returns (o, lse) or (o, lse, stats_dict); outputs are freshly allocated."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    sd = _stats_dict(B, H, N, q.device) if stats else None
    _check(fa_fwd(q, k, v, o, lse, causal, scale, stable, beta, sd, stream))
    return (o, lse, sd) if stats else (o, lse)


def quantize_fp8(x, stream=None):
    """Dynamic per-tensor E4M3 scaling of a contiguous CUDA bfloat16 tensor.

    Returns (x8, descale): x8 holds the E4M3 codes as uint8 with x's shape, descale is a
    1-element FP32 CUDA tensor; x is represented by x8 * descale.
    """
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("expected a contiguous CUDA bfloat16 tensor")
    x8 = torch.empty(x.shape, device=x.device, dtype=torch.uint8)
    descale = torch.empty(1, device=x.device, dtype=torch.float32)
    _check(fa_quantize_fp8(x, x8, descale, stream))
    return x8, descale


def forward_fp8(q8, k8, v8, descale, causal: bool = True, scale=None, stable: int = 1, beta: float = 1.25,
                stats: bool = False, stream=None):
    """FP8 forward: q8, k8, v8 are uint8 E4M3 codes [B, H, N, d]; descale is an FP32 CUDA
    tensor of 3 per-tensor scales (Q, K, V).  Returns (o, lse) or (o, lse, stats_dict)."""
    for t in (q8, k8, v8):
        if not (t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous() and t.dim() == 4 and t.shape == q8.shape):
            raise ValueError("expected contiguous CUDA uint8 tensors of one shape [B, H, N, d]")
    if not (descale.is_cuda and descale.dtype == torch.float32 and descale.numel() == 3 and descale.is_contiguous()):
        raise ValueError("descale must be a contiguous CUDA float32 tensor of 3 elements")
    B, H, N, d = q8.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty((B, H, N, d), device=q8.device, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32)
    sd = _stats_dict(B, H, N, q8.device) if stats else None
    _check(fa_fwd_fp8(q8, k8, v8, descale, o, lse, causal, scale, stable, beta, sd, stream))
    return (o, lse, sd) if stats else (o, lse)


def backward(q, k, v, o, lse, do, causal: bool = True, scale=None, workspace=None, want_delta: bool = False,
             stream=None):
    """Returns (dq, dk, dv) or (dq, dk, dv, delta)."""
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if want_delta else None
    _check(fa_bwd(q, k, v, o, lse, do, dq, dk, dv, delta, causal, scale, workspace, stream))
    return (dq, dk, dv, delta) if want_delta else (dq, dk, dv)


def device_status(stream=None):
    """Synchronise and raise if a kernel reported a device-side error."""
    _check(fa_device_status(stream))
