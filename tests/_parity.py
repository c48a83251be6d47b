"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: BF16 outputs and gradients vs FP64, relative Frobenius error; LSE absolute.
REL_TOL = 1e-2
LSE_TOL = 1e-3


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(got, ref) -> float:
    got, ref = f64(got), f64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def per_head_rel(got, ref):
    got, ref = f64(got), f64(ref)
    B, H = ref.shape[:2]
    return np.array([[rel_fro(got[b, h], ref[b, h]) for h in range(H)] for b in range(B)])


def assert_close_bf16(name, got, ref, tol=REL_TOL):
    per = per_head_rel(got, ref)
    tot = rel_fro(got, ref)
    assert tot <= tol and per.max() <= tol, f"{name}: rel Frobenius {tot:.3e}, worst head {per.max():.3e} > {tol}"
    return tot


def assert_lse(got, ref, tol=LSE_TOL):
    err = float(np.max(np.abs(f64(got) - f64(ref))))
    assert err <= tol, f"lse: max abs err {err:.3e} > {tol}"
    return err


def to_dev(w, dev="cuda"):
    return tuple(t.to(dev) for t in (w.q, w.k, w.v, w.do))


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from numerics_tcgen05_tmem_gb300 import build
    build.build()
