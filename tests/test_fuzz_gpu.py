"""Seeded random shapes and modes through the C ABI, each checked in full against the oracle.

Every case draws B, H, N (ragged, up to 1500), d in {64, 128}, causal, stable in {0, 1, 2},
beta and scale from a fixed seed, then compares the BF16 forward, the backward and the FP8
forward with the FP64 oracle at the same tolerances as the targeted tests.
"""
import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from oracle import attention as A
from oracle import fp8 as F
from tests._parity import assert_close_bf16, assert_lse, rel_fro, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def draw(i):
    rng = np.random.default_rng(90210 + i)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    N = int(rng.integers(1, 1500))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    stable = int(rng.integers(0, 3))
    beta = float(rng.uniform(1.0, 1.6))
    scale = float(rng.uniform(0.03, 0.3))
    std = float(rng.uniform(0.5, 2.0))
    w = inputs.random_case(B, H, N, d, causal, seed=4000 + i, std=std)
    return inputs.Workload(f"fuzz{i}", w.q, w.k, w.v, w.do, causal, scale, stable, beta)


@pytest.mark.parametrize("i", range(12))
def test_random_case(i):
    w = draw(i)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=w.stable, beta=w.beta)
    dq, dk, dv = binding.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    binding.device_status()
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal, stable=min(w.stable, 1), beta=w.beta)
    assert_close_bf16("o", o, ref["o"])
    assert_lse(lse, ref["lse"])
    g = A.backward(w.q, w.k, w.v, ref["o"], ref["lse"], w.do, w.scale, w.causal)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close_bf16(name, got, g[name])
    # FP8 forward of the same problem, inputs quantised by the oracle
    codes, ds = [], []
    for t in (w.q, w.k, w.v):
        c, s = F.quantize_per_tensor(t.float().numpy())
        codes.append(c)
        ds.append(s)
    ds = np.array(ds, dtype=np.float32)
    o8, lse8 = binding.forward_fp8(*(torch.from_numpy(c).cuda() for c in codes), torch.from_numpy(ds).cuda(),
                                   causal=w.causal, scale=w.scale, stable=w.stable, beta=w.beta)
    binding.device_status()
    ref8 = F.forward_fp8(*codes, ds, w.scale, w.causal, stable=min(w.stable, 1), beta=w.beta)
    assert rel_fro(o8, ref8["o"]) <= 6e-2
    assert_lse(lse8, ref8["lse"])
