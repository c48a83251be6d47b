"""GPU parity of the backward (fa_bwd through the C ABI) against the FP64 oracle.

The oracle's gradients are the exact gradients of the FP64 forward from the
same BF16 inputs; the GPU backward runs on the GPU forward's O and LSE.
"""
import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import binding, inputs
from oracle import attention as A
from tests._parity import assert_close_bf16, f64, rel_fro, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def run_fwd_bwd(w, stable=1, beta=1.25):
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=w.causal, scale=w.scale, stable=stable, beta=beta)
    dq, dk, dv, delta = binding.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, want_delta=True)
    binding.device_status()
    return o, lse, dq, dk, dv, delta


def oracle_grads(w, heads=None):
    q, k, v, do = w.q, w.k, w.v, w.do
    f = A.forward(q, k, v, w.scale, w.causal)
    return A.backward(q, k, v, f["o"], f["lse"], do, w.scale, w.causal)


def check(w, res, ref, sel=None):
    o, lse, dq, dk, dv, delta = res
    pick = (lambda t: t) if sel is None else sel
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close_bf16(name, pick(got), ref[name])


@pytest.mark.parametrize("stable", [0, 1])
def test_tiny_ties(stable):
    w = inputs.tiny_ties()
    res = run_fwd_bwd(w, stable)
    check(w, res, oracle_grads(w))


def test_delta_is_rowsum_of_do_times_o():
    # delta = rowsum(dO o O) of the GPU's own O, in FP32
    w = inputs.gpt2_small(B=2, H=3, N=700)
    o, lse, dq, dk, dv, delta = run_fwd_bwd(w)
    want = (f64(w.do) * f64(o)).sum(axis=-1)
    assert rel_fro(delta, want) <= 1e-5


def test_gpt2_small_full():
    w = inputs.gpt2_small()
    check(w, run_fwd_bwd(w), oracle_grads(w))


def test_sink_heads():
    w = inputs.gpt2_medium_sink()
    res = run_fwd_bwd(w, 1, 1.25)
    bs = [0, 15]
    sub = inputs.Workload("sub", w.q[bs], w.k[bs], w.v[bs], w.do[bs], w.causal, w.scale, 1, 1.25)
    check(sub, res, oracle_grads(sub), sel=lambda t: t[bs])


@pytest.mark.parametrize("N", [1, 17, 100, 128, 129, 255, 256, 300, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_shapes(N, d, causal):
    w = inputs.random_case(2, 2, N, d, causal, seed=N * 11 + d, std=1.2)
    check(w, run_fwd_bwd(w), oracle_grads(w))


@pytest.mark.parametrize("stable", [0, 1])
def test_llama7b_full_size_sampled_heads(stable):
    # the backward after a plain or a stabilised forward (it reads only O and LSE)
    w = inputs.llama7b_long()
    res = run_fwd_bwd(w, stable)
    heads = [0, 31]
    ws = inputs.llama7b_long(heads=heads)
    check(ws, res, oracle_grads(ws), sel=lambda t: t[:, heads])


@pytest.mark.parametrize("stable", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_extreme_16k_sampled_head(causal, stable):
    w = inputs.extreme_16k(causal=causal)
    res = run_fwd_bwd(w, stable)
    ws = inputs.extreme_16k(causal=causal, heads=[9])
    check(ws, res, oracle_grads(ws), sel=lambda t: t[:, [9]])


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [4096, 4097])
def test_d64_item_walk_length_boundary_sampled_head(N, causal):
    # d = 64: up to 4096 keys the backward runs one CTA per SM walking the (key tile, head)
    # items (here 512 or more of them), from 4097 keys one CTA per item; both against the oracle
    w = inputs.random_case(2, 8, N, 64, causal, seed=N + 31 * causal, std=1.0)
    res = run_fwd_bwd(w)
    b, h = 1, 5
    sub = inputs.Workload("sub", w.q[b:b + 1, h:h + 1], w.k[b:b + 1, h:h + 1], w.v[b:b + 1, h:h + 1],
                          w.do[b:b + 1, h:h + 1], causal, w.scale, 1, 1.25)
    check(sub, res, oracle_grads(sub), sel=lambda t: t[b:b + 1, h:h + 1])


def test_repeat_calls_reuse_workspace():
    w = inputs.gpt2_small(B=1, H=4, N=1024)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    ws = torch.empty(binding.fa_bwd_workspace_size(*q.shape), device=q.device, dtype=torch.uint8)
    g1 = binding.backward(q, k, v, o, lse, do, scale=w.scale, workspace=ws)
    g2 = binding.backward(q, k, v, o, lse, do, scale=w.scale, workspace=ws)
    binding.device_status()
    for a, b in zip(g1, g2):
        # dK, dV are deterministic; dQ sums FP32 atomics in any order
        assert rel_fro(a, b) <= 1e-3


def test_invalid_workspace_rejected():
    w = inputs.tiny_ties()
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    small = torch.empty(binding.fa_bwd_workspace_size(*q.shape) - 256, device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    rc = binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, None, True, w.scale, small)
    assert rc == binding.FA_ERR_INVALID_ARG
    assert binding.fa_device_status() == binding.FA_OK


def test_nonfinite_gradients_are_reported():
    w = inputs.random_case(1, 2, 256, 64, True, seed=4)
    q, k, v, do = to_dev(w)
    o, lse = binding.forward(q, k, v, causal=True, scale=w.scale)
    binding.device_status()
    do[0, 0, 200, 5] = float("nan")
    ws = torch.empty(binding.fa_bwd_workspace_size(*q.shape), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, None, True, w.scale, ws) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_WARN_NONFINITE
    do[0, 0, 200, 5] = 0.0
    assert binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, None, True, w.scale, ws) == binding.FA_OK
    assert binding.fa_device_status() == binding.FA_OK


def test_longest_sequence_sampled_head():
    # 32k tokens (the largest size tested): gradients of one head checked against the oracle
    w = inputs.random_case(1, 2, 32768, 128, True, seed=322, std=1.0)
    res = run_fwd_bwd(w)
    sub = inputs.Workload("sub", w.q[:, :1], w.k[:, :1], w.v[:, :1], w.do[:, :1], True, w.scale, 1, 1.25)
    check(sub, res, oracle_grads(sub), sel=lambda t: t[:, :1])


@pytest.mark.parametrize("scale", [0.01, 1.0])
def test_unusual_scales(scale):
    w = inputs.random_case(1, 2, 700, 128, True, seed=int(scale * 1000) + 4, std=1.0)
    w = inputs.Workload("scaled", w.q, w.k, w.v, w.do, True, scale, 1, 1.25)
    check(w, run_fwd_bwd(w), oracle_grads(w))
