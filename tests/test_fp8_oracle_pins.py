"""Pins of the FP8 oracle (E4M3 codec, per-tensor dynamic scaling, FP8 forward, FP8 emulation).

The codec is checked against torch's float8_e4m3fn (a library implementation of the same
format) and against values derived by hand from the format's definition; the forward
against the FP64 attention definition under known scalings.
"""
import numpy as np
import pytest
import torch

from numerics_tcgen05_tmem_gb300 import inputs
from oracle import attention as A
from oracle import emulation as E
from oracle import fp8 as F


def torch_codes(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_matches_torch():
    c = np.arange(256, dtype=np.uint8)
    want = torch.tensor(c).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(F.decode_e4m3(c), want)


def test_decode_hand_values():
    assert F.decode_e4m3(0x7E) == 448.0 and F.decode_e4m3(0xFE) == -448.0
    assert F.decode_e4m3(0x01) == 2.0 ** -9 and F.decode_e4m3(0x08) == 2.0 ** -6
    assert F.decode_e4m3(0x38) == 1.0 and F.decode_e4m3(0x78) == 256.0
    assert np.isnan(F.decode_e4m3(0x7F)) and np.isnan(F.decode_e4m3(0xFF))
    assert F.decode_e4m3(0x80) == 0.0 and np.signbit(F.decode_e4m3(0x80))


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(200000) * 50,
        rng.standard_normal(100000) * 2.0 ** -7,      # subnormal region
        rng.uniform(-448, 448, 100000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    np.testing.assert_array_equal(F.encode_e4m3(x), torch_codes(x))


def test_encode_midpoints_round_to_even():
    vals = F.decode_e4m3(np.arange(0, 0x7F, dtype=np.uint8))    # all finite non-negative values, increasing
    assert np.all(np.diff(vals) > 0)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)       # exact: at most 5 significant bits
    got = F.encode_e4m3(mids)
    lo = np.arange(0, 0x7E, dtype=np.uint8)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)    # the even neighbour
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(F.encode_e4m3(-mids), want | 0x80)
    np.testing.assert_array_equal(got, torch_codes(mids))


def test_encode_hand_values_and_saturation():
    cases = [(448.0, 0x7E), (464.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E), (-np.inf, 0xFE),
             (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (1.5 * 2.0 ** -9, 0x02), (1.0625, 0x38), (1.1875, 0x3A),
             (-0.0, 0x80), (0.0, 0x00), (256.0, 0x78), (2.0 ** -6, 0x08), (7 * 2.0 ** -9, 0x07)]
    for x, code in cases:
        assert int(F.encode_e4m3(np.float32(x))) == code, (x, hex(int(F.encode_e4m3(np.float32(x)))), hex(code))
    assert int(F.encode_e4m3(np.float32(np.nan))) == 0x7F


def test_round_trip_bound():
    # nearest rounding: error at most half a quantum (2^(E-4) relative to the binade, 2^-10 subnormal)
    x = np.random.default_rng(3).uniform(-448, 448, 100000).astype(np.float32)
    y = F.decode_e4m3(F.encode_e4m3(x))
    a = np.abs(x.astype(np.float64))
    E_ = np.maximum(np.floor(np.log2(np.maximum(a, 1e-300))), -6)
    assert np.all(np.abs(y - x) <= 2.0 ** (E_ - 4) * (1 + 1e-12))


def test_quantize_per_tensor():
    w = inputs.llama7b_long(heads=[3])
    for t in (w.q, w.k, w.v):
        codes, ds = F.quantize_per_tensor(t.float().numpy())
        assert ds.dtype == np.float32
        assert ds == np.float32(np.abs(t.float().numpy()).max()) / np.float32(448)
        # the largest element lands on the largest finite code; nothing saturates past it
        assert (codes & 0x7F).max() == 0x7E
        deq = F.dequantize(codes, ds)
        x = t.double().numpy()
        big = np.abs(x) >= 2.0 ** -6 * float(ds)
        assert np.all(np.abs(deq - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-30)
    codes, ds = F.quantize_per_tensor(np.zeros((3, 5), dtype=np.float32))
    assert ds == np.float32(1) and not codes.any()


def _dyadic(seed, shape, lim=16):
    # k/8 with |k| <= 16: exactly representable in E4M3 (at most 4 significant bits)
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(-lim, lim + 1, shape, generator=g).double() / 8).numpy()


def test_forward_fp8_applies_each_descale():
    q, k, v = (_dyadic(s, (1, 2, 40, 16)) for s in (1, 2, 3))
    cq, ck, cv = (F.encode_e4m3(x) for x in (q, k, v))
    assert np.array_equal(F.decode_e4m3(cq), q)
    base = A.forward(q, k, v, 0.25, True)
    r = F.forward_fp8(cq, ck, cv, (2.0, 0.5, 4.0), 0.25, True)
    # dq * dk = 1 leaves the scores alone; dv = 4 scales O by 4 and leaves the LSE alone
    np.testing.assert_allclose(r["o"], 4 * base["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(r["lse"], base["lse"], rtol=1e-13)
    r2 = F.forward_fp8(cq, ck, cv, (2.0, 1.0, 1.0), 0.25, True, stable=1)
    want = A.forward(2 * q, k, v, 0.25, True, stable=1)
    np.testing.assert_allclose(r2["o"], want["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(r2["rs"], want["rs"])
    np.testing.assert_array_equal(r2["rm"], 2 * A.forward(q, k, v, 0.25, True, stable=1)["rm"])


def test_fp8_emulation_rounds_more_entries_to_one():
    # tiny ties: E4M3 keeps 3 mantissa bits, so every P~ that BF16 rounds to 1.0 also
    # rounds to 1.0 in E4M3 (after the 2^8 scaling), and entries down to 1 - 2^-5 join them
    w = inputs.tiny_ties()
    b = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=0, precision="bf16")
    f = E.blocked_forward(w.q, w.k, w.v, w.scale, w.causal, stable=0, precision="fp8")
    assert np.all(f["ones"] >= b["ones"]) and f["ones"].sum() > b["ones"].sum()
    ref = A.forward(w.q, w.k, w.v, w.scale, w.causal)
    rep = ref["rs"] > 1
    assert np.all(f["ones"][rep] >= ref["rs"][rep])


def test_fp8_emulation_within_derived_tolerance():
    # E4M3 rounding of P~ leaves a relative error up to 2^-4 per entry (rms ~ 2^-4/sqrt(3));
    # O averages it over many keys of independent V, so the relative Frobenius error of O
    # sits near 0.036 -- the FP8 tolerance is 6e-2
    w = inputs.random_case(1, 2, 384, 128, True, seed=21, std=1.0)
    ds = []
    deq = []
    for t in (w.q, w.k, w.v):
        c, s = F.quantize_per_tensor(t.float().numpy())
        ds.append(s)
        deq.append(F.dequantize(c, s))
    ref = A.forward(*deq, w.scale, True)
    em = E.blocked_forward(*deq, w.scale, True, precision="fp8")
    err = np.linalg.norm(em["o"] - ref["o"]) / np.linalg.norm(ref["o"])
    assert 5e-3 < err < 6e-2, err
    assert np.max(np.abs(em["lse"] - ref["lse"])) < 1e-3
