"""FP8 (E4M3) encoding, per-tensor dynamic scaling and the FP8 forward -- TEST INFRASTRUCTURE ONLY.

Part of the oracle: plain CPU code that the CUDA library is checked against.  It shares no
code with the CUDA path; only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import it.

Sources (page title, section):
  * ijyty.com/news/896914 (BF16 FlashAttention stability), §6.1: the stabilised shift
    carries over to FP8 training when it is paired with dynamic scaling factors.
  * The same page, §2.1 / §4.1: the online softmax and the shift rule, unchanged.

Readings where the page is silent (it names FP8 and dynamic scaling, nothing more):
  * Format: E4M3 in its finite variant -- 1 sign bit, 4 exponent bits with bias 7, 3
    mantissa bits; exponent field 0 holds subnormals (m/8 * 2^-6); the code with every
    exponent and mantissa bit set is NaN; there is no infinity; the largest finite value
    is 1.75 * 2^8 = 448.
  * Conversion to E4M3 rounds to nearest, ties to even, and saturates: a finite value
    beyond +-448 becomes +-448 (infinities too); NaN becomes the NaN code 0x7F.
  * Dynamic per-tensor scaling: descale = amax(|X|) / 448 in FP32 (1 when X is all zero),
    X8 = E4M3(X / descale) with the division in FP32, so that the largest element lands on
    the largest finite code.  X is represented by X8 * descale.
  * FP8 forward: S_raw = (Q8 dq)(K8 dk)^T and O = softmax(scale S_raw) (V8 dv), i.e. the
    FP64 attention of the dequantised tensors; ties, the row maximum and the shift rule are
    taken on these dequantised raw scores (positive scaling keeps equality and sign).
  * On the GPU the unnormalised probabilities P~ are rounded to E4M3 for the P~V product
    after multiplication by 2^8 (P~ <= 1 would otherwise leave the top of the E4M3 range
    unused and put P~ < 2^-6 into subnormals); ``emulation.blocked_forward`` with
    precision="fp8" reproduces that rounding.

Parity status: ``decode_e4m3`` is pinned against torch's float8_e4m3fn for all 256 codes,
``encode_e4m3`` against torch's conversion on every FP32 value in range that the test draws
and against hand-derived ties, subnormals and saturation; ``quantize_per_tensor`` by the
round-trip bound and amax landing on 448; ``forward_fp8`` reduces to ``attention.forward``
of the dequantised inputs (checked on exactly representable inputs).
"""
from __future__ import annotations

import numpy as np

from . import attention

E4M3_MAX = 448.0
E4M3_NAN = 0x7F
P_SCALE_LOG2 = 8  # P~ is multiplied by 2^8 before its E4M3 rounding (GPU P~V product)


def decode_e4m3(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8) as float64; NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m / 8.0 * 2.0 ** -6
    norm = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    val = sign * np.where(e == 0, sub, norm)
    return np.where((e == 15) & (m == 7), np.nan, val)


def encode_e4m3(x) -> np.ndarray:
    """Round float values (FP32 or FP64) to E4M3 codes: nearest, ties to even, saturating."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    sat = ~nan & (a > E4M3_MAX)
    reg = ~nan & ~sat
    ar = np.where(reg, a, 1.0)
    # exponent of the quantum: values below 2^-6 share the subnormal quantum 2^-9
    _, ex = np.frexp(ar)                       # ar = f * 2^ex with f in [0.5, 1)
    E = np.maximum(ex - 1, -6)                 # floor(log2 ar), clamped to the subnormal range
    E = np.where(ar == 0.0, -6, E)
    quantum = np.exp2((E - 3).astype(np.float64))
    n = ar / quantum                           # exact: division by a power of two
    n = np.round(n)                            # numpy rounds half to even
    carry = n >= 16
    E = np.where(carry, E + 1, E)
    n = np.where(carry, n / 2, n)
    n = n.astype(np.int64)
    subn = (E == -6) & (n < 8)
    efield = np.where(subn, 0, E + 7)
    mfield = np.where(subn, n, n - 8)
    code = (efield << 3) | mfield
    # rounding can carry past 448 only from values already > 448, which saturate above
    code = np.where(sat, 0x7E, code)
    code = np.where(sign & ~nan, code | 0x80, code)
    code = np.where(nan, E4M3_NAN, code)
    out[...] = code.astype(np.uint8)
    return out


def quantize_per_tensor(x):
    """Dynamic per-tensor scaling: returns (E4M3 codes, descale as np.float32)."""
    xf = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(xf))) if xf.size else np.float32(0)
    descale = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
    y = (xf / descale).astype(np.float32)
    return encode_e4m3(y), descale


def dequantize(codes, descale) -> np.ndarray:
    return decode_e4m3(codes) * np.float64(np.float32(descale))


def forward_fp8(q8, k8, v8, descale, scale: float, causal: bool, stable: int = 0, beta: float = 1.25):
    """FP64 attention of the dequantised FP8 inputs; returns ``attention.forward``'s dict."""
    dq, dk, dv = (np.float32(s) for s in descale)
    return attention.forward(dequantize(q8, dq), dequantize(k8, dk), dequantize(v8, dv), scale, causal,
                             stable=stable, beta=beta)
