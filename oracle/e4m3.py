"""FP8 E4M3 codec (test infrastructure; see the package docstring).

The Pie pages list ``dtype.e4m3`` as a KV-cache type of the FP8 and NVFP4
deployments ("Write a model in Poem", section 2 "Deployments"; "Poem ops",
"Data types") but do not define the format.  The plainest reading is the OCP
8-bit floating point E4M3 format, written out here from its definition:

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0: subnormal, value = (-1)^s * 2^-6 * m/8;
* exponent field 1..15: value = (-1)^s * 2^(e-7) * (1 + m/8);
* the single pattern S.1111.111 is NaN; there are no infinities, so the
  largest finite magnitude is 2^8 * 1.75 = 448.

Encoding rounds to the nearest representable value, ties to the code with an
even mantissa, and saturates to +-448 ("satfinite").  The quantised KV value
is ``encode(float32(x) * inv_scale)`` with ``inv_scale = float32(1 / scale)``
computed once; both are float32 operations, the precision the kernel takes
the same integer decision in.

Pins: exhaustive decode table against the values the format definition fixes
(``tests/golden/e4m3_points.txt``) and against PyTorch's independent
float8_e4m3fn type; encode by brute-force nearest search against PyTorch's
RNE cast over every bf16 input.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode_table() -> np.ndarray:
    """Value of each of the 256 codes, float64 (NaN for S.1111.111)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = (code >> 7) & 1
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            v = np.nan
        elif e == 0:
            v = 2.0 ** -6 * (m / 8.0)
        else:
            v = 2.0 ** (e - 7) * (1.0 + m / 8.0)
        out[code] = -v if s else v
    return out


_TABLE = decode_table()
# finite non-negative codes 0x00..0x7E are strictly increasing in value
_POS_VALUES = _TABLE[:0x7F].copy()


def decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 codes, nearest-even, saturating to +-448.

    NaN inputs map to 0x7F (never produced by the synthetic workloads).
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << 7
    # index of the first table value >= a
    hi = np.searchsorted(_POS_VALUES, a, side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _POS_VALUES[lo]
    dhi = _POS_VALUES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a >= MAX_FINITE, np.uint8(0x7E), code)  # satfinite
    code = code | sign
    code = np.where(np.isnan(x), np.uint8(NAN_CODE), code)
    return code.astype(np.uint8)


def quantize(x_f32: np.ndarray, scale: float) -> np.ndarray:
    """KV quantisation: one float32 multiply by float32(1/scale), then encode."""
    inv = np.float32(1.0) / np.float32(scale)
    with np.errstate(over="ignore"):
        prod = (np.asarray(x_f32, dtype=np.float32) * inv).astype(np.float32)
    return encode(prod)


def dequantize(codes: np.ndarray, scale: float) -> np.ndarray:
    """Dequantised KV value: code value times the float32 scale, in float64."""
    return decode(codes) * np.float64(np.float32(scale))
