"""e4m3 ("fn" variant) codec and the per-token row quantiser, from the format definition.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never imports this.

Format (8 bits, s eeee mmm, exponent bias 7, no infinities):
  * e = 0:            value = (-1)^s · m · 2^-9            (subnormals, and ±0)
  * 1 <= e <= 15:     value = (-1)^s · (1 + m/8) · 2^(e-7)
  * e = 15, m = 7:    NaN (the only non-finite encoding)
The largest finite magnitude is 1.75 · 2^8 = 448.

Encoding rounds to the nearest representable value, ties to the even code (even
mantissa), and saturates finite magnitudes above 448 to ±448.

The pages say only that the served KV cache is quantised to low bit-width ([A]
§"推理参数与 128K 上下文的使用注意"; [B] §"方法适配": about 6 bits on average, format
unpublished). The e4m3 cache with one fp32 scale per token (scale = amax/448 over the
token's 576 cached elements; a zero row gets scale 1) stands in for it. The division
x/scale is taken in fp32 (IEEE round-to-nearest), so the integer code is decided in
the same precision a GPU encoder uses.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def code_value(code: int) -> float:
    """Value of one 8-bit code, straight from the bit-field definition."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        v = m * 2.0 ** -9
    else:
        v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


DECODE_TABLE = np.array([code_value(c) for c in range(256)], dtype=np.float64)
# Non-negative finite values in code order 0x00..0x7E; strictly increasing.
_POS = DECODE_TABLE[:0x7F].copy()


def decode(codes) -> np.ndarray:
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """fp32 values → uint8 codes (round to nearest, ties to even, saturate at ±448)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 1, 0x7E)   # _POS[hi-1] < a <= _POS[hi]
    lo = hi - 1
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo)
    mag = np.where(a >= E4M3_MAX, 0x7E, mag)
    code = (mag | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(NAN_CODE), code).astype(np.uint8)


def quantize_rows(x):
    """Per-row quantiser: x [T, D] (fp32 values) → (codes uint8 [T, D], scales fp32 [T]).

    scale = amax/448 in fp32 (amax = max |x| over the row; an all-zero row gets 1),
    code  = encode(x / scale) with the division in fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return encode(y), scale


def dequantize_rows(codes, scales) -> np.ndarray:
    """codes [T, D], scales [T] → fp64 values code·scale."""
    return decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]
