"""e2m3 (6-bit float) codec, its per-group quantiser and the 3-byte packing of the
~6-bit cache reading, from the format definition.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never imports this.

The pages report the served KV cache at about 6 bits per element ([A]
§"推理参数与 128K 上下文的使用注意"; [B] §"瓶颈": 128K tokens x 60 layers at 6 bits
≈ 3.4 GB for one sequence) without its format. The reading taken here, which a later
decode kernel is to match:

Format (6 bits, s ee mmm, exponent bias 1, no infinities and no NaN):
  * e = 0:            value = (-1)^s · m · 2^-3            (subnormals, and ±0)
  * 1 <= e <= 3:      value = (-1)^s · (1 + m/8) · 2^(e-1)
The largest magnitude is 1.875 · 2^2 = 7.5; the positive values are k/8 for k = 0..15,
k/4 for k = 8..15 and k/2 for k = 8..15.

Grouping: each cached token's 576 elements form nine groups of 64 consecutive
elements; group g has one fp32 scale = amax_g / 7.5 (an all-zero group gets 1), and
code = encode(x / scale) with the division in fp32. Encoding rounds to the nearest
value, ties to the even code (even mantissa), and saturates at ±7.5; inputs are
finite (cache rows are bf16 values).

Packing: four consecutive codes c0..c3 of a token form the 24-bit little-endian word
c0 | c1 << 6 | c2 << 12 | c3 << 18, stored as its three bytes in order; a token is 432
bytes of codes plus nine fp32 scales (36 bytes), 468 bytes in all against 580 for the
e4m3 codes with one scale per token.
"""

from __future__ import annotations

import numpy as np

E2M3_MAX = 7.5
GROUP = 64
CODE_BITS = 6


def code_value(code: int) -> float:
    """Value of one 6-bit code, straight from the bit-field definition."""
    s = (code >> 5) & 1
    e = (code >> 3) & 0x3
    m = code & 0x7
    if e == 0:
        v = m * 2.0 ** -3
    else:
        v = (1.0 + m / 8.0) * 2.0 ** (e - 1)
    return -v if s else v


DECODE_TABLE = np.array([code_value(c) for c in range(64)], dtype=np.float64)
# Non-negative values in code order 0x00..0x1F; strictly increasing.
_POS = DECODE_TABLE[:0x20].copy()


def decode(codes) -> np.ndarray:
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8) & 0x3F]


def encode(x) -> np.ndarray:
    """Finite fp32 values → 6-bit codes in uint8 (nearest, ties to even, saturate at ±7.5)."""
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("e2m3 encodes finite values only")
    a = np.abs(x).astype(np.float64)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 1, 0x1F)   # _POS[hi-1] < a <= _POS[hi]
    lo = hi - 1
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo)
    mag = np.where(a >= E2M3_MAX, 0x1F, mag)
    return (mag | (np.signbit(x).astype(np.int64) << 5)).astype(np.uint8)


def quantize_groups(x):
    """x [T, D] (fp32 values, D a multiple of 64) → (codes uint8 [T, D], scales fp32 [T, D/64]).

    scale_g = amax_g / 7.5 in fp32 over each 64-element group (an all-zero group gets 1),
    code    = encode(x / scale_g) with the division in fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    T, D = x.shape
    if D % GROUP:
        raise ValueError("the row length must be a multiple of 64")
    g = x.reshape(T, D // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(E2M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (g / scale[..., None]).astype(np.float32)
    return encode(y).reshape(T, D), scale


def dequantize_groups(codes, scales) -> np.ndarray:
    """Inverse of quantize_groups in fp64: value = decode(code) · scale of its group."""
    codes = np.asarray(codes, dtype=np.uint8)
    T, D = codes.shape
    v = decode(codes).reshape(T, D // GROUP, GROUP) * np.asarray(scales, dtype=np.float64)[..., None]
    return v.reshape(T, D)


def pack(codes) -> np.ndarray:
    """6-bit codes [..., 4n] → bytes [..., 3n]: four codes per little-endian 24-bit word."""
    c = np.asarray(codes, dtype=np.uint32) & 0x3F
    if c.shape[-1] % 4:
        raise ValueError("the code count must be a multiple of 4")
    c = c.reshape(*c.shape[:-1], -1, 4)
    w = c[..., 0] | (c[..., 1] << 6) | (c[..., 2] << 12) | (c[..., 3] << 18)
    b = np.stack([w & 0xFF, (w >> 8) & 0xFF, (w >> 16) & 0xFF], axis=-1)
    return b.reshape(*b.shape[:-2], -1).astype(np.uint8)


def unpack(packed) -> np.ndarray:
    """Bytes [..., 3n] → 6-bit codes [..., 4n] (inverse of pack)."""
    b = np.asarray(packed, dtype=np.uint32)
    if b.shape[-1] % 3:
        raise ValueError("the byte count must be a multiple of 3")
    b = b.reshape(*b.shape[:-1], -1, 3)
    w = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16)
    c = np.stack([(w >> (6 * k)) & 0x3F for k in range(4)], axis=-1)
    return c.reshape(*c.shape[:-2], -1).astype(np.uint8)


def bytes_per_token(d: int = 576) -> int:
    """Packed codes plus the group scales of one cached token of d elements."""
    return d * CODE_BITS // 8 + (d // GROUP) * 4
