"""e2m3 (6-bit float) codec, its block quantiser and the 3-byte packing of the ~6-bit
cache reading, from the format definitions.

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

Blocks (the published microscaling layout for 6-bit elements, MXFP6 E2M3): each cached
token's 576 elements form eighteen blocks of 32 consecutive elements; block b shares
one power-of-two scale X_b = 2^(floor(log2 amax_b) - 2), the 2 being the exponent of
e2m3's largest value (7.5 = 1.875 · 2^2), stored as the 8-bit biased exponent
(E8M0: byte = exponent + 127, clamped to 0..254); an all-zero block gets X = 1. Each
element's code is encode(x / X); x / X is exact (a power of two) and lies in [0, 8), so
only elements above 7.5 · X saturate. Power-of-two block scales are what the tensor
cores' block-scaled 8/6/4-bit MMA applies inside the K reduction; a per-token scale
(the e4m3 stand-in) can be pulled out of QK^T, a per-block one cannot. Encoding rounds
to the nearest value, ties to the even code (even mantissa), and saturates at ±7.5;
inputs are finite (cache rows are bf16 values).

Packing: four consecutive codes c0..c3 of a token form the 24-bit little-endian word
c0 | c1 << 6 | c2 << 12 | c3 << 18, stored as its three bytes in order; a token is 432
bytes of codes plus eighteen scale bytes, 450 bytes in all against 580 for the e4m3
codes with one fp32 scale per token.
"""

from __future__ import annotations

import numpy as np

E2M3_MAX = 7.5
E2M3_EMAX = 2          # exponent of the largest e2m3 value
BLOCK = 32
CODE_BITS = 6
SCALE_BIAS = 127


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


def block_exponents(x) -> np.ndarray:
    """x [T, D] fp32 → the shared exponent of each 32-element block, floor(log2 amax) - 2,
    clamped to -127..127 (0 for an all-zero block), as int64 [T, D/32]."""
    x = np.asarray(x, dtype=np.float32)
    T, D = x.shape
    if D % BLOCK:
        raise ValueError("the row length must be a multiple of 32")
    amax = np.max(np.abs(x.reshape(T, D // BLOCK, BLOCK)), axis=-1).astype(np.float64)
    _, e = np.frexp(amax)                   # amax = f · 2^e with f in [0.5, 1): floor(log2 amax) = e - 1
    se = np.clip(e.astype(np.int64) - 1 - E2M3_EMAX, -SCALE_BIAS, SCALE_BIAS)
    return np.where(amax > 0, se, 0)


def quantize_blocks(x):
    """x [T, D] (fp32 values, D a multiple of 32) → (codes uint8 [T, D], scale bytes uint8 [T, D/32]).

    code = encode(x · 2^-se) for the block's shared exponent se; scale byte = se + 127.
    """
    x = np.asarray(x, dtype=np.float32)
    T, D = x.shape
    se = block_exponents(x)
    y = np.ldexp(x.reshape(T, D // BLOCK, BLOCK), (-se)[..., None].astype(np.int32)).astype(np.float32)
    return encode(y).reshape(T, D), (se + SCALE_BIAS).astype(np.uint8)


def dequantize_blocks(codes, scale_bytes) -> np.ndarray:
    """Inverse of quantize_blocks in fp64: value = decode(code) · 2^(byte - 127) of its block."""
    codes = np.asarray(codes, dtype=np.uint8)
    T, D = codes.shape
    x = 2.0 ** (np.asarray(scale_bytes, dtype=np.float64) - SCALE_BIAS)
    v = decode(codes).reshape(T, D // BLOCK, BLOCK) * x[..., None]
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
    """Packed codes plus the block scale bytes of one cached token of d elements."""
    return d * CODE_BITS // 8 + d // BLOCK
