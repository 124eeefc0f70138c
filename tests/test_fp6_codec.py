"""Pins of the e2m3 codec, block quantiser and 3-byte packing (oracle/fp6_e2m3.py)
against the format's definition, stated here independently of the oracle's code:
the positive e2m3 values are three grids (k/8 below 2, k/4 from 2 to 4, k/2 from 4 to
7.5), the sign bit negates, encoding is nearest-with-ties-to-even by brute force over
that grid, a block's shared exponent is floor(log2 amax) - 2 (math.frexp), and the
packing is a little-endian 24-bit word per four codes."""

import numpy as np
import pytest

from oracle import fp6_e2m3 as F

# the positive values by their grids, not by the bit fields
GRID = np.array(sorted({k / 8 for k in range(16)} | {k / 4 for k in range(8, 16)} | {k / 2 for k in range(8, 16)}))


def test_positive_values_are_the_three_grids():
    assert len(GRID) == 32
    np.testing.assert_array_equal(F.DECODE_TABLE[:32], GRID)


def test_sign_bit_negates():
    np.testing.assert_array_equal(F.DECODE_TABLE[32:], -GRID)
    assert np.signbit(F.DECODE_TABLE[32])   # -0


@pytest.mark.parametrize("code,value", [(0b001000, 1.0), (0b011111, 7.5), (0b000001, 0.125), (0b010100, 3.0),
                                        (0b111011, -5.5), (0b000111, 0.875), (0b101001, -1.125)])
def test_code_value_definition(code, value):
    assert F.code_value(code) == value


def test_encode_roundtrips_every_value():
    codes = np.arange(64, dtype=np.uint8)
    np.testing.assert_array_equal(F.encode(F.DECODE_TABLE.astype(np.float32)), codes)


def _brute(x):
    """Nearest grid value by exhaustive search; ties to the even grid index; saturate."""
    a = abs(float(x))
    d = np.abs(GRID - a)
    best = np.flatnonzero(d == d.min())
    k = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]
    return np.copysign(GRID[k], x)


def test_encode_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(6)
    mids = (GRID[1:] + GRID[:-1]) / 2
    xs = np.concatenate([rng.uniform(-9, 9, 4000), mids, -mids, GRID, [7.75, 8.0, 1e6, -1e6]]).astype(np.float32)
    got = F.decode(F.encode(xs))
    want = np.array([_brute(x) for x in xs])
    np.testing.assert_array_equal(got, want)


def test_ties_go_to_the_even_code():
    assert F.encode(np.float32(0.0625)) == 0          # between codes 0 and 1
    assert F.encode(np.float32(0.1875)) == 2          # between codes 1 and 2
    assert F.encode(np.float32(1.9375)) == 0b010000   # between 1.875 (odd code 15) and 2.0 (code 16)
    assert F.encode(np.float32(7.25)) == 0b011110     # between 7.0 (code 30) and 7.5 (code 31)


def test_saturates_and_rejects_non_finite():
    np.testing.assert_array_equal(F.decode(F.encode(np.array([100.0, -100.0, 7.75], np.float32))), [7.5, -7.5, 7.5])
    with pytest.raises(ValueError):
        F.encode(np.array([np.nan], np.float32))


def test_quantize_blocks_properties():
    import math
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((5, 576)) * rng.choice([1e-30, 1e-3, 1.0, 30.0, 1e30], size=(5, 18)).repeat(32, axis=1))
    x[2, 64:96] = 0.0                                  # an all-zero block
    x = x.astype(np.float32)
    codes, sbytes = F.quantize_blocks(x)
    assert codes.shape == (5, 576) and sbytes.shape == (5, 18) and sbytes.dtype == np.uint8
    g = x.reshape(5, 18, 32).astype(np.float64)
    for t in range(5):
        for b in range(18):
            amax = float(np.abs(g[t, b]).max())
            if amax == 0:
                assert sbytes[t, b] == 127 and np.all(codes[t, 32 * b:32 * b + 32] & 0x1F == 0)
                continue
            m, e = math.frexp(amax)                    # amax = m 2^e, m in [0.5, 1)
            se = e - 1 - 2
            assert sbytes[t, b] == se + 127
            assert 4.0 <= amax / 2.0 ** se < 8.0
    # every element within half a grid step of its binade, or saturated at 7.5 X
    X = 2.0 ** (sbytes.astype(np.float64) - 127)[..., None]
    back = F.dequantize_blocks(codes, sbytes).reshape(5, 18, 32)
    y = np.abs(g / X)
    half = np.where(y < 2, 1 / 16, np.where(y < 4, 1 / 8, 1 / 4))
    err = np.abs(back - g) / X
    sat = y > 7.5
    assert np.all(err[~sat] <= half[~sat])
    assert np.all(np.abs(err[sat] - (y[sat] - 7.5)) <= 1e-12)


def test_pack_bit_layout():
    np.testing.assert_array_equal(F.pack(np.array([1, 2, 3, 4])), [0x81, 0x30, 0x10])
    np.testing.assert_array_equal(F.pack(np.array([63, 63, 63, 63])), [0xFF, 0xFF, 0xFF])
    np.testing.assert_array_equal(F.pack(np.array([0, 0, 0, 63])), [0x00, 0x00, 0xFC])
    np.testing.assert_array_equal(F.pack(np.array([63, 0, 0, 0])), [0x3F, 0x00, 0x00])
    np.testing.assert_array_equal(F.pack(np.array([0, 63, 0, 0])), [0xC0, 0x0F, 0x00])


def test_pack_roundtrip_and_sizes():
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 64, size=(3, 576)).astype(np.uint8)
    packed = F.pack(codes)
    assert packed.shape == (3, 432)
    np.testing.assert_array_equal(F.unpack(packed), codes)


def test_bytes_per_token_and_the_pages_6bit_arithmetic():
    assert F.bytes_per_token() == 432 + 18
    # [B] §瓶颈: 128K tokens x 60 layers of (512 + 64) elements at 6 bits is about 3.4 GB
    codes_only = 131072 * 60 * 576 * 6 / 8
    assert abs(codes_only / 1e9 - 3.4) < 0.01
