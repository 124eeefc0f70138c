"""Pins for the e4m3 codec of the oracle: checked against torch's float8_e4m3fn
conversion (a library routine) and against properties fixed by the format."""

import numpy as np
import pytest
import torch

from oracle import fp8_e4m3 as F
from workloads import bf16_bits_to_f32


def test_decode_table_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.DECODE_TABLE
    nan_ref, nan_ours = np.isnan(ref), np.isnan(ours)
    np.testing.assert_array_equal(nan_ref, nan_ours)
    np.testing.assert_array_equal(ours[~nan_ours], ref[~nan_ref])
    assert F.DECODE_TABLE[0x7E] == 448.0 and F.DECODE_TABLE[0x01] == 2.0 ** -9


def _torch_encode(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_on_every_bf16_pattern_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bf16_bits_to_f32(bits)
    ok = np.isfinite(x) & (np.abs(x) < 464.0)     # torch does not saturate; above 464 it makes NaN
    np.testing.assert_array_equal(F.encode(x[ok]), _torch_encode(x[ok]))


def test_encode_matches_torch_on_ties_and_random_fp32():
    rng = np.random.default_rng(0)
    # exact midpoints between neighbouring codes (ties) and their fp32 neighbours
    v = F.DECODE_TABLE[:0x7F]
    mid = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    cand = np.concatenate([mid, np.nextafter(mid, 0, dtype=np.float32),
                           np.nextafter(mid, 1e9, dtype=np.float32)])
    cand = np.concatenate([cand, -cand, (rng.standard_normal(200000) * 40).astype(np.float32)])
    cand = cand[np.abs(cand) < 464.0]
    np.testing.assert_array_equal(F.encode(cand), _torch_encode(cand))


def test_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 464.0, 1000.0, 3.0e38, -500.0, np.nan], dtype=np.float32)
    c = F.encode(x)
    assert list(c[:5]) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert c[5] == F.NAN_CODE


def test_quantize_rows_properties():
    rng = np.random.default_rng(1)
    x = bf16_bits_to_f32((rng.standard_normal((64, 576)).astype(np.float32).view(np.uint32) >> 16)
                         .astype(np.uint16))
    codes, scales = F.quantize_rows(x)
    assert scales.dtype == np.float32
    amax = np.max(np.abs(x), axis=1)
    np.testing.assert_array_equal(scales, (amax / np.float32(448)).astype(np.float32))
    # the largest element of each row lands on ±448
    i = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(F.decode(codes[np.arange(64), i])) == 448.0)
    # rounding error bounded by half an e4m3 step: relative 2^-4 for normals,
    # absolute 2^-10·scale in the subnormal range
    deq = F.dequantize_rows(codes, scales)
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scales[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    # zero row
    z_codes, z_scale = F.quantize_rows(np.zeros((1, 576), dtype=np.float32))
    assert z_scale[0] == 1.0 and np.all(z_codes == 0)


@pytest.mark.parametrize("code", [0x00, 0x08, 0x38, 0x7E, 0x80, 0xB5])
def test_code_value_definition(code):
    s, e, m = code >> 7, (code >> 3) & 0xF, code & 7
    expect = ((-1) ** s) * ((1 + m / 8) * 2.0 ** (e - 7) if e else m * 2.0 ** -9)
    assert F.code_value(code) == expect
