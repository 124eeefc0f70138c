"""The e4m3 tensor-core kernel turns each cache code into an f16 operand by moving bits:
sign to bit 15, the low seven bits (four exponent bits, three mantissa bits) to bits
7..13. The claim stated beside that kernel is that the resulting f16 is exactly 2^-8
times the code's value for every finite code, normal and subnormal alike (the f16
exponent bias exceeds e4m3's by 8, and an e4m3 subnormal lands on an f16 subnormal of
the same scaled value). This checks the claim against the oracle's decoder, which is
written from the format definition; the GPU test test_fp8_every_code_through_tensor_cores
checks the kernel itself."""

import numpy as np

from oracle import fp8_e4m3 as F


def _moved_bits_f16(code: int) -> np.float16:
    bits = ((code & 0x80) << 8) | ((code & 0x7F) << 7)
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


def test_every_finite_code_maps_to_its_value_times_2_pow_minus_8():
    for code in range(256):
        if code & 0x7F == 0x7F:          # the two NaN codes are outside the cache's domain
            continue
        got = float(_moved_bits_f16(code)) * 256.0
        want = F.code_value(code)
        assert got == want, f"code {code:#04x}: {got} != {want}"


def test_subnormal_codes_stay_exact_and_nonzero():
    for code in list(range(1, 8)) + list(range(0x81, 0x88)):
        h = _moved_bits_f16(code)
        assert h != 0 and float(h) * 256.0 == F.code_value(code)
