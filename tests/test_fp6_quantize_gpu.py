"""mla_quantize_fp6 against the oracle's e2m3 codec (oracle/fp6_e2m3.py), bit for bit:
the packed bytes and the block scale bytes of seeded bf16 rows with blocks of very
different magnitudes (down to bf16 subnormals), all-zero blocks, negative zeros and
values that fall exactly on the rounding ties."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import bits_to_torch_bf16
from oracle import fp6_e2m3 as F6

pytestmark = pytest.mark.gpu


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 576)) * rng.choice([1e-39, 1e-20, 1e-2, 1.0, 30.0, 1e30], size=(n, 18)).repeat(32, axis=1)
    x[0, 64:96] = 0.0                                       # an all-zero block
    x[1, :64] = -0.0                                        # negative zeros
    # two blocks whose scale is exactly 1 (amax 7.5) holding every tie of the e2m3 grid
    grid = np.array(sorted({k / 8 for k in range(16)} | {k / 4 for k in range(8, 16)} | {k / 2 for k in range(8, 16)}))
    ties = (grid[1:] + grid[:-1]) / 2
    g = np.zeros(64)
    g[0] = g[32] = 7.5
    g[1:32] = ties
    g[33:64] = -ties
    x[2, 128:192] = g
    return W.f32_to_bf16_bits(x.astype(np.float32))


def test_quantize_fp6_bit_exact(cuda_device):
    bits = _rows(3000, 66)
    rows = bits_to_torch_bf16(bits, cuda_device)
    packed, scales = mla.quantize_fp6(rows)
    torch.cuda.synchronize()
    x = W.bf16_bits_to_f32(bits)
    codes, ref_scales = F6.quantize_blocks(x)
    np.testing.assert_array_equal(scales.cpu().numpy(), ref_scales)
    np.testing.assert_array_equal(packed.cpu().numpy(), F6.pack(codes))
    # the tie blocks have scale 1 (byte 127) and decode to the oracle's even choices
    assert ref_scales[2, 4] == 127 and ref_scales[2, 5] == 127
    np.testing.assert_array_equal(F6.unpack(packed[2].cpu().numpy())[128:192], codes[2, 128:192])


def test_quantize_fp6_empty_and_one_row(cuda_device):
    rows = torch.zeros(0, 576, dtype=torch.bfloat16, device=cuda_device)
    packed, scales = mla.quantize_fp6(rows)
    assert packed.shape == (0, 432) and scales.shape == (0, 18)
    bits = _rows(3, 67)[2:3]
    packed, scales = mla.quantize_fp6(bits_to_torch_bf16(bits, cuda_device))
    torch.cuda.synchronize()
    codes, ref_scales = F6.quantize_blocks(W.bf16_bits_to_f32(bits))
    np.testing.assert_array_equal(packed.cpu().numpy(), F6.pack(codes))
    np.testing.assert_array_equal(scales.cpu().numpy(), ref_scales)
