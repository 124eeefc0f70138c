// mla_quantize_fp6: bf16 cache rows → the ~6-bit cache format (e2m3 codes in blocks of
// 32 elements sharing one power-of-two scale byte, four codes packed in three bytes). The pages
// report a cache of about 6 bits per element ("DeepSeek-V2 机制拆解",
// §推理参数与 128K 上下文的使用注意; "DeepSeek-V2 … 中文验证版", §瓶颈) without its
// format; this is the format read for it (include/mla.h, mla_quantize_fp6).
//
// One warp per 576-element row. Lane l holds elements 2l and 2l + 1 of each 64-element
// slice (one coalesced 4-byte load per slice), so lanes 0-15 hold one 32-element block
// and lanes 16-31 the next. A block's amax comes from a shuffle reduction over its 16
// lanes; its shared exponent is floor(log2 amax) - 2, read from amax's exponent field
// (clamped to -127..127; 0 for an all-zero block), and y = x · 2^-exponent is exact. The
// code is found from y's binade: the e2m3 values are k/8 below 2, k/4 from 2 to 4 and
// k/2 from 4 to 7.5, so y times 8, 4 or 2 (exact) rounded to the nearest integer with
// ties to even is the grid index, and index and code have the same parity.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kFp6Warps = 8;
constexpr int kSlices = kRow / 64;          // nine 64-element slices, two blocks each
constexpr int kBlocks = kRow / 32;          // eighteen 32-element blocks
constexpr int kPackedRow = kRow * 6 / 8;    // 432 bytes

__device__ __forceinline__ uint32_t e2m3_code(float y) {
  const uint32_t sgn = (__float_as_uint(y) >> 31) << 5;
  const float a = fabsf(y);
  uint32_t mag;
  if (a >= 7.5f) {
    mag = 31u;                                         // saturate at 7.5
  } else if (a < 2.f) {
    mag = (uint32_t)__float2int_rn(a * 8.f);           // k/8, k = 0..16 (16 is 2.0, code 16)
  } else if (a < 4.f) {
    mag = (uint32_t)__float2int_rn(a * 4.f) + 8u;      // k/4, k = 8..16 → codes 16..24
  } else {
    mag = (uint32_t)__float2int_rn(a * 2.f) + 16u;     // k/2, k = 8..15 → codes 24..31
  }
  return sgn | mag;
}

__global__ void __launch_bounds__(kFp6Warps * 32)
quantize_fp6_kernel(const __nv_bfloat16* __restrict__ rows, int64_t n, uint8_t* __restrict__ packed,
                    uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kFp6Warps + (threadIdx.x >> 5);
  if (r >= n) return;
  const __nv_bfloat162* src = reinterpret_cast<const __nv_bfloat162*>(rows + r * kRow);
  uint8_t* dst = packed + r * kPackedRow;
#pragma unroll
  for (int g = 0; g < kSlices; ++g) {
    const float2 x = __bfloat1622float2(src[g * 32 + lane]);
    float amax = fmaxf(fabsf(x.x), fabsf(x.y));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xFFu);   // 0 for zero and subnormal amax
    const int se = amax > 0.f ? max(-127, min(127, ebits - 127 - 2)) : 0;
    // se <= 254 - 129 = 125, so 2^-se has the exponent field 127 - se in 2..254: a normal fp32
    const float inv = __uint_as_float((uint32_t)(127 - se) << 23);
    const uint32_t c0 = e2m3_code(__fmul_rn(x.x, inv)), c1 = e2m3_code(__fmul_rn(x.y, inv));
    // codes 4t .. 4t + 3 of the slice sit in lanes 2t (c0, c1) and 2t + 1 (c2, c3)
    const uint32_t pair = c0 | (c1 << 6);
    const uint32_t other = __shfl_xor_sync(0xffffffffu, pair, 1);
    if ((lane & 1) == 0) {
      const uint32_t w = pair | (other << 12);
      uint8_t* o = dst + g * 48 + 3 * (lane >> 1);
      o[0] = (uint8_t)(w & 0xFFu);
      o[1] = (uint8_t)((w >> 8) & 0xFFu);
      o[2] = (uint8_t)((w >> 16) & 0xFFu);
    }
    if ((lane & 15) == 0) scales[r * kBlocks + 2 * g + (lane >> 4)] = (uint8_t)(se + 127);
  }
}

}  // namespace

}  // namespace mla

extern "C" mla_status mla_quantize_fp6(const void* rows, int64_t num_rows, uint8_t* packed, uint8_t* scales,
                                       cudaStream_t stream) {
  if (!rows || !packed || !scales) return MLA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(rows) & 15u) return MLA_ERR_INVALID_ARG;
  if (num_rows < 0 || num_rows > ((int64_t)1 << 33)) return MLA_ERR_INVALID_ARG;
  if (num_rows == 0) return MLA_OK;
  const int64_t blocks = mla::ceil_div64(num_rows, mla::kFp6Warps);
  mla::quantize_fp6_kernel<<<(unsigned)blocks, mla::kFp6Warps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(rows), num_rows, packed, scales);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
