// mla_quantize_fp6: bf16 cache rows → the ~6-bit cache format (e2m3 codes in groups of
// 64 elements with one fp32 scale each, four codes packed in three bytes). The pages
// report a cache of about 6 bits per element ("DeepSeek-V2 机制拆解",
// §推理参数与 128K 上下文的使用注意; "DeepSeek-V2 … 中文验证版", §瓶颈) without its
// format; this is the format read for it (include/mla.h, mla_quantize_fp6).
//
// One warp per 576-element row. Lane l holds elements 2l and 2l + 1 of each of the nine
// 64-element groups (one coalesced 4-byte load per group); the group's amax comes from a
// shuffle reduction, scale = amax / 7.5 and y = x / scale are IEEE fp32 divisions, and
// the code is found from y's binade: the e2m3 values are k/8 below 2, k/4 from 2 to 4 and
// k/2 from 4 to 7.5, so y times 8, 4 or 2 (exact) rounded to the nearest integer with
// ties to even is the grid index, and index and code have the same parity.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kFp6Warps = 8;
constexpr int kGroups = kRow / 64;          // nine groups of 64
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
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kFp6Warps + (threadIdx.x >> 5);
  if (r >= n) return;
  const __nv_bfloat162* src = reinterpret_cast<const __nv_bfloat162*>(rows + r * kRow);
  uint8_t* dst = packed + r * kPackedRow;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const float2 x = __bfloat1622float2(src[g * 32 + lane]);
    float amax = fmaxf(fabsf(x.x), fabsf(x.y));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 7.5f) : 1.f;
    const uint32_t c0 = e2m3_code(__fdiv_rn(x.x, scale)), c1 = e2m3_code(__fdiv_rn(x.y, scale));
    // codes 4t .. 4t + 3 of the group sit in lanes 2t (c0, c1) and 2t + 1 (c2, c3)
    const uint32_t pair = c0 | (c1 << 6);
    const uint32_t other = __shfl_xor_sync(0xffffffffu, pair, 1);
    if ((lane & 1) == 0) {
      const uint32_t w = pair | (other << 12);
      uint8_t* o = dst + g * 48 + 3 * (lane >> 1);
      o[0] = (uint8_t)(w & 0xFFu);
      o[1] = (uint8_t)((w >> 8) & 0xFFu);
      o[2] = (uint8_t)((w >> 16) & 0xFFu);
    }
    if (lane == 0) scales[r * kGroups + g] = scale;
  }
}

}  // namespace

}  // namespace mla

extern "C" mla_status mla_quantize_fp6(const void* rows, int64_t num_rows, uint8_t* packed, float* scales,
                                       cudaStream_t stream) {
  if (!rows || !packed || !scales) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(rows) & 15u) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (num_rows < 0 || num_rows > ((int64_t)1 << 33)) return MLA_ERR_INVALID_ARG;
  if (num_rows == 0) return MLA_OK;
  const int64_t blocks = mla::ceil_div64(num_rows, mla::kFp6Warps);
  mla::quantize_fp6_kernel<<<(unsigned)blocks, mla::kFp6Warps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(rows), num_rows, packed, scales);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
