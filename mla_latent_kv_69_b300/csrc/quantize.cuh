// Per-token e4m3 quantisation of one 576-element bf16 cache row by one warp:
// scale = amax/448 (1 for a zero row), code = e4m3(x / scale) with an IEEE fp32 division
// and the round-to-nearest, saturating hardware conversion. The pages only say the
// served cache is low-bit ("DeepSeek-V2 机制拆解", §推理参数与 128K 上下文的使用注意);
// this is the stand-in format.
#pragma once
#include "common.cuh"

namespace mla {

__device__ __forceinline__ void quantize_row_e4m3(const __nv_bfloat16* __restrict__ row, uint8_t* __restrict__ codes,
                                                  float* __restrict__ scale_out, int lane) {
  const __nv_bfloat162* src = reinterpret_cast<const __nv_bfloat162*>(row);
  float2 x[kRow / 64];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < kRow / 64; ++k) {
    x[k] = __bfloat1622float2(src[k * 32 + lane]);
    amax = fmaxf(amax, fmaxf(fabsf(x[k].x), fabsf(x[k].y)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint16_t* dst = reinterpret_cast<uint16_t*>(codes);
#pragma unroll
  for (int k = 0; k < kRow / 64; ++k) {
    const float2 y = make_float2(__fdiv_rn(x[k].x, scale), __fdiv_rn(x[k].y, scale));
    dst[k * 32 + lane] = (uint16_t)__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
  }
  if (lane == 0) *scale_out = scale;
}

}  // namespace mla
