// mla_up_v: o[b,h,:] = W_UV[h] · o_lat[b,h,:]  (W_UV applied after the latent-space
// weighted sum; "DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈).
#include "common.cuh"

namespace mla {
namespace {

constexpr int kUpBT = 16;          // batch rows per block (W_UV[h] rows reused across them)
constexpr int kUpWarps = 8;

__global__ void __launch_bounds__(kUpWarps * 32)
up_v_simt(const float* __restrict__ o_lat, const __nv_bfloat16* __restrict__ w_uv, int B, int n_h,
          float* __restrict__ o) {
  __shared__ float2 os[kUpBT][kLatent / 2];
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kUpBT;
  const int nb = min(kUpBT, B - b0);
  for (int i = threadIdx.x; i < kUpBT * (kLatent / 2); i += blockDim.x) {
    int bi = i / (kLatent / 2), j = i % (kLatent / 2);
    os[bi][j] = bi < nb ? reinterpret_cast<const float2*>(o_lat + ((int64_t)(b0 + bi) * n_h + h) * kLatent)[j]
                        : make_float2(0.f, 0.f);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int d = warp; d < kNope; d += kUpWarps) {
    const __nv_bfloat162* wrow =
        reinterpret_cast<const __nv_bfloat162*>(w_uv + ((int64_t)h * kNope + d) * kLatent);
    float2 w[kLatent / 64];
#pragma unroll
    for (int k = 0; k < kLatent / 64; ++k) w[k] = __bfloat1622float2(wrow[k * 32 + lane]);
    for (int bi = 0; bi < nb; ++bi) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < kLatent / 64; ++k) {
        float2 v = os[bi][k * 32 + lane];
        acc = fmaf(w[k].x, v.x, acc);
        acc = fmaf(w[k].y, v.y, acc);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) o[((int64_t)(b0 + bi) * n_h + h) * kNope + d] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_up_v(const float* o_lat, const __nv_bfloat16* w_uv, int B, int n_h, float* o,
                        cudaStream_t st) {
  dim3 grid(n_h, ceil_div(B, kUpBT));
  up_v_simt<<<grid, kUpWarps * 32, 0, st>>>(o_lat, w_uv, B, n_h, o);
  return cudaGetLastError();
}

}  // namespace mla
