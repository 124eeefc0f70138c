// mla_combine: log-sum-exp merge of split-KV partials. For a partition of one
// sequence's tokens into splits with normalised outputs o_s and log-normalisers
// lse_s: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s. Empty splits
// (lse_s = -inf) weigh 0.
//
// One warp per (sequence, head): each lane owns 16 of the 512 latent values (four
// float4, strided so that a warp load is 512 contiguous bytes); the split loop is
// unrolled so that several splits' loads are in flight together.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int B, int S, int n_h,
               float* __restrict__ o_lat, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * kWarps + (threadIdx.x >> 5), b = blockIdx.y;
  griddep_launch_dependents();
  griddep_wait();   // the partials come from the previous kernel
  if (h >= n_h) return;
  const float* lp = lse_part + (int64_t)b * S * n_h + h;
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lp[(int64_t)s * n_h]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float4* out = reinterpret_cast<float4*>(o_lat + ((int64_t)b * n_h + h) * kLatent);
  if (m == -INFINITY) {
#pragma unroll
    for (int k = 0; k < 4; ++k) out[lane + 32 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_out && lane == 0) lse_out[(int64_t)b * n_h + h] = -INFINITY;
    return;
  }
  float z = 0.f;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t sstride = (int64_t)n_h * kLatent / 4;   // float4 per split
  const float4* src = reinterpret_cast<const float4*>(o_part + ((int64_t)b * S * n_h + h) * kLatent) + lane;
  constexpr int kU = 4;
  for (int s0 = 0; s0 < S; s0 += kU) {
    float w[kU];
    float4 v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int s = s0 + u;
      const float l = s < S ? lp[(int64_t)s * n_h] : -INFINITY;
      w[u] = l == -INFINITY ? 0.f : __expf(l - m);
      if (w[u] != 0.f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = src[s * sstride + 32 * k];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      z += w[u];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = fmaf(w[u], v[u][k].x, acc[k].x);
        acc[k].y = fmaf(w[u], v[u][k].y, acc[k].y);
        acc[k].z = fmaf(w[u], v[u][k].z, acc[k].z);
        acc[k].w = fmaf(w[u], v[u][k].w, acc[k].w);
      }
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out[lane + 32 * k] = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
  if (lse_out && lane == 0) lse_out[(int64_t)b * n_h + h] = m + logf(z);
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int S, int n_h,
                           float* o_lat, float* lse, cudaStream_t st) {
  dim3 grid(ceil_div(n_h, kWarps), B);
  return launch_overlapped(combine_kernel, grid, dim3(kWarps * 32), 0, st, o_part, lse_part, B, S, n_h, o_lat, lse);
}

}  // namespace mla
