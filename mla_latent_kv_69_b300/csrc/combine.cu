// mla_combine: log-sum-exp merge of split-KV partials. For a partition of one
// sequence's tokens into splits with normalised outputs o_s and log-normalisers
// lse_s: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s. Empty splits
// (lse_s = -inf) weigh 0.
#include "common.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(128)
combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int B, int S,
               int n_h, float* __restrict__ o_lat, float* __restrict__ lse_out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const float* lp = lse_part + (int64_t)b * S * n_h + h;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lp[(int64_t)s * n_h]);
  float4* out = reinterpret_cast<float4*>(o_lat + ((int64_t)b * n_h + h) * kLatent);
  if (m == -INFINITY) {
    out[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_out && threadIdx.x == 0) lse_out[(int64_t)b * n_h + h] = -INFINITY;
    return;
  }
  float z = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < S; ++s) {
    const float l = lp[(int64_t)s * n_h];
    if (l == -INFINITY) continue;
    const float w = __expf(l - m);
    z += w;
    const float4 v = reinterpret_cast<const float4*>(
        o_part + (((int64_t)b * S + s) * n_h + h) * kLatent)[threadIdx.x];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const float inv = 1.f / z;
  out[threadIdx.x] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse_out && threadIdx.x == 0) lse_out[(int64_t)b * n_h + h] = m + logf(z);
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int S, int n_h,
                           float* o_lat, float* lse, cudaStream_t st) {
  dim3 grid(n_h, B);
  combine_kernel<<<grid, kLatent / 4, 0, st>>>(o_part, lse_part, B, S, n_h, o_lat, lse);
  return cudaGetLastError();
}

}  // namespace mla
