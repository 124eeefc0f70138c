// mla_absorb_q: q_lat[b,h] = [ W_UK[h]^T q^C[b,h] ‖ RoPE(q^R[b,h], pos[b]) ].
// "DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈 (W_UK folded into the
// query side) and §解耦 RoPE 与 YaRN (the 64-wide decoupled query carries position).
#include "common.cuh"

namespace mla {
namespace {

constexpr int kAbsorbBT = 16;       // batch rows sharing one pass over W_UK[h]
constexpr int kAbsorbThreads = 256; // 2 output columns per thread → 512

__global__ void __launch_bounds__(kAbsorbThreads)
absorb_q_simt(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ w_uk,
              const int32_t* __restrict__ pos, int B, int n_h, float rope_base,
              __nv_bfloat16* __restrict__ q_lat) {
  __shared__ float qs[kAbsorbBT][kNope];
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kAbsorbBT;
  const int nb = min(kAbsorbBT, B - b0);
  for (int i = threadIdx.x; i < kAbsorbBT * kNope; i += blockDim.x) {
    int bi = i / kNope, d = i % kNope;
    qs[bi][d] = bi < nb ? __bfloat162float(q[((int64_t)(b0 + bi) * n_h + h) * kQ + d]) : 0.f;
  }
  __syncthreads();

  const int c = threadIdx.x * 2;
  float acc[kAbsorbBT][2];
#pragma unroll
  for (int bi = 0; bi < kAbsorbBT; ++bi) acc[bi][0] = acc[bi][1] = 0.f;
  const __nv_bfloat162* w =
      reinterpret_cast<const __nv_bfloat162*>(w_uk + (int64_t)h * kNope * kLatent + c);
  for (int d = 0; d < kNope; ++d) {
    float2 wv = __bfloat1622float2(w[d * (kLatent / 2)]);
#pragma unroll
    for (int bi = 0; bi < kAbsorbBT; ++bi) {
      acc[bi][0] = fmaf(qs[bi][d], wv.x, acc[bi][0]);
      acc[bi][1] = fmaf(qs[bi][d], wv.y, acc[bi][1]);
    }
  }
#pragma unroll
  for (int bi = 0; bi < kAbsorbBT; ++bi) {
    if (bi < nb) {
      *reinterpret_cast<__nv_bfloat162*>(q_lat + ((int64_t)(b0 + bi) * n_h + h) * kRow + c) =
          __floats2bfloat162_rn(acc[bi][0], acc[bi][1]);
    }
  }

  // Decoupled query: rotate-half pairs (i, i+32), angle pos * base^(-i/32). The angle
  // and its sine/cosine are taken in fp64: positions reach 131071 rad on pair 0.
  if (threadIdx.x < kRope / 2) {
    const int i = threadIdx.x;
    const double inv_freq = pow((double)rope_base, -2.0 * i / (double)kRope);
    for (int bi = 0; bi < nb; ++bi) {
      const int b = b0 + bi;
      double sn, cs;
      sincos((double)pos[b] * inv_freq, &sn, &cs);
      const __nv_bfloat16* qr = q + ((int64_t)b * n_h + h) * kQ + kNope;
      const double x1 = __bfloat162float(qr[i]);
      const double x2 = __bfloat162float(qr[i + kRope / 2]);
      __nv_bfloat16* out = q_lat + ((int64_t)b * n_h + h) * kRow + kLatent;
      out[i] = __float2bfloat16_rn((float)(x1 * cs - x2 * sn));
      out[i + kRope / 2] = __float2bfloat16_rn((float)(x2 * cs + x1 * sn));
    }
  }
}

}  // namespace

cudaError_t launch_absorb_q(const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const int32_t* pos,
                            int B, int n_h, float rope_base, __nv_bfloat16* q_lat, cudaStream_t st) {
  dim3 grid(n_h, ceil_div(B, kAbsorbBT));
  absorb_q_simt<<<grid, kAbsorbThreads, 0, st>>>(q, w_uk, pos, B, n_h, rope_base, q_lat);
  return cudaGetLastError();
}

}  // namespace mla
