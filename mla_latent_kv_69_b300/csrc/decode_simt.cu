// Scalar (CUDA-core, fp32) split-KV decode over the latent cache. It implements every
// convention of mla_decode_fwd (row addressing, splits, masking, e4m3 scales, outputs)
// in the plainest GPU form, and serves the configurations the tensor-core kernel
// does not (mla_decode_kernel reports which one runs).
//
// Per block: one (split, sequence, group of 16 heads). Tiles of 32 tokens are staged
// in shared memory as fp32; scores, an online softmax with a running maximum, and
// the latent-space accumulation o += p · c_t run on CUDA cores.
#include "common.cuh"

namespace mla {
namespace {

constexpr int kSimtHeads = 16;
constexpr int kSimtTile = 32;
constexpr int kSimtThreads = 256;
constexpr int kPad = kRow + 1;   // 577: conflict-free column walks

struct SimtSmem {
  float q[kSimtHeads][kPad];
  float c[kSimtTile][kPad];
  float p[kSimtHeads][kSimtTile];
  float m[kSimtHeads];
  float l[kSimtHeads];
  float corr[kSimtHeads];
  int valid[kSimtTile];
};

__device__ inline float load_elem_bf16(const void* data, int64_t row, int col) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(data)[row * kRow + col]);
}

__global__ void __launch_bounds__(kSimtThreads)
decode_simt_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int s = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * kSimtHeads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = max(p.seq_lens[b], 0);
  int st, en;
  split_range(L, p.S, s, &st, &en);

  for (int i = tid; i < kSimtHeads * kRow; i += kSimtThreads) {
    int hh = i / kRow, d = i % kRow;
    sm.q[hh][d] = __bfloat162float(p.q_lat[((int64_t)b * p.n_h + h0 + hh) * kRow + d]);
  }
  if (tid < kSimtHeads) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  const int hh = tid / 16;           // head owned in the accumulation phase
  const int dlane = tid % 16;        // dims dlane + 16k
  float acc[kLatent / 16];
#pragma unroll
  for (int k = 0; k < kLatent / 16; ++k) acc[k] = 0.f;
  __syncthreads();

  for (int t0 = st; t0 < en; t0 += kSimtTile) {
    // Stage up to 32 rows; each warp takes rows warp, warp+8, ...
    for (int r = warp; r < kSimtTile; r += kSimtThreads / 32) {
      const int t = t0 + r;
      int64_t row = -1;
      if (t < en) {
        row = cache_row(p, b, t);
        if (row < 0) record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
      }
      float sc = 1.f;
      if (row >= 0 && p.kv_dtype == MLA_KV_FP8_E4M3) sc = p.scales[row];
      for (int d = lane; d < kRow; d += 32) {
        float v = 0.f;
        if (row >= 0) {
          if (p.kv_dtype == MLA_KV_BF16) {
            v = load_elem_bf16(p.data, row, d);
          } else {
            const __nv_fp8_storage_t code = reinterpret_cast<const uint8_t*>(p.data)[row * kRow + d];
            v = __half2float(__half(__nv_cvt_fp8_to_halfraw(code, __NV_E4M3))) * sc;
          }
        }
        sm.c[r][d] = v;
      }
      if (lane == 0) sm.valid[r] = row >= 0;
    }
    __syncthreads();

    // Scores: thread → head tid/16, tokens tid%16 and tid%16 + 16.
    {
      const int sh = tid / 16;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = (tid % 16) + 16 * half;
        float a = 0.f;
        for (int d = 0; d < kRow; ++d) a = fmaf(sm.q[sh][d], sm.c[r][d], a);
        sm.p[sh][r] = sm.valid[r] ? a * p.scale : -INFINITY;
      }
    }
    __syncthreads();

    // Online softmax, one thread per head.
    if (tid < kSimtHeads) {
      float mt = -INFINITY;
      for (int r = 0; r < kSimtTile; ++r) mt = fmaxf(mt, sm.p[tid][r]);
      const float m_old = sm.m[tid];
      const float m_new = fmaxf(m_old, mt);
      float corr = 1.f, sum = 0.f;
      if (m_new == -INFINITY) {
        for (int r = 0; r < kSimtTile; ++r) sm.p[tid][r] = 0.f;
      } else {
        corr = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
        for (int r = 0; r < kSimtTile; ++r) {
          const float e = expf(sm.p[tid][r] - m_new);
          sm.p[tid][r] = e;
          sum += e;
        }
        sm.m[tid] = m_new;
      }
      sm.l[tid] = sm.l[tid] * corr + sum;
      sm.corr[tid] = corr;
    }
    __syncthreads();

    const float corr = sm.corr[hh];
#pragma unroll 4
    for (int k = 0; k < kLatent / 16; ++k) {
      const int d = dlane + 16 * k;
      float a = acc[k] * corr;
      for (int r = 0; r < kSimtTile; ++r) a = fmaf(sm.p[hh][r], sm.c[r][d], a);
      acc[k] = a;
    }
    __syncthreads();
  }

  const int h = h0 + hh;
  const float l = sm.l[hh];
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* out = p.o_part + (((int64_t)b * p.S + s) * p.n_h + h) * kLatent;
#pragma unroll
  for (int k = 0; k < kLatent / 16; ++k) out[dlane + 16 * k] = acc[k] * inv;
  if (dlane == 0) {
    p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] = l > 0.f ? sm.m[hh] + logf(l) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams& p, cudaStream_t st) {
  const int smem = (int)sizeof(SimtSmem);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.S, p.B, p.n_h / kSimtHeads);
  decode_simt_kernel<<<grid, kSimtThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
