// mla_up_v: o[b,h,:] = W_UV[h] · o_lat[b,h,:]  (W_UV applied after the latent-space
// weighted sum; "DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈).
//
// Per head a small GEMM with the head dimension as M:
//     o[b, h, d] = sum_j W_UV[h, d, j] o_lat[b, h, j]        (M = 128 d, N = batch, K = 512 j)
// One CTA per (head, tile of up to 32 sequences). All of W_UV[h] (128 KB, a K-major
// operand) is requested by TMA at once, four 32 KB boxes of two 64-column chunks on
// their own barriers. Meanwhile the threads convert the CTA's o_lat rows: the tensor
// core takes bf16, so each fp32 value is split as hi = bf16(x), lo = bf16(x - hi) and
// both halves enter the same MMA as 2 x N columns (W·hi + W·lo carries ~16
// significant bits of o_lat instead of 8). The epilogue adds the two column halves.
// A second instance merges the split partials itself (mla_combine_up_v): the threads form
// each sequence's log-sum-exp weights, then build the operand rows as the weighted sums
// of the slots, so the merge costs no launch and o_lat no round trip through memory.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kNB = 32;                      // sequences per CTA; MMA N = 2 x round16(nb) <= 64
constexpr int kThreads = 256;                // eight warps stage the operand; the epilogue splits the columns
constexpr int kChunks = kLatent / 64;        // 8 K-chunks of 64 j
constexpr int kWBox = 2 * kNope * 128;       // two chunks of W_UV[h]: 128 d rows x 128 j (32 KB)
constexpr int kXChunk = 2 * kNB * 128;       // one chunk of the (hi, lo) rows: up to 64 rows x 64 j (8 KB)
constexpr int OFF_W = 0;                     // four boxes = all of W_UV[h]
constexpr int OFF_X = 4 * kWBox;             // eight chunks
constexpr int kMaxFusedSlots = MLA_MAX_SPLITS;   // the merge's weights: kNB sequences x every slot (32 KB)
constexpr int OFF_CW = OFF_X + kChunks * kXChunk;
constexpr int OFF_BAR = OFF_CW + kNB * kMaxFusedSlots * 4;
constexpr int kSmem = OFF_BAR + 64;
constexpr uint64_t kWaitNs = 2000000000ull;

// kMerge: the operand is merged from the split partials on the fly (mla_combine's
// log-sum-exp merge) instead of read from o_lat; o_lat and lse are then written as
// by-products when their pointers are given.
template <bool kMerge>
__global__ void __launch_bounds__(kThreads, 1)
up_v_tc(const __grid_constant__ CUtensorMap wmap, const float* __restrict__ o_lat, const float* __restrict__ lse_part,
        int S, int B, int n_h, float* __restrict__ o, float* __restrict__ o_lat_out, float* __restrict__ lse_out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int h = blockIdx.x, b0 = blockIdx.y * kNB;
  const int nb = min(kNB, B - b0);
  const int NP = (nb + 15) & ~15;   // rows [0, NP) hold hi, [NP, 2 NP) lo
  const int N = 2 * NP;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // [0..3] W boxes, [4] X ready, [5] done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 48);
  volatile int* ok_word = reinterpret_cast<volatile int*>(smem + OFF_BAR + 52);
  const bool aligned = (smem_u32(smem) & 1023u) == 0;   // the 128B swizzle needs 1024-byte aligned tiles
  griddep_launch_dependents();

  if (aligned) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
      mbar_init(&bars[4], kThreads);
      mbar_init(&bars[5], 1);
      *ok_word = 1;
      fence_mbar_init_cluster();
    }
    if (warp == 0) {
      tmem_alloc(tmem_slot, 64);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (aligned) {
    const uint32_t tmem = *tmem_slot;
    const volatile int never = 0;
    if (threadIdx.x == 0) {
      const uint64_t pol = l2_policy_evict_first();
      prefetch_tmap(&wmap);
      for (int i = 0; i < 4; ++i) {
        mbar_arrive_expect_tx(&bars[i], kWBox);
        tma_load_3d(smem + OFF_W + i * kWBox, &wmap, &bars[i], 0, h * kNope, 2 * i, pol);
      }
    }
    griddep_wait();   // o_lat (or the partials) come from the previous kernel
    float* cw = reinterpret_cast<float*>(smem + OFF_CW);   // [n][s] merge weights
    if constexpr (kMerge) {
      // per sequence: m = max_s lse_s, w_s = exp(lse_s - m) / sum_s exp(lse_s - m);
      // slots with lse = -inf weigh 0, a sequence without any gives o_lat = 0, lse = -inf
      for (int n = threadIdx.x; n < nb; n += kThreads) {
        const float* lp = lse_part + (int64_t)(b0 + n) * S * n_h + h;
        float m = -INFINITY;
        for (int sl = 0; sl < S; ++sl) m = fmaxf(m, lp[(int64_t)sl * n_h]);
        float z = 0.f;
        for (int sl = 0; sl < S; ++sl) {
          const float l = lp[(int64_t)sl * n_h];
          const float wgt = (m == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - m);
          cw[n * kMaxFusedSlots + sl] = wgt;
          z += wgt;
        }
        const float inv = z > 0.f ? 1.f / z : 0.f;
        for (int sl = 0; sl < S; ++sl) cw[n * kMaxFusedSlots + sl] *= inv;
        if (lse_out) lse_out[(int64_t)(b0 + n) * n_h + h] = z > 0.f ? m + logf(z) : -INFINITY;
      }
      __syncthreads();
    }
    // o_lat rows → bf16 hi/lo rows of every chunk (K-major, 128B swizzle). Item idx is
    // one float4 of a valid row: sequence n = idx / 128, columns 4 (idx % 128) .. +4.
    // Merged, it is the weighted sum over the slots; else the slot is o_lat itself.
    constexpr int kU = 4;                      // items per thread in flight
    constexpr int kS = kMerge ? 4 : 1;         // slots per item in flight
    const int items = nb * 128;
    const int64_t row_stride = (int64_t)S * n_h * kLatent;   // floats from sequence b to b + 1
#pragma unroll 1
    for (int base = threadIdx.x; base < items; base += kThreads * kU) {
      float4 acc[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int s0 = 0; s0 < S; s0 += kS) {
        float4 a[kU][kS];
        float wt[kU][kS];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int idx = base + u * kThreads;
          const int n = idx >> 7;
#pragma unroll
          for (int k = 0; k < kS; ++k) {
            const int sl = s0 + k;
            const bool valid = idx < items && sl < S;
            wt[u][k] = valid ? (kMerge ? cw[n * kMaxFusedSlots + sl] : 1.f) : 0.f;
            a[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (wt[u][k] != 0.f) {
              const float4* src = reinterpret_cast<const float4*>(o_lat + (b0 + n) * row_stride +
                                                                  ((int64_t)sl * n_h + h) * kLatent) +
                                  (idx & 127);
              a[u][k] = kMerge ? __ldcs(src) : *src;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int k = 0; k < kS; ++k) {
            acc[u].x = fmaf(wt[u][k], a[u][k].x, acc[u].x);
            acc[u].y = fmaf(wt[u][k], a[u][k].y, acc[u].y);
            acc[u].z = fmaf(wt[u][k], a[u][k].z, acc[u].z);
            acc[u].w = fmaf(wt[u][k], a[u][k].w, acc[u].w);
          }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = base + u * kThreads;
        if (idx >= items) continue;
        const int n = idx >> 7, f4 = idx & 127;
        if (kMerge && o_lat_out)
          reinterpret_cast<float4*>(o_lat_out + ((int64_t)(b0 + n) * n_h + h) * kLatent)[f4] = acc[u];
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[u].x, acc[u].y);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[u].z, acc[u].w);
        const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
        const __nv_bfloat162 l0 = __floats2bfloat162_rn(acc[u].x - f0.x, acc[u].y - f0.y);
        const __nv_bfloat162 l1 = __floats2bfloat162_rn(acc[u].z - f1.x, acc[u].w - f1.y);
        // column 4 f4 sits in chunk f4 / 16, 16-byte unit (f4 / 2) % 8, half f4 % 2
        const int c = f4 >> 4, qc = (f4 >> 1) & 7, half = f4 & 1;
        unsigned char* xs = smem + OFF_X + c * kXChunk + 8 * half;
        const int rh = n, rl = NP + n;
        *reinterpret_cast<uint2*>(xs + rh * 128 + ((qc ^ (rh & 7)) << 4)) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
        *reinterpret_cast<uint2*>(xs + rl * 128 + ((qc ^ (rl & 7)) << 4)) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
      }
    }
    // rows nb .. NP - 1 of both halves are zero: (NP - nb) rows x 2 halves x 8 chunks x 128 B
    for (int z = threadIdx.x; z < (NP - nb) * 2 * kChunks * 8; z += kThreads) {
      const int unit = z & 7, c = (z >> 3) & 7, r2 = z >> 6;
      const int r = (r2 >> 1) + nb + ((r2 & 1) ? NP : 0);
      *reinterpret_cast<uint4*>(smem + OFF_X + c * kXChunk + r * 128 + unit * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars[4]);
    if (threadIdx.x == 0) {
      const uint32_t idesc = idesc_f16(128, N, false, false, false);
      bool ok = mbar_wait(&bars[4], 0, &never, kWaitNs);
      for (int c = 0; ok && c < kChunks; ++c) {
        if ((c & 1) == 0) ok = mbar_wait(&bars[c >> 1], 0, &never, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        const uint32_t wt = smem_u32(smem + OFF_W + (c >> 1) * kWBox + (c & 1) * (kNope * 128));
        const uint32_t xt = smem_u32(smem + OFF_X + c * kXChunk);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, sdesc_sw128(wt + 32 * kk, 16, 1024), sdesc_sw128(xt + 32 * kk, 16, 1024), idesc,
                 (c | kk) ? 1u : 0u);
      }
      if (!ok) *ok_word = 0;
      mma_commit(&bars[5]);
      // loads still in flight land before the CTA may leave
      for (int i = 0; i < 4; ++i) mbar_wait(&bars[i], 0, &never, kWaitNs / 4);
    }
    __syncthreads();   // orders ok_word
    // epilogue: lane d holds W_UV[h, d, :] · hi in column n and · lo in column NP + n;
    // warp w reads TMEM lanes 32 (w % 4) .. +32 (its lane quarter), column groups of 16
    // alternating between warps w and w + 4
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bars[5], 0, &never, kWaitNs));
    tc_fence_after();
    if (done && *ok_word) {
      const int quarter = warp & 3;
      const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
      const int d = 32 * quarter + lane;
#pragma unroll 1
      for (int c0 = 16 * (warp >> 2); c0 < NP; c0 += 32) {
        uint32_t rh[16], rl[16];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                     : "=r"(rh[0]), "=r"(rh[1]), "=r"(rh[2]), "=r"(rh[3]), "=r"(rh[4]), "=r"(rh[5]), "=r"(rh[6]),
                       "=r"(rh[7]), "=r"(rh[8]), "=r"(rh[9]), "=r"(rh[10]), "=r"(rh[11]), "=r"(rh[12]), "=r"(rh[13]),
                       "=r"(rh[14]), "=r"(rh[15])
                     : "r"(trow + c0));
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                     : "=r"(rl[0]), "=r"(rl[1]), "=r"(rl[2]), "=r"(rl[3]), "=r"(rl[4]), "=r"(rl[5]), "=r"(rl[6]),
                       "=r"(rl[7]), "=r"(rl[8]), "=r"(rl[9]), "=r"(rl[10]), "=r"(rl[11]), "=r"(rl[12]), "=r"(rl[13]),
                       "=r"(rl[14]), "=r"(rl[15])
                     : "r"(trow + NP + c0));
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x)
          if (c0 + x < nb)
            o[((int64_t)(b0 + c0 + x) * n_h + h) * kNope + d] = __uint_as_float(rh[x]) + __uint_as_float(rl[x]);
      }
    }
    tc_fence_before();
  }
  if (!aligned) griddep_wait();
  __syncthreads();
  tc_fence_after();
  if (aligned && warp == 0) tmem_dealloc(*tmem_slot, 64);
}


// W_UV viewed as (64 j, row n_h*128 + d, 8 chunks of 64 j); box = 128 d rows x two chunks
bool wuv_map(const __nv_bfloat16* w_uv, int n_h, CUtensorMap* wmap) {
  const uint64_t dims[3] = {64, (uint64_t)n_h * kNope, kChunks};
  const uint64_t strides[2] = {(uint64_t)kLatent * 2, 128};
  const uint32_t box[3] = {64, kNope, 2};
  return encode_tiled(tmap_desc(w_uv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      wmap);
}

}  // namespace

cudaError_t launch_up_v(const float* o_lat, const __nv_bfloat16* w_uv, int B, int n_h, float* o,
                        cudaStream_t st) {
  CUtensorMap wmap;
  if (!wuv_map(w_uv, n_h, &wmap)) return cudaErrorInvalidValue;
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t attr_err = smem_attr_once(up_v_tc<false>, kSmem, attr_done);
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(n_h, ceil_div(B, kNB));
  return launch_overlapped(up_v_tc<false>, grid, dim3(kThreads), kSmem, st, wmap, o_lat, (const float*)nullptr, 1, B,
                           n_h, o, (float*)nullptr, (float*)nullptr);
}

cudaError_t launch_combine_up_v(const float* o_part, const float* lse_part, int S, const __nv_bfloat16* w_uv, int B,
                                int n_h, float* o, float* o_lat, float* lse, cudaStream_t st) {
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
  if (S < 1 || S > kMaxFusedSlots) return cudaErrorInvalidValue;
  CUtensorMap wmap;
  if (!wuv_map(w_uv, n_h, &wmap)) return cudaErrorInvalidValue;
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t attr_err = smem_attr_once(up_v_tc<true>, kSmem, attr_done);
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(n_h, ceil_div(B, kNB));
  return launch_overlapped(up_v_tc<true>, grid, dim3(kThreads), kSmem, st, wmap, o_part, lse_part, S, B, n_h, o,
                           o_lat, lse);
}

}  // namespace mla
