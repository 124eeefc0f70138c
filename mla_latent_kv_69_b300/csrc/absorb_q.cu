// mla_absorb_q: q_lat[b,h] = [ W_UK[h]^T q^C[b,h] ‖ RoPE(q^R[b,h], pos[b]) ].
// "DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈 (W_UK folded into the
// query side) and §解耦 RoPE 与 YaRN (the 64-wide decoupled query carries position).
//
// Per head the absorbed query is a small GEMM with the latent dimension as M:
//     q_lat[b, h, j] = sum_d W_UK[h, d, j] q^C[b, h, d]      (M = 512 j, N = batch, K = 128 d)
// One CTA per (head, tile of up to 128 sequences, 128-row M-tile): the call is a single
// short wave whose time is each CTA's load latency, so the weights are spread over four
// times as many CTAs as heads. The query tile, shared memory and TMEM are sized for the
// batch (N sequences, a multiple of 16), so that up to four CTAs fit on an SM and the
// 4 n_h CTAs of a small batch run in one wave. The 32 KB M-tile of W_UK[h] (an MN-major
// operand: j is contiguous) and the batch tile of q^C arrive by TMA; tcgen05 accumulates
// one 128 x N fp32 tile in TMEM and the epilogue rounds it to bf16. The weight bytes
// dominate: W_UK is read from HBM once per call.
//
// The decoupled part is rotated on CUDA cores with the exactly reduced angles of
// rope.cuh.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"
#include "rope.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kNB = 128;                     // at most this many sequences per CTA (the MMA N)
constexpr int kThreads = 128;
constexpr int kWTile = 2 * 128 * 128;        // one M-tile of W_UK[h]: two 64-j chunks x 128 d rows (32 KB)
constexpr int kMTiles = 4;                   // 512 latent dims = four 128-row M-tiles, one per CTA
constexpr int OFF_W = 0;                     // this CTA's M-tile
constexpr int OFF_Q = kWTile;                // q^C tile: two 64-d chunks x nbox rows x 128 B
constexpr int kBarBytes = 64;                // barriers, TMEM slot and flag after the q^C tile
constexpr int kSmemMax = OFF_Q + 2 * kNB * 128 + kBarBytes;

// rows of the q^C box (and MMA N bound) for a batch of B: a multiple of 16, at most kNB
inline int q_box_rows(int B) { return B >= kNB ? kNB : ((B + 15) & ~15); }
// TMEM columns for N <= nbox accumulator columns: a power of two, at least 32
inline int tmem_cols_for(int nbox) {
  int c = 32;
  while (c < nbox) c <<= 1;
  return c;
}
constexpr uint64_t kWaitNs = 2000000000ull;

__global__ void __launch_bounds__(kThreads, 2)
absorb_q_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap qmap,
            const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ pos, int B, int n_h, int nbox,
            int tcols, const RopeTurns turns, __nv_bfloat16* __restrict__ q_lat) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int h = blockIdx.x, b0 = blockIdx.y * nbox, mt = blockIdx.z;
  const int nb = min(nbox, B - b0);
  const int N = (nb + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int off_bar = OFF_Q + 2 * nbox * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off_bar);   // [0] W M-tile, [1] q tile, [2] MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_bar + 48);
  volatile int* ok_word = reinterpret_cast<volatile int*>(smem + off_bar + 52);
  const bool aligned = (smem_u32(smem) & 1023u) == 0;   // the 128B swizzle needs 1024-byte aligned tiles
  griddep_launch_dependents();

  if (aligned) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
      *ok_word = 0;
      fence_mbar_init_cluster();
    }
    if (warp == 0) {
      tmem_alloc(tmem_slot, (uint32_t)tcols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (aligned) {
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
      const uint64_t pol = l2_policy_evict_first();
      prefetch_tmap(&qmap);
      prefetch_tmap(&wmap);
      // the weights do not depend on the previous kernel
      mbar_arrive_expect_tx(&bars[0], kWTile);
      tma_load_3d(smem + OFF_W, &wmap, &bars[0], 0, h * kNope, 2 * mt, pol);
      griddep_wait();
      mbar_arrive_expect_tx(&bars[1], 2 * nbox * 128);
      tma_load_4d(smem + OFF_Q, &qmap, &bars[1], 0, h, b0, 0, pol);
      const uint32_t idesc = idesc_f16(128, N, false, /*a_mn=*/true, /*b_mn=*/false);
      const volatile int never = 0;
      bool ok = mbar_wait(&bars[1], 0, &never, kWaitNs) && mbar_wait(&bars[0], 0, &never, kWaitNs);
      if (ok) {
        tc_fence_after();
        const uint32_t wt = smem_u32(smem + OFF_W);
        const uint32_t qt = smem_u32(smem + OFF_Q);
#pragma unroll
        for (int kk = 0; kk < kNope / 16; ++kk) {
          // A: 16 d rows of 128 B (64 j) per 64-j chunk, chunks 16 KB apart; B: q rows, K-major
          const uint64_t a = sdesc_sw128(wt + kk * 2048, 128 * 128, 1024);
          const uint64_t bq = sdesc_sw128(qt + (kk >> 2) * (nbox * 128) + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem, a, bq, idesc, kk > 0 ? 1u : 0u);
        }
      }
      *ok_word = ok ? 1 : 0;
      mma_commit(&bars[2]);
      // loads still in flight land before the CTA may leave
      mbar_wait(&bars[1], 0, &never, kWaitNs / 4);
      mbar_wait(&bars[0], 0, &never, kWaitNs / 4);
    }

    griddep_wait();   // q and pos may come from the previous kernel; q_lat may still be read by it
    // decoupled query, overlapping the tensor-core work: thread (n, g) rotates pairs
    // 8g .. 8g+7 of sequence n; every load of a pass is issued before any math. The four
    // CTAs of a head share the batch tile's sequences, 32 at a time.
#pragma unroll 1
    for (int n0 = (kThreads / 4) * mt; n0 < nb; n0 += kMTiles * (kThreads / 4)) {
      const int n = n0 + (threadIdx.x >> 2), g = threadIdx.x & 3;
      if (n < nb) {
        const int64_t row = (int64_t)(b0 + n) * n_h + h;
        const uint4 u1 = *reinterpret_cast<const uint4*>(q + row * kQ + kNope + 8 * g);
        const uint4 u2 = *reinterpret_cast<const uint4*>(q + row * kQ + kNope + kRope / 2 + 8 * g);
        const int ps = pos[b0 + n];
        const __nv_bfloat162* x1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&u2);
        uint32_t o1[4], o2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a1 = __bfloat1622float2(x1[e]), a2 = __bfloat1622float2(x2[e]);
          float r1[2], r2[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int i = 8 * g + 2 * e + k;
            float sn, cs;
            rope_sincos(ps, turns.f[i], &sn, &cs);
            const float y1 = k ? a1.y : a1.x, y2 = k ? a2.y : a2.x;
            r1[k] = y1 * cs - y2 * sn;
            r2[k] = y2 * cs + y1 * sn;
          }
          const __nv_bfloat162 v1 = __floats2bfloat162_rn(r1[0], r1[1]);
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(r2[0], r2[1]);
          o1[e] = *reinterpret_cast<const uint32_t*>(&v1);
          o2[e] = *reinterpret_cast<const uint32_t*>(&v2);
        }
        __nv_bfloat16* out = q_lat + row * kRow + kLatent;
        *reinterpret_cast<uint4*>(out + 8 * g) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *reinterpret_cast<uint4*>(out + kRope / 2 + 8 * g) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
      }
    }

    __syncthreads();   // orders ok_word

    // epilogue: lane j of M-tile mt holds q_lat[b0 + n, h, 128 mt + j] in column n
    const volatile int never = 0;
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bars[2], 0, &never, kWaitNs));
    tc_fence_after();
    if (done && *ok_word) {
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
      const int j = 128 * mt + 32 * warp + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        MLA_TMEM_LD32(trow + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (c0 + x < nb)
            q_lat[((int64_t)(b0 + c0 + x) * n_h + h) * kRow + j] = __float2bfloat16_rn(__uint_as_float(r[x]));
      }
    }
    tc_fence_before();
  }
  if (!aligned) griddep_wait();
  __syncthreads();
  tc_fence_after();
  if (aligned && warp == 0) tmem_dealloc(*tmem_slot, (uint32_t)tcols);
}

}  // namespace

cudaError_t launch_absorb_q(const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const int32_t* pos,
                            int B, int n_h, const RopeSpec& rope, __nv_bfloat16* q_lat, cudaStream_t st) {
  // W_UK viewed as (64 j, row n_h*128 + d, 8 chunks of 64 j); box = one M-tile (2 chunks)
  CUtensorMap wmap, qmap;
  {
    const uint64_t dims[3] = {64, (uint64_t)n_h * kNope, kLatent / 64};
    const uint64_t strides[2] = {(uint64_t)kLatent * 2, 128};
    const uint32_t box[3] = {64, kNope, 2};
    if (!encode_tiled(tmap_desc(w_uk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      &wmap))
      return cudaErrorInvalidValue;
  }
  // q viewed as (64 d, head, sequence, 64-d chunk); box = one head, nbox sequences, q^C's 2 chunks
  const int nbox = q_box_rows(B);
  {
    const uint64_t dims[4] = {64, (uint64_t)n_h, (uint64_t)B, 3};
    const uint64_t strides[3] = {(uint64_t)kQ * 2, (uint64_t)n_h * kQ * 2, 128};
    const uint32_t box[4] = {64, 1, (uint32_t)nbox, 2};
    if (!encode_tiled(tmap_desc(q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      &qmap))
      return cudaErrorInvalidValue;
  }
  const RopeTurns turns = rope_turns(rope);
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t attr_err = smem_attr_once(absorb_q_tc, kSmemMax, attr_done);
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(n_h, ceil_div(B, nbox), kMTiles);
  const int smem = OFF_Q + 2 * nbox * 128 + kBarBytes;
  return launch_overlapped(absorb_q_tc, grid, dim3(kThreads), smem, st, wmap, qmap, q, pos, B, n_h, nbox,
                           tmem_cols_for(nbox), turns, q_lat);
}

}  // namespace mla
