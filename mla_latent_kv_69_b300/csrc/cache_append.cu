// mla_cache_append: the cache rows of new tokens.
//     c_KV[t] = W_DKV h[t]                      (512: the down-projected latent)
//     k^R[t]  = RoPE(W_KR h[t], pos[t])         (64: the shared key, turned at its own position)
//     row[t]  = bf16([c_KV[t] ‖ k^R[t]]) at token pos[t] of sequence seq[t]
// "DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈 (each token's hidden state is
// down-projected to the cached latent, d_c = 512) and §解耦 RoPE 与 YaRN (the decoupled
// shared key is what carries the position, so it is rotated when it is made).
//
// The projection is one GEMM with the 576 weight rows as M and the new tokens as N:
//     out[j, t] = sum_k W[j, k] h[t, k]        (M: four 128-row tiles of W_DKV and the
//                                              64 rows of W_KR; N: up to 128 tokens; K: d)
// With a decode step's few hundred tokens the work is the weight stream (576·d bf16 read
// once), so K is split over a cluster of 8 CTAs: every CTA streams 1/8 of one M-tile's
// weights and of the tokens' hidden states through a 4-stage TMA ring into tcgen05
// MMAs, each CTA's fp32 partial goes from TMEM to its shared memory, and after a cluster
// barrier CTA r of the cluster sums the 8 partials of its 16 rows (or 4 RoPE pairs)
// over distributed shared memory, rotates, rounds to bf16 and writes the rows. For an
// e4m3 cache the rows go to the caller's staging buffer and a second kernel quantises
// them per token into the cache (quantize.cuh).
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "quantize.cuh"
#include "rope.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kSplit = 8;                     // CTAs of a cluster, one K slice each
constexpr int kMTiles = 5;                    // 4 x 128 rows of W_DKV, then W_KR's 64 rows
constexpr int kNT = 128;                      // tokens per CTA (the MMA N, padded to 16)
constexpr int kThreads = 128;
constexpr int kStages = 4;
constexpr int kBoxBytes = 128 * 128;          // 128 rows x 64 bf16 (one 128B-swizzled K chunk)
constexpr int kStage = 2 * kBoxBytes;         // weights + hidden states of one K chunk
constexpr int kPStride = 132;                 // fp32 per token in the partial (4 words of padding)
constexpr int OFF_BAR = kStages * kStage;     // the partial reuses the ring once the MMAs are done
constexpr int kSmem = OFF_BAR + 128;
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(kNT * kPStride * 4 <= OFF_BAR, "the partial fits in the ring");

struct AppendParams {
  const int32_t* seq_ids;       // [T]
  const int32_t* pos;           // [T]
  __nv_bfloat16* rows;          // bf16 cache rows (written), or nullptr when staging
  __nv_bfloat16* staging;       // [T, 576] for an e4m3 cache, else nullptr
  const int32_t* block_table;   // [num_seqs, max_pages] or nullptr (contiguous)
  int64_t seq_stride;           // contiguous: rows between sequences
  int64_t num_rows;             // rows of the cache
  int32_t max_pages, num_seqs;
  int32_t T, d;
  int32_t* status;
};

// Cache row of new token t, or -1 (recorded as MLA_ERR_DEVICE_BOUNDS by the caller)
// when its sequence, position or page falls outside the cache.
__device__ __forceinline__ int64_t dest_row(const AppendParams& p, int t) {
  const int seq = p.seq_ids[t], pos = p.pos[t];
  if (seq < 0 || seq >= p.num_seqs || pos < 0) return -1;
  if (!p.block_table) {
    if (pos >= p.seq_stride) return -1;
    const int64_t row = (int64_t)seq * p.seq_stride + pos;
    return row < p.num_rows ? row : -1;
  }
  if ((pos >> 6) >= p.max_pages) return -1;
  const int page = p.block_table[(int64_t)seq * p.max_pages + (pos >> 6)];
  if (page < 0 || (int64_t)page * 64 >= p.num_rows) return -1;
  return (int64_t)page * 64 + (pos & 63);
}

__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kThreads, 1)
cache_append_kernel(const __grid_constant__ CUtensorMap wdkv_map, const __grid_constant__ CUtensorMap wkr_map,
                    const __grid_constant__ CUtensorMap h_map, const AppendParams p, const RopeTurns turns) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const int mt = blockIdx.x / kSplit;
  const int t0 = blockIdx.y * kNT;
  const int nt = min(kNT, p.T - t0);
  const int N = (nt + 15) & ~15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);   // [0..3] full, [4..7] empty, [8] MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 80);
  volatile int* ok_word = reinterpret_cast<volatile int*>(smem + OFF_BAR + 84);
  // the 128B swizzle needs 1024-byte aligned stages; the layout is the same in every CTA
  const bool aligned = (smem_u32(smem) & 1023u) == 0;
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * kStages + 1; ++i) mbar_init(&bars[i], 1);
    *ok_word = aligned ? 1 : 0;
    if (!aligned) record_status(p.status, MLA_ERR_UNSUPPORTED);
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kc = p.d / kSplit;        // K of this CTA (a multiple of 64)
  const int nch = kc / 64;
  const int k0 = (int)rank * kc;
  const int wrow0 = mt < 4 ? 128 * mt : 0;
  const uint32_t wbytes = mt < 4 ? kBoxBytes : kBoxBytes / 2;   // W_KR: 64 rows
  const volatile int never = 0;

  if (*ok_word) {
    if (warp == 0 && lane == 0) {
      // ---- TMA producer: K chunk c → stage c % 4 (weights and hidden states) ----
      const uint64_t pol_w = l2_policy_evict_first();   // every weight byte is read once
      const uint64_t pol_h = l2_policy_evict_last();    // the hidden states are read by all 5 M-tiles
      const CUtensorMap* wmap = mt < 4 ? &wdkv_map : &wkr_map;
      prefetch_tmap(wmap);
      prefetch_tmap(&h_map);
      griddep_wait();   // h, seq_ids and pos may come from the previous kernel
      bool ok = true;
      int c = 0;
      for (; c < nch; ++c) {
        const int s = c % kStages;
        if (c >= kStages && !mbar_wait(&bars[kStages + s], (uint32_t)(((c / kStages) - 1) & 1), &never, kWaitNs)) {
          ok = false;
          break;
        }
        unsigned char* st = smem + s * kStage;
        mbar_arrive_expect_tx(&bars[s], wbytes + kBoxBytes);
        tma_load_2d(st, wmap, &bars[s], k0 + 64 * c, wrow0, pol_w);
        tma_load_2d(st + kBoxBytes, &h_map, &bars[s], k0 + 64 * c, t0, pol_h);
      }
      if (!ok) {
        record_status(p.status, MLA_ERR_TIMEOUT);
        *ok_word = 0;
      }
      // loads still in flight land before their stage is reused or the CTA leaves
      for (int i = c > kStages ? c - kStages : 0; i < c; ++i)
        mbar_wait(&bars[i % kStages], (uint32_t)((i / kStages) & 1), &never, kWaitNs);
    } else if (warp == 1 && lane == 0) {
      // ---- out[j, t] += W[j, k] h[t, k]: 4 MMAs of 128 x N x 16 per K chunk ----
      const uint32_t idesc = idesc_f16(128, N, false, false, false);
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const int s = c % kStages;
        if (!mbar_wait(&bars[s], (uint32_t)((c / kStages) & 1), &never, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t wa = smem_u32(smem + s * kStage), hb = wa + kBoxBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, sdesc_sw128(wa + 32 * kk, 16, 1024), sdesc_sw128(hb + 32 * kk, 16, 1024), idesc,
                 (c | kk) ? 1u : 0u);
        mma_commit(&bars[kStages + s]);
      }
      if (!ok) {
        record_status(p.status, MLA_ERR_TIMEOUT);
        *ok_word = 0;
      }
      mma_commit(&bars[2 * kStages]);   // arrives once every MMA issued above is complete
    }
  }

  // ---- the CTA's fp32 partial: TMEM lane j (weight row), column n (token) → P[n][j] ----
  float* P = reinterpret_cast<float*>(smem);
  if (aligned) {
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bars[2 * kStages], 0, &never, kWaitNs));
    tc_fence_after();
    if (!done) {
      if (lane == 0) record_status(p.status, MLA_ERR_TIMEOUT);
      *ok_word = 0;
    } else if (*ok_word) {
      const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t r[32];
        MLA_TMEM_LD32(trow + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (c0 + x < N) P[(c0 + x) * kPStride + 32 * warp + lane] = __uint_as_float(r[x]);
      }
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's partial is in its shared memory (release / acquire)

  // ---- thread i ↔ token t0 + i: sum the cluster's 8 partials of this CTA's rows over
  // distributed shared memory, rotate the key, round to bf16, write ----
  bool all_ok = true;
  for (int q = 0; q < kSplit; ++q) all_ok = all_ok && ld_cluster_u32(mapa(smem_u32(smem + OFF_BAR + 84), q)) != 0u;
  if (all_ok && (int)threadIdx.x < nt) {
    const int t = t0 + threadIdx.x;
    const int64_t row = dest_row(p, t);
    if (row < 0) {
      record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    } else {
      __nv_bfloat16* dst = p.staging ? p.staging + (int64_t)t * kRow : p.rows + row * kRow;
      const uint32_t pbase = smem_u32(P) + (uint32_t)(threadIdx.x * kPStride) * 4u;
      if (mt < 4) {   // latent columns 128 mt + 16 r .. + 15
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll 1
        for (int q = 0; q < kSplit; ++q) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 x = ld_cluster_v4_f32(mapa(pbase + (uint32_t)(16 * rank + 4 * v) * 4u, q));
            acc[4 * v] += x.x; acc[4 * v + 1] += x.y; acc[4 * v + 2] += x.z; acc[4 * v + 3] += x.w;
          }
        }
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
          w[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        uint4* o = reinterpret_cast<uint4*>(dst + 128 * mt + 16 * rank);
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
      } else {        // RoPE pairs (i, i + 32), i = 4 r .. 4 r + 3
        float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int q = 0; q < kSplit; ++q) {
          const float4 x = ld_cluster_v4_f32(mapa(pbase + (uint32_t)(4 * rank) * 4u, q));
          const float4 y = ld_cluster_v4_f32(mapa(pbase + (uint32_t)(32 + 4 * rank) * 4u, q));
          a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
          b[0] += y.x; b[1] += y.y; b[2] += y.z; b[3] += y.w;
        }
        const int ps = p.pos[t];
        float r1[4], r2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float sn, cs;
          rope_sincos(ps, turns.f[4 * rank + e], &sn, &cs);
          r1[e] = a[e] * cs - b[e] * sn;
          r2[e] = b[e] * cs + a[e] * sn;
        }
        const __nv_bfloat162 u0 = __floats2bfloat162_rn(r1[0], r1[1]), u1 = __floats2bfloat162_rn(r1[2], r1[3]);
        const __nv_bfloat162 v0 = __floats2bfloat162_rn(r2[0], r2[1]), v1 = __floats2bfloat162_rn(r2[2], r2[3]);
        *reinterpret_cast<uint2*>(dst + kLatent + 4 * rank) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&u0), *reinterpret_cast<const uint32_t*>(&u1));
        *reinterpret_cast<uint2*>(dst + kLatent + kRope / 2 + 4 * rank) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&v0), *reinterpret_cast<const uint32_t*>(&v1));
      }
    }
  }
  cluster_sync();   // no CTA leaves while the others read its partial
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// e4m3 cache: one warp per new token quantises its staged bf16 row into the cache.
constexpr int kQuantWarps = 8;

__global__ void __launch_bounds__(kQuantWarps * 32)
append_quantize_kernel(const AppendParams p, uint8_t* __restrict__ codes, float* __restrict__ scales) {
  griddep_launch_dependents();
  griddep_wait();   // the staged rows come from the previous kernel
  const int t = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int64_t row = dest_row(p, t);   // an invalid row was recorded by the projection kernel
  if (row < 0) return;
  quantize_row_e4m3(p.staging + (int64_t)t * kRow, codes + row * kRow, scales + row, threadIdx.x & 31);
}

bool row_map(const void* base, int64_t rows, int d, int box_rows, CUtensorMap* map) {
  const uint64_t dims[2] = {(uint64_t)d, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)d * 2};
  const uint32_t box[2] = {64, (uint32_t)box_rows};
  return encode_tiled(tmap_desc(base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      map);
}

}  // namespace

cudaError_t launch_cache_append(const __nv_bfloat16* h, const __nv_bfloat16* w_dkv, const __nv_bfloat16* w_kr,
                                const int32_t* seq_ids, const int32_t* pos, int T, int d, float rope_base,
                                const mla_cache& cache, int num_seqs, __nv_bfloat16* staging, int32_t* status,
                                cudaStream_t st) {
  CUtensorMap wdkv_map, wkr_map, h_map;
  if (!row_map(w_dkv, kLatent, d, 128, &wdkv_map) || !row_map(w_kr, kRope, d, kRope, &wkr_map) ||
      !row_map(h, T, d, kNT, &h_map))
    return cudaErrorInvalidValue;
  AppendParams p{};
  p.seq_ids = seq_ids;
  p.pos = pos;
  const bool fp8 = cache.dtype == MLA_KV_FP8_E4M3;
  p.rows = fp8 ? nullptr : static_cast<__nv_bfloat16*>(const_cast<void*>(cache.data));
  p.staging = fp8 ? staging : nullptr;
  p.block_table = cache.block_table;
  p.seq_stride = cache.seq_stride_tokens;
  p.num_rows = cache.num_rows;
  p.max_pages = cache.max_pages;
  p.num_seqs = num_seqs;
  p.T = T;
  p.d = d;
  p.status = status;
  static std::atomic<int> attr_done[kMaxDevices];
  cudaError_t e = smem_attr_once(cache_append_kernel, kSmem, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(cache_append_kernel, dim3(kMTiles * kSplit, (unsigned)ceil_div(T, kNT)), dim3(kThreads),
                        kSmem, st, wdkv_map, wkr_map, h_map, p, rope_turns(rope_base));
  if (e != cudaSuccess || !fp8) return e;
  return launch_overlapped(append_quantize_kernel, dim3((unsigned)ceil_div(T, kQuantWarps)), dim3(kQuantWarps * 32),
                           0, st, p, static_cast<uint8_t*>(const_cast<void*>(cache.data)),
                           const_cast<float*>(cache.scales));
}

}  // namespace mla
