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
// weights and of the tokens' hidden states through a TMA ring that holds all of them at
// once where they fit (d = 5120: up to 80 new tokens) into tcgen05
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
constexpr int kMaxStages = 12;
constexpr int kBoxBytes = 128 * 128;          // 128 weight rows x 64 bf16 (one 128B-swizzled K chunk)
constexpr int kPPad = 4;                      // fp32 of padding per row of the partial
constexpr int kBarBytes = 256;
constexpr int kSmemMax = 232448;
constexpr uint64_t kWaitNs = 2000000000ull;

// Shared memory: a ring of `stages` stages (the K chunk's weights, then its hidden
// states: hrows token rows of 128 bytes), then the barriers. The fp32 partial reuses the
// ring once the MMAs are done. Enough stages that every K chunk of the CTA is in flight
// at once when they fit.
struct Ring {
  int hrows, stage, stages, bar_off, smem;
};
Ring ring_for(int T, int nch) {
  Ring r;
  r.hrows = T >= kNT ? kNT : ((T + 15) & ~15);
  r.stage = kBoxBytes + r.hrows * 128;
  const int cap = (kSmemMax - kBarBytes) / r.stage;
  r.stages = nch < cap ? nch : cap;
  if (r.stages > kMaxStages) r.stages = kMaxStages;
  const int ring = r.stages * r.stage, part = 128 * (r.hrows + kPPad) * 4;
  r.bar_off = ((ring > part ? ring : part) + 1023) & ~1023;
  r.smem = r.bar_off + kBarBytes;
  return r;
}

struct AppendParams {
  const int32_t* seq_ids;       // [T]
  const int32_t* pos;           // [T]
  __nv_bfloat16* rows;          // bf16 cache rows (written), or nullptr when staging
  __nv_bfloat16* staging;       // [T, 576] for an e4m3 cache, else nullptr
  const int32_t* block_table;   // [num_seqs, max_pages] or nullptr (contiguous)
  int32_t hrows, stage, stages, bar_off;   // the Ring of this launch
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
  const int stages = p.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);   // [stages] full, [stages] empty, MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (2 * kMaxStages + 1));
  volatile int* ok_word = reinterpret_cast<volatile int*>(smem + p.bar_off + 8 * (2 * kMaxStages + 1) + 4);
  // the 128B swizzle needs 1024-byte aligned stages; the layout is the same in every CTA
  const bool aligned = (smem_u32(smem) & 1023u) == 0;
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * stages; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[2 * kMaxStages], 1);
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
        const int s = c % stages;
        if (c >= stages && !mbar_wait(&bars[stages + s], (uint32_t)(((c / stages) - 1) & 1), &never, kWaitNs)) {
          ok = false;
          break;
        }
        unsigned char* st = smem + s * p.stage;
        mbar_arrive_expect_tx(&bars[s], wbytes + (uint32_t)p.hrows * 128u);
        tma_load_2d(st, wmap, &bars[s], k0 + 64 * c, wrow0, pol_w);
        tma_load_2d(st + kBoxBytes, &h_map, &bars[s], k0 + 64 * c, t0, pol_h);
      }
      if (!ok) {
        record_status(p.status, MLA_ERR_TIMEOUT);
        *ok_word = 0;
      }
      // loads still in flight land before their stage is reused or the CTA leaves
      for (int i = c > stages ? c - stages : 0; i < c; ++i)
        mbar_wait(&bars[i % stages], (uint32_t)((i / stages) & 1), &never, kWaitNs);
    } else if (warp == 1 && lane == 0) {
      // ---- out[j, t] += W[j, k] h[t, k]: 4 MMAs of 128 x N x 16 per K chunk ----
      const uint32_t idesc = idesc_f16(128, N, false, false, false);
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const int s = c % stages;
        if (!mbar_wait(&bars[s], (uint32_t)((c / stages) & 1), &never, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t wa = smem_u32(smem + s * p.stage), hb = wa + kBoxBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, sdesc_sw128(wa + 32 * kk, 16, 1024), sdesc_sw128(hb + 32 * kk, 16, 1024), idesc,
                 (c | kk) ? 1u : 0u);
        mma_commit(&bars[stages + s]);
      }
      if (!ok) {
        record_status(p.status, MLA_ERR_TIMEOUT);
        *ok_word = 0;
      }
      mma_commit(&bars[2 * kMaxStages]);   // arrives once every MMA issued above is complete
    }
  }

  // ---- the CTA's fp32 partial: TMEM lane j (weight row), column n (token) → P[j][n],
  // rows of hrows + 4 floats ----
  const int PS = p.hrows + kPPad;
  float* P = reinterpret_cast<float*>(smem);
  if (aligned) {
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bars[2 * kMaxStages], 0, &never, kWaitNs));
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
        for (int v = 0; v < 8; ++v)
          if (c0 + 4 * v < N)
            reinterpret_cast<float4*>(P + (32 * warp + lane) * PS + c0)[v] =
                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]), __uint_as_float(r[4 * v + 2]),
                            __uint_as_float(r[4 * v + 3]));
      }
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's partial is in its shared memory (release / acquire)

  // ---- sum the cluster's 8 partials of this CTA's rows over distributed shared memory
  // (rank order, so the result does not depend on timing), rotate the key, round to
  // bf16, write. Thread (g, u): warp g, tokens 4u .. 4u + 3; a warp's loads of one row
  // are 512 contiguous bytes. Latent tiles: rows 16 r + 4 g .. + 3; the key tile: the
  // pair (i, i + 32), i = 4 r + g ----
  bool all_ok = true;
  const uint32_t ok_addr = smem_u32(smem + p.bar_off + 8 * (2 * kMaxStages + 1) + 4);
  for (int q = 0; q < kSplit; ++q) all_ok = all_ok && ld_cluster_u32(mapa(ok_addr, q)) != 0u;
  const int u = lane, g = warp;
  if (all_ok && 4 * u < nt) {
    int64_t rows[4];
    __nv_bfloat16* dst[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + 4 * u + k;
      rows[k] = 4 * u + k < nt ? dest_row(p, t) : -2;
      if (rows[k] == -1) record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
      dst[k] = rows[k] < 0 ? nullptr : (p.staging ? p.staging + (int64_t)t * kRow : p.rows + rows[k] * kRow);
    }
    const uint32_t pbase = smem_u32(P) + (uint32_t)(4 * u) * 4u;
    if (mt < 4) {   // latent columns 128 mt + 16 r + 4 g .. + 3
      const int j0 = 16 * (int)rank + 4 * g;
      float4 x[kSplit][4];
#pragma unroll
      for (int q = 0; q < kSplit; ++q)
#pragma unroll
        for (int v = 0; v < 4; ++v) x[q][v] = ld_cluster_v4_f32(mapa(pbase + (uint32_t)((j0 + v) * PS) * 4u, q));
      float acc[4][4];   // [row][token]
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
#pragma unroll
        for (int q = 0; q < kSplit; ++q) {
          acc[v][0] += x[q][v].x; acc[v][1] += x[q][v].y; acc[v][2] += x[q][v].z; acc[v][3] += x[q][v].w;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!dst[k]) continue;
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0][k], acc[1][k]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2][k], acc[3][k]);
        *reinterpret_cast<uint2*>(dst[k] + 128 * mt + j0) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      }
    } else {        // the RoPE pair (i, i + 32)
      const int i = 4 * (int)rank + g;
      float4 x[kSplit], y[kSplit];
#pragma unroll
      for (int q = 0; q < kSplit; ++q) {
        x[q] = ld_cluster_v4_f32(mapa(pbase + (uint32_t)(i * PS) * 4u, q));
        y[q] = ld_cluster_v4_f32(mapa(pbase + (uint32_t)((i + kRope / 2) * PS) * 4u, q));
      }
      float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kSplit; ++q) {
        a[0] += x[q].x; a[1] += x[q].y; a[2] += x[q].z; a[3] += x[q].w;
        b[0] += y[q].x; b[1] += y[q].y; b[2] += y[q].z; b[3] += y[q].w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!dst[k]) continue;
        float sn, cs;
        rope_sincos(p.pos[t0 + 4 * u + k], turns.f[i], &sn, &cs);
        dst[k][kLatent + i] = __float2bfloat16_rn(a[k] * cs - b[k] * sn);
        dst[k][kLatent + kRope / 2 + i] = __float2bfloat16_rn(b[k] * cs + a[k] * sn);
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
                                const int32_t* seq_ids, const int32_t* pos, int T, int d, const RopeSpec& rope,
                                const mla_cache& cache, int num_seqs, __nv_bfloat16* staging, int32_t* status,
                                cudaStream_t st) {
  const Ring ring = ring_for(T, d / kSplit / 64);
  CUtensorMap wdkv_map, wkr_map, h_map;
  if (!row_map(w_dkv, kLatent, d, 128, &wdkv_map) || !row_map(w_kr, kRope, d, kRope, &wkr_map) ||
      !row_map(h, T, d, ring.hrows, &h_map))
    return cudaErrorInvalidValue;
  AppendParams p{};
  p.hrows = ring.hrows;
  p.stage = ring.stage;
  p.stages = ring.stages;
  p.bar_off = ring.bar_off;
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
  cudaError_t e = smem_attr_once(cache_append_kernel, kSmemMax, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(cache_append_kernel, dim3(kMTiles * kSplit, (unsigned)ceil_div(T, kNT)), dim3(kThreads),
                        ring.smem, st, wdkv_map, wkr_map, h_map, p, rope_turns(rope));
  if (e != cudaSuccess || !fp8) return e;
  return launch_overlapped(append_quantize_kernel, dim3((unsigned)ceil_div(T, kQuantWarps)), dim3(kQuantWarps * 32),
                           0, st, p, static_cast<uint8_t*>(const_cast<void*>(cache.data)),
                           const_cast<float*>(cache.scales));
}

}  // namespace mla
