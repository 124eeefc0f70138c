// Tensor-core split-KV decode over the MLA latent cache (sm_103a: tcgen05 + TMEM + TMA).
//
// With W_UK folded into the query and W_UV applied after the latent-space sum
// ("DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈), all n_h heads of one
// sequence attend over the same 576-wide cache rows, so every tile of tokens is two
// dense contractions with the heads as the M dimension:
//     S[128 x 128] = Q[128 x 576] · C[128 x 576]^T       (scores, fp32 in TMEM)
//     O[128 x 512] += P[128 x 128] · C[128 x 0:512]      (latent output, fp32 in TMEM)
// O alone fills the 512 TMEM columns of an SM, so a work unit (sequence b, split s)
// runs on a cluster of two CTAs that exchange only P:
//   score CTA (rank 0)  Q (bf16) in TMEM columns 0..287, S in columns 288..415.
//       For each 128-token tile it streams the nine 64-dim column slices of the rows
//       (16 KB each) through a ring of four 3-slice groups, issues S = Q·C^T as 36 MMAs
//       of N = 128, and runs the online softmax on eight warps (two threads per head,
//       64 tokens each). P (bf16) is written to a local staging panel and bulk-copied
//       to the value CTA, one 64-token panel at a time.
//   value CTA (rank 1)  owns the 128 x 512 fp32 O accumulator (all of its TMEM).
//       It reads the c_KV part of the same rows itself (an L2 hit shortly after the
//       score CTA's read; each cache byte comes from HBM once) into a 3-stage ring and
//       issues O += P·V per 64-token step as 8 MMAs of N = 256, V being the cache
//       rows read as an MN-major operand.
// The TMA engine spends a roughly fixed time per box row, so loads use 3D tensor maps
// (64 columns x rows x column chunks) that fetch several 128-byte chunks of each row
// per instruction; the shared-memory image is the same chunk-major 128B-swizzled
// layout as one 2D box per chunk. The value CTA starts loading only once the score
// CTA holds Q (the query load goes first), and its epilogue stages O in swizzled
// shared memory and writes it with 3D TMA stores.
// A tensor-core instruction costs at least ~64 cycles whatever N <= 128, so the score
// side uses N = 128 token tiles; the shared-memory link between the two SMs is narrow
// (~20 B/clk), so only P (16 KB per 64 tokens) crosses it, never fp32 scores.
//
// The running maximum of each head is only raised when a tile exceeds it by 2^8; the
// rare raise is voted across the softmax warps and O rows are rescaled by the value
// CTA before the tile's PV. Every wait is bounded (2 s); on expiry the CTA records
// MLA_ERR_TIMEOUT in the status word, tells the peer to stop, drains its own copies
// and tensor-core work, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "decode_tc.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTile = 128;                 // tokens per score tile (the N of S = Q·C^T)
constexpr int kHalf = 64;                  // tokens per value step (= one page)
constexpr int kBox = 64 * 128;             // one TMA box: 64 rows x 64 bf16 (128 B rows, 128B swizzle)
constexpr int kSlice = 2 * kBox;           // one column slice of a score tile: 128 rows x 64 dims
constexpr int kGroup = 3 * kSlice;         // score ring slot: three slices (one TMA instruction)
constexpr int kRing = 4;
constexpr int kCStages = 3;
constexpr int kCStage = 8 * kBox;          // value stage: 64 rows x 512 dims
constexpr int kPanel = 128 * 128;          // P for 64 tokens: 128 heads x 64 bf16
constexpr int kHdr = 512 + 16;             // 128 fp32 rescale factors and a flag word (with panel 0)
constexpr int kFinBytes = 128 * 2 * 4;     // final (m, l) per head
constexpr int kThreads = 320;              // warp 0 TMA, warp 1 MMA, warps 2..9 row warps
constexpr uint64_t kWaitNs = kDecodeWaitNs;
constexpr float kRescaleLog2 = 8.f;

constexpr uint32_t kQCol = 0;              // score CTA TMEM: Q as bf16 pairs (288 columns)
constexpr uint32_t kSCol = 288;            // score CTA TMEM: S (128 columns)
constexpr uint32_t kOCol = 0;              // value CTA TMEM: O (512 columns)

// Shared memory (offsets from the 1024-byte aligned dynamic base).
//   score CTA
constexpr int S_RING = 0;                              // kRing x 48 KB (Q is staged in slots 0..2 first)
constexpr int S_PANEL = S_RING + kRing * kGroup;       // 2 x 16 KB P panels, send side
constexpr int S_HDR = S_PANEL + 2 * kPanel;            // rescale factors + flag sent with panel 0
constexpr int S_MX = S_HDR + 1024;                     // [2 halves][128] fp32: tile maxima, then l halves
constexpr int S_END = S_MX + 2 * 128 * 4;
//   value CTA
constexpr int V_CST = 0;                               // kCStages x 64 KB
constexpr int V_PANEL = V_CST + kCStages * kCStage;    // 2 x 16 KB P panels, receive side; the final (m, l) lands in panel 0
constexpr int V_HDR = V_PANEL + 2 * kPanel;
constexpr int V_END = V_HDR + 1024;
//   both (same offset in both CTAs: remote arrivals and copies address it by offset)
constexpr int OFF_BAR = (S_END > V_END ? S_END : V_END);
enum Bar {
  SB_SLOT_FULL = 0,                       // [kRing] score: slice group landed
  SB_SLOT_EMPTY = SB_SLOT_FULL + kRing,   // [kRing] score: QK MMAs done with the group
  SB_QFULL = SB_SLOT_EMPTY + kRing,       // score: Q landed in slots 0..2
  SB_QREADY = SB_QFULL + 1,               // score: Q copied into TMEM (256)
  SB_SFULL = SB_QREADY + 1,               // score: S written
  SB_SFREE = SB_SFULL + 1,                // score: S read by the softmax threads (256)
  SB_PFREE = SB_SFREE + 1,                // [2] score: the value CTA's PV finished with panel j (remote commit)
  SB_FLUSH = SB_PFREE + 2,                // score MMA warp: all MMAs done
  VB_CFULL = SB_FLUSH + 1,                // [kCStages] value: stage landed
  VB_CEMPTY = VB_CFULL + kCStages,        // [kCStages] value: PV done with the stage
  VB_PFULL = VB_CEMPTY + kCStages,        // [2] value: P panel j received (bulk copy bytes)
  VB_FIN = VB_PFULL + 2,                  // value: final (m, l) received
  VB_FLUSH = VB_FIN + 1,                  // value MMA warp: all MMAs done
  VB_CREQ = VB_FLUSH + 1,                 // value: command for the row warps (1)
  VB_CDONE = VB_CREQ + 1,                 // value: row warps finished it (256)
  VB_GO = VB_CDONE + 1,                   // value: the score CTA holds Q (remote arrival)
  B_COUNT = VB_GO + 1
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;   // tmem base, abort flag, command word, O-initialised flag
constexpr int kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(S_PANEL % 1024 == 0 && V_PANEL % 1024 == 0 && kGroup % 1024 == 0, "swizzle alignment");

enum Cmd { CMD_ZERO = 1, CMD_RESCALE = 2, CMD_DONE = 4 };

__device__ __forceinline__ void give_up(const DecodeParams& p, volatile int* abort_flag, unsigned char* smem,
                                        uint32_t peer) {
  record_status(p.status, MLA_ERR_TIMEOUT);
  *abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(smem + OFF_MISC + 4), peer), 1u);
}

// Slot and use index of score group k (tile k / 3, column chunks 3 (k % 3) .. +2). Q
// occupies slots 0..2 before the first cache group, so group k goes to slot
// (3 + k) % kRing and that slot has held (3 + k) / kRing - [slot < 3] cache groups before.
__device__ __forceinline__ int group_slot(int k) { return (3 + k) % kRing; }
__device__ __forceinline__ int group_prior_uses(int k) {
  const int r = group_slot(k);
  return (3 + k) / kRing - (r < 3 ? 1 : 0);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap smap,
                 const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap omap,
                 float scale_log2) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x >> 1;
  const int b = unit / p.S, s = unit % p.S;
  const int L = max(p.seq_lens[b], 0);
  int st, en;
  split_range(L, p.S, s, &st, &en);
  const int n_tiles = (en - st + kTile - 1) / kTile;
  const int n_halves = 2 * n_tiles;
  griddep_launch_dependents();

  if (n_tiles == 0) {   // empty split: nothing crosses the cluster
    griddep_wait();
    if (rank == 1) {
      float* o = p.o_part + ((int64_t)b * p.S + s) * p.n_h * kLatent;
      for (int i = threadIdx.x; i < p.n_h * kLatent / 4; i += kThreads)
        reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h = threadIdx.x; h < p.n_h; h += kThreads)
        p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] = -INFINITY;
    }
    return;
  }
  if (smem_u32(smem) & 1023u) {   // the 128B swizzle needs 1024-byte aligned slots (same in both CTAs)
    griddep_wait();
    if (threadIdx.x == 0) record_status(p.status, MLA_ERR_UNSUPPORTED);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* cmd_word = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
  volatile int* o_init_word = reinterpret_cast<volatile int*>(smem + OFF_MISC + 12);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *o_init_word = 0;
    for (int k = 0; k < kRing; ++k) {
      mbar_init(&bars[SB_SLOT_FULL + k], 1);
      mbar_init(&bars[SB_SLOT_EMPTY + k], 1);
    }
    mbar_init(&bars[SB_QFULL], 1);
    mbar_init(&bars[SB_QREADY], 256);
    mbar_init(&bars[SB_SFULL], 1);
    mbar_init(&bars[SB_SFREE], 256);
    mbar_init(&bars[SB_PFREE], 1);
    mbar_init(&bars[SB_PFREE + 1], 1);
    mbar_init(&bars[SB_FLUSH], 1);
    for (int k = 0; k < kCStages; ++k) {
      mbar_init(&bars[VB_CFULL + k], 1);
      mbar_init(&bars[VB_CEMPTY + k], 1);
    }
    mbar_init(&bars[VB_PFULL], 1);
    mbar_init(&bars[VB_PFULL + 1], 1);
    mbar_init(&bars[VB_FIN], 1);
    mbar_init(&bars[VB_FLUSH], 1);
    mbar_init(&bars[VB_CREQ], 1);
    mbar_init(&bars[VB_CDONE], 256);
    mbar_init(&bars[VB_GO], 1);
    if (rank == 1) {   // the first tile's P panels and the final message may arrive any time after the cluster sync
      mbar_arrive_expect_tx(&bars[VB_PFULL], kPanel + kHdr);
      mbar_arrive_expect_tx(&bars[VB_PFULL + 1], kPanel);
      mbar_arrive_expect_tx(&bars[VB_FIN], kFinBytes);
    }
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any remote arrival or copy
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (rank == 0) {
    // =============================== score CTA =========================================
    if (warp == 0) {
      if (lane == 0) {
        // ---- TMA producer: Q, then three column slices of a tile per instruction ----
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();   // c_KV is read again by the value CTA
        prefetch_tmap(&smap);
        prefetch_tmap(&qmap);
        const int qrows = p.n_h < 128 ? p.n_h : 128;
        griddep_wait();   // q_lat comes from the previous kernel
        mbar_arrive_expect_tx(&bars[SB_QFULL], 9 * qrows * 128);
        for (int g = 0; g < 3; ++g)
          tma_load_3d(smem + S_RING + g * kGroup, &qmap, &bars[SB_QFULL], 0, b * p.n_h, 3 * g, pol_first);
        const bool paged = p.block_table != nullptr;
        int issued = 0;
        HalfInfo h0{}, h1{};
        int pg0 = page_ahead(p, b, st, 0), pg1 = page_ahead(p, b, st, 1);   // one tile ahead
        for (int k = 0; k < 3 * n_tiles; ++k) {
          const int i = k / 3, g = k % 3;
          const int r = group_slot(k), prior = group_prior_uses(k);
          bool ok = true;
          if (r < 3 && prior == 0) ok = mbar_wait(&bars[SB_QREADY], 0, abort_flag, kWaitNs);
          if (ok && prior > 0) ok = mbar_wait(&bars[SB_SLOT_EMPTY + r], (prior - 1) & 1, abort_flag, kWaitNs);
          if (!ok) {
            give_up(p, abort_flag, smem, peer);
            break;
          }
          if (g == 0) {
            h0 = half_info(p, b, st, en, 2 * i, true, pg0);
            h1 = half_info(p, b, st, en, 2 * i + 1, true, pg1);
            pg0 = page_ahead(p, b, st, 2 * i + 2);
            pg1 = page_ahead(p, b, st, 2 * i + 3);
          }
          unsigned char* dst = smem + S_RING + r * kGroup;
          const uint64_t pol = g < 2 ? pol_last : pol_first;   // chunk 8 (the RoPE key) is read once
          if (!paged) {
            // 128 consecutive rows: one 3D box (the rows past a ragged end are masked)
            if (h0.load) {
              mbar_arrive_expect_tx(&bars[SB_SLOT_FULL + r], kGroup);
              tma_load_3d(dst, &smap, &bars[SB_SLOT_FULL + r], 0, h0.row0, 3 * g, pol);
            } else {
              mbar_arrive(&bars[SB_SLOT_FULL + r]);
            }
          } else {
            // two pages: one 64-row box per page and column chunk (slice c: page 0 rows
            // at +0, page 1 rows at +8 KB)
            const uint32_t bytes = 3 * ((h0.load ? kBox : 0) + (h1.load ? kBox : 0));
            if (bytes) {
              mbar_arrive_expect_tx(&bars[SB_SLOT_FULL + r], bytes);
              for (int c = 0; c < 3; ++c) {
                if (h0.load) tma_load_3d(dst + c * kSlice, &smap, &bars[SB_SLOT_FULL + r], 0, h0.row0, 3 * g + c, pol);
                if (h1.load)
                  tma_load_3d(dst + c * kSlice + kBox, &smap, &bars[SB_SLOT_FULL + r], 0, h1.row0, 3 * g + c, pol);
              }
            } else {
              mbar_arrive(&bars[SB_SLOT_FULL + r]);
            }
          }
          issued = k + 1;
        }
        // Loads still in flight land before the CTA may leave.
        const volatile int never = 0;
        mbar_wait(&bars[SB_QFULL], 0, &never, kWaitNs / 4);
        for (int k = max(0, issued - kRing); k < issued; ++k)
          mbar_wait(&bars[SB_SLOT_FULL + group_slot(k)], group_prior_uses(k) & 1, &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- S = Q · C^T, 36 MMAs of 128 x 128 x 16 per tile ----
        const uint32_t idq = idesc_f16(128, kTile, false, false, false);
        bool ok = mbar_wait(&bars[SB_QREADY], 0, abort_flag, kWaitNs);
        if (ok) mbar_arrive_remote(&bars[VB_GO], 1);   // the value CTA may start its loads
        for (int i = 0; ok && i < n_tiles; ++i) {
          if (i > 0 && !mbar_wait(&bars[SB_SFREE], (i - 1) & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int g = 0; g < 3; ++g) {
            const int k = 3 * i + g, r = group_slot(k);
            if (!mbar_wait(&bars[SB_SLOT_FULL + r], group_prior_uses(k) & 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t base = smem_u32(smem + S_RING + r * kGroup);
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tmem + kSCol, tmem + kQCol + 8 * (4 * (3 * g + c) + kk),
                       sdesc_sw128(base + c * kSlice + 32 * kk, 16, 1024), idq, (g | c | kk) ? 1u : 0u);
            mma_commit(&bars[SB_SLOT_EMPTY + r]);
          }
          if (!ok) break;
          mma_commit(&bars[SB_SFULL]);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[SB_FLUSH]);
        const volatile int never = 0;
        mbar_wait(&bars[SB_FLUSH], 0, &never, kWaitNs);
      }
    } else {
      // ---- softmax: thread (h, j) owns head h, tokens [64 j, 64 j + 64) of each tile ----
      const int q = warp & 3;
      const int h = q * 32 + lane;
      const int j = (warp - 2) >> 2;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      // Q rows → TMEM (packed bf16 pairs; heads beyond n_h are zero)
      if (warp_wait(&bars[SB_QFULL], 0, abort_flag)) {
#pragma unroll 1
        for (int c = j; c < 9; c += 2) {
          uint32_t r[32];
          const unsigned char* row = smem + S_RING + (c / 3) * kGroup + (c % 3) * ((p.n_h < 128 ? p.n_h : 128) * 128) + h * 128;
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const uint4 v = h < p.n_h ? *reinterpret_cast<const uint4*>(row + ((x ^ (h & 7)) << 4))
                                      : make_uint4(0u, 0u, 0u, 0u);
            r[4 * x] = v.x; r[4 * x + 1] = v.y; r[4 * x + 2] = v.z; r[4 * x + 3] = v.w;
          }
          MLA_TMEM_ST32(trow + kQCol + 32 * c, r);
        }
        tmem_wait_st();
      } else {
        give_up(p, abort_flag, smem, peer);
      }
      tc_fence_before();
      mbar_arrive(&bars[SB_QREADY]);

      float m_run = -INFINITY, l_run = 0.f;
      float* mx = reinterpret_cast<float*>(smem + S_MX);
      const uint32_t panel_remote = mapa(smem_u32(smem + V_PANEL + j * kPanel), 1);
      const uint32_t hdr_remote = mapa(smem_u32(smem + V_HDR), 1);
      const uint32_t pfull_remote = mapa(smem_u32(&bars[VB_PFULL + j]), 1);
      // Every thread runs every iteration and every named barrier; after an abort the
      // waits return at once and the tiles are processed as fully masked.
      int pg = page_ahead(p, b, st, j);   // this thread's half of the next tile, fetched ahead
      for (int i = 0; i < n_tiles; ++i) {
        uint32_t sr[64];
        const bool got = warp_wait(&bars[SB_SFULL], i & 1, abort_flag);
        if (got) {
          tc_fence_after();
          MLA_TMEM_LD32(trow + kSCol + 64 * j, sr);
          MLA_TMEM_LD32(trow + kSCol + 64 * j + 32, (sr + 32));
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(&bars[SB_SFREE]);
        const int nv = got ? half_info(p, b, st, en, 2 * i + j, false, pg).nvalid : 0;
        pg = page_ahead(p, b, st, 2 * i + 2 + j);
        // Row maximum on the raw scores (the scale is positive); tokens past the split
        // (ragged tiles only) become -inf so that their weight is exactly 0.
        if (nv < 64) {
#pragma unroll
          for (int t = 0; t < 64; ++t)
            if (t >= nv) sr[t] = __float_as_uint(-INFINITY);
        }
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int t = 8; t < 64; ++t) m8[t & 7] = fmaxf(m8[t & 7], __uint_as_float(sr[t]));
        const float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * scale_log2;
        // Raise the running maximum only when the tile exceeds it by 2^8 (rare); the
        // two threads of a head agree on the new value through shared memory.
        float fac = 1.f;
        bool row_rescale = false;
        const uint32_t nneed = named_popc(1, 256, mt > m_run + kRescaleLog2);
        if (nneed) {   // mx is reused from tile to tile: the vote above orders it
          mx[j * 128 + h] = mt;
          named_sync(1, 256);
          const float mrow = fmaxf(mx[h], mx[128 + h]);
          if (mrow > m_run + kRescaleLog2) {
            if (m_run != -INFINITY) {
              fac = ex2(m_run - mrow);
              row_rescale = true;
            }
            l_run *= fac;
            m_run = mrow;
          }
        }
        const uint32_t nres = nneed ? named_popc(1, 256, row_rescale) : 0u;
        // p = 2^(s * scale - m) as one packed FMA and an SFU exp2 per element; P is
        // rounded to bf16 for the tensor core, l accumulates the fp32 values.
        uint32_t pk[32];
        float lsum = 0.f;
        if (m_run != -INFINITY) {
          const float2 c2 = make_float2(scale_log2, scale_log2);
          const float2 nm2 = make_float2(-m_run, -m_run);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const float2 xy = ffma2(make_float2(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])), c2, nm2);
            const float2 pp = make_float2(ex2(xy.x), ex2(xy.y));
            const __nv_bfloat162 v = __floats2bfloat162_rn(pp.x, pp.y);
            pk[t] = *reinterpret_cast<const uint32_t*>(&v);
            acc[t & 3] = fadd2(acc[t & 3], pp);
          }
          const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
          lsum = (a01.x + a23.x) + (a01.y + a23.y);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) pk[t] = 0u;
        }
        l_run += lsum;
        // The staging panel is free once the value CTA's PV on the previous tile has read it.
        if (i > 0) mbar_wait<true>(&bars[SB_PFREE + j], (i - 1) & 1, abort_flag, kWaitNs);
        unsigned char* stg = smem + S_PANEL + j * kPanel;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(stg + h * 128 + ((c ^ (h & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (j == 0) {
          reinterpret_cast<float*>(smem + S_HDR)[h] = fac;
          if (h == 0) reinterpret_cast<uint32_t*>(smem + S_HDR + 512)[0] = nres;
        }
        fence_proxy_async_smem();
        named_sync(2 + j, 128);
        if (q == 0 && lane == 0 && !*abort_flag) {
          bulk_copy_to_peer(panel_remote, stg, kPanel, pfull_remote);
          if (j == 0) bulk_copy_to_peer(hdr_remote, smem + S_HDR, kHdr, pfull_remote);
        }
      }
      // final (m, l) of each head → the value CTA's panel 0, once its last PV has read it
      named_sync(1, 256);
      mx[j * 128 + h] = l_run;
      named_sync(1, 256);
      if (j == 0) {
        float* fin = reinterpret_cast<float*>(smem + S_PANEL);
        const bool ok = mbar_wait<true>(&bars[SB_PFREE], (n_tiles - 1) & 1, abort_flag, kWaitNs);
        fin[2 * h] = m_run;
        fin[2 * h + 1] = mx[h] + mx[128 + h];
        fence_proxy_async_smem();
        named_sync(2, 128);
        if (q == 0 && lane == 0 && ok && !*abort_flag)
          bulk_copy_to_peer(mapa(smem_u32(smem + V_PANEL), 1), fin, kFinBytes, mapa(smem_u32(&bars[VB_FIN]), 1));
      }
    }
  } else {
    // =============================== value CTA =========================================
    if (warp == 0) {
      if (lane == 0) {
        // ---- TMA producer: c_KV of every 64-token step (evict-first: last reader) ----
        const uint64_t pol = l2_policy_evict_first();
        prefetch_tmap(&vmap);
        int issued = 0;
        // Start once the score CTA has Q: its query load goes first.
        if (!mbar_wait<true>(&bars[VB_GO], 0, abort_flag, kWaitNs)) give_up(p, abort_flag, smem, peer);
        int pg = page_ahead(p, b, st, 0);
        for (int u = 0; u < n_halves && !*abort_flag; ++u) {
          const int sg = u % kCStages;
          if (u >= kCStages &&
              !mbar_wait(&bars[VB_CEMPTY + sg], ((u / kCStages) - 1) & 1, abort_flag, kWaitNs)) {
            give_up(p, abort_flag, smem, peer);
            break;
          }
          const HalfInfo hi = half_info(p, b, st, en, u, false, pg);
          pg = page_ahead(p, b, st, u + 1);
          if (hi.load) {
            mbar_arrive_expect_tx(&bars[VB_CFULL + sg], kCStage);
            tma_load_3d(smem + V_CST + sg * kCStage, &vmap, &bars[VB_CFULL + sg], 0, hi.row0, 0, pol);
          } else {
            mbar_arrive(&bars[VB_CFULL + sg]);
          }
          issued = u + 1;
        }
        const volatile int never = 0;
        for (int u = max(0, issued - kCStages); u < issued; ++u)
          mbar_wait(&bars[VB_CFULL + u % kCStages], (u / kCStages) & 1, &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- O += P · V, 8 MMAs of 128 x 256 x 16 per 64-token step ----
        const uint32_t idv = idesc_f16(128, 256, false, false, true);
        int ncmd = 0, nflush = 0;
        bool ok = true, o_init = false;
        const volatile int never = 0;
        int pg = page_ahead(p, b, st, 0);
        for (int u = 0; u < n_halves; ++u) {
          const int i = u >> 1, j = u & 1, sg = u % kCStages;
          if (!mbar_wait(&bars[VB_CFULL + sg], (u / kCStages) & 1, abort_flag, kWaitNs) ||
              !mbar_wait<true>(&bars[VB_PFULL + j], i & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          if (i + 1 < n_tiles) mbar_arrive_expect_tx(&bars[VB_PFULL + j], j == 0 ? kPanel + kHdr : kPanel);
          const HalfInfo hi = half_info(p, b, st, en, u, false, pg);
          pg = page_ahead(p, b, st, u + 1);
          const unsigned char* msg = smem + V_PANEL + j * kPanel;
          int c = 0;
          if (j == 0 && o_init && *reinterpret_cast<const volatile uint32_t*>(smem + V_HDR + 512) != 0u)
            c |= CMD_RESCALE;
          if (hi.nvalid > 0 && hi.nvalid < kHalf) c |= CMD_ZERO;
          if (c) {
            if (c & CMD_RESCALE) {   // O must be quiescent before its rows are rescaled
              mma_commit(&bars[VB_FLUSH]);
              if (!mbar_wait(&bars[VB_FLUSH], nflush & 1, &never, kWaitNs)) {
                ok = false;
                break;
              }
              ++nflush;
            }
            *cmd_word = (u << 8) | c;
            mbar_arrive(&bars[VB_CREQ]);
            if (!mbar_wait(&bars[VB_CDONE], ncmd & 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            ++ncmd;
          }
          if (hi.nvalid > 0) {
            tc_fence_after();
            const uint32_t pb = smem_u32(msg);
            const uint32_t vb = smem_u32(smem + V_CST + sg * kCStage);
#pragma unroll
            for (int kk = 0; kk < kHalf / 16; ++kk) {
              const uint64_t a = sdesc_sw128(pb + 32 * kk, 16, 1024);
#pragma unroll
              for (int nh = 0; nh < 2; ++nh) {
                const uint64_t bd = sdesc_sw128(vb + 4 * nh * kBox + kk * 2048, kBox, 1024);
                mma_ss(tmem + kOCol + 256 * nh, a, bd, idv, (o_init || kk > 0) ? 1u : 0u);
              }
            }
            o_init = true;
          }
          mma_commit(&bars[VB_CEMPTY + sg]);
          mma_commit_mc(&bars[SB_PFREE + j], 0x1);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[VB_FLUSH]);   // O final before the epilogue reads it
        mbar_wait(&bars[VB_FLUSH], nflush & 1, &never, kWaitNs);
        *o_init_word = o_init ? 1 : 0;
        *cmd_word = CMD_DONE;
        mbar_arrive(&bars[VB_CREQ]);
      }
    } else {
      // ---- row warps: commands from the PV issuer, then the epilogue ----
      const int q = warp & 3;
      const int h = q * 32 + lane;
      const int j = (warp - 2) >> 2;
      const int tid = threadIdx.x - 64;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      int k = 0;
      bool ok = true;
      while (true) {
        if (!warp_wait(&bars[VB_CREQ], k & 1, abort_flag)) {
          ok = false;
          give_up(p, abort_flag, smem, peer);
          break;
        }
        ++k;
        const int c = *cmd_word;
        if (c & CMD_DONE) break;
        const int u = c >> 8;
        if (c & CMD_ZERO) {   // rows of a ragged step beyond the split: zero V so that 0·V stays 0
          const int nvalid = half_info(p, b, st, en, u, false).nvalid;
          unsigned char* cst = smem + V_CST + (u % kCStages) * kCStage;
          for (int idx = tid; idx < (kHalf - nvalid) * 64; idx += 256) {
            const int row = nvalid + (idx >> 6), box = (idx >> 3) & 7, chunk = idx & 7;
            *reinterpret_cast<uint4*>(cst + box * kBox + row * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        if (c & CMD_RESCALE) {
          tc_fence_after();
          const float f = reinterpret_cast<const float*>(smem + V_HDR)[h];
          if (__any_sync(0xffffffffu, f != 1.f)) {
            uint32_t r[32];
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
              const uint32_t col = kOCol + 256 * j + 32 * cc;
              MLA_TMEM_LD32(trow + col, r);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * f);
              MLA_TMEM_ST32(trow + col, r);
            }
            tmem_wait_st();
          }
          tc_fence_before();
        }
        mbar_arrive(&bars[VB_CDONE]);
      }
      // epilogue: o_part = O / l, lse_part = (m + log2 l) · ln 2, staged in shared memory
      // (the c_KV stages are idle now) so that the global stores are coalesced rows
      griddep_wait();   // o_part may still be read by the previous kernel of the stream
      const bool fin_ok = ok && warp_wait<true>(&bars[VB_FIN], 0, abort_flag);
      tc_fence_after();
      const float* fin = reinterpret_cast<const float*>(smem + V_PANEL);
      const float m = fin[2 * h];
      const float l = fin[2 * h + 1];
      const bool good = fin_ok && *o_init_word != 0 && l > 0.f;
      const float inv = good ? 1.f / l : 0.f;
      // Each row warp owns 32 heads x 256 columns: eight 32-column chunks, each scaled,
      // staged 128B-swizzled in a 4 KB buffer of the warp's own and written at once by a
      // TMA store that the warp issues; four buffers per warp rotate, so the stores
      // overlap the TMEM reads of the next chunks.
      const int rows = p.n_h < 128 ? p.n_h : 128;
      const int wrows = rows < 32 ? rows : 32;
      const bool wlive = 32 * q < rows;
      unsigned char* wst = smem + V_CST + (warp - 2) * 16384;
      const int orow0 = (b * p.S + s) * p.n_h + 32 * q;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        const int chunk = 8 * j + cc;
        uint32_t r[32];
        MLA_TMEM_LD32(trow + kOCol + 32 * chunk, r);
        tmem_wait_ld();
        if (!wlive) continue;
        unsigned char* buf = wst + (cc & 3) * 4096;
        if (cc >= 4) {   // this buffer's previous store has to have read it
          if (lane == 0) bulk_wait_group_read<3>();
          __syncwarp();
        }
        if (lane < wrows) {
          unsigned char* dst = buf + lane * 128;
#pragma unroll
          for (int x = 0; x < 8; ++x)
            *reinterpret_cast<float4*>(dst + ((x ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(r[4 * x]) * inv, __uint_as_float(r[4 * x + 1]) * inv,
                            __uint_as_float(r[4 * x + 2]) * inv, __uint_as_float(r[4 * x + 3]) * inv);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&omap, buf, 0, orow0, chunk);
          bulk_commit_group();
        }
      }
      if (wlive && lane == 0) bulk_wait_group0();
      if (j == 0 && h < p.n_h)
        p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] =
            good ? (m + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
      tc_fence_before();
    }
  }

  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
}

// ------------------------------------ host side ---------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3D map over rows of 576 bf16 seen as (64 columns, row, 64-column chunk), the chunk
// stride being 128 bytes; a box of `box_rows` rows x `box_chunks` chunks lands in
// shared memory chunk-major, each chunk a 128B-swizzled [box_rows][64] block.
bool make_row_map(const void* base, int64_t rows, int box_rows, int box_chunks, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kRow / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)kRow * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D map over the fp32 partial results [rows][512] seen as (32 values, row, 16 chunks of
// 32), 128B swizzle; a box is `box_rows` rows (32, or n_h when smaller) x one chunk.
bool make_out_map(float* base, int64_t rows, int box_rows, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {32, (cuuint64_t)rows, (cuuint64_t)(kLatent / 32)};
  cuuint64_t strides[2] = {(cuuint64_t)kLatent * 4, 128};
  cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool decode_tc_supported(const DecodeParams& p) {
  return (p.kv_dtype == MLA_KV_BF16 || p.kv_dtype == MLA_KV_FP8_E4M3) && p.num_rows >= 1 &&
         p.num_rows < (int64_t)INT_MAX - 2 * kTile;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int max_seq_len, cudaStream_t st) {
  (void)max_seq_len;
  // score side: 128 rows x 3 chunks (contiguous) or, for paged caches, 64 rows x 1 chunk
  // through the value map; value side: 64 rows x 8 chunks; queries: n_h rows x 3 chunks
  // (partial-result store: n_h rows x 8 chunks of 32 fp32)
  CUtensorMap smap, vmap, qmap, omap;
  if (!make_row_map(p.data, p.num_rows, p.block_table ? 64 : kTile, p.block_table ? 1 : 3, &smap) ||
      !make_row_map(p.data, p.num_rows, 64, 8, &vmap) ||
      !make_row_map(p.q_lat, (int64_t)p.B * p.n_h, p.n_h < 128 ? p.n_h : 128, 3, &qmap) ||
      !make_out_map(p.o_part, (int64_t)p.B * p.S * p.n_h, p.n_h < 32 ? p.n_h : 32, &omap))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  const int64_t ctas = 2ll * p.B * p.S;
  return launch_overlapped(decode_tc_kernel, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes, st, p, smap, vmap,
                           qmap, omap, scale_log2);
}

int decode_tc_num_splits(int B, int tiles, int n_h, int sms) {
  (void)n_h;
  const int pairs = sms / 2 > 0 ? sms / 2 : 1;
  int best = 1;
  double best_t = 1e30;
  for (int S = 1; S <= MLA_MAX_SPLITS && S <= tiles; ++S) {
    const int per = ceil_div(tiles, S);
    const int waves = ceil_div(B * S, pairs);
    // time in 64-token tile units: waves of `per` tiles plus a fixed start/drain cost
    // per unit (~4 tiles: Q load, pipeline fill, the 256 KB partial-result write), plus
    // the merge reading the partials back
    const double t = waves * (per + 4.0) + 2.0 * (double)B * S / pairs;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  return best;
}

}  // namespace mla
