// Tensor-core split-KV decode over the MLA latent cache (sm_103a: tcgen05 + TMEM + TMA).
//
// With W_UK folded into the query and W_UV applied after the latent-space sum
// ("DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈), all n_h heads of one
// sequence attend over the same 576-wide cache rows, so every tile of tokens is two
// dense contractions with the heads as the M dimension:
//     S[128 x 128] = Q[128 x 576] · C[128 x 576]^T       (scores, fp32 in TMEM)
//     O[128 x 512] += P[128 x 128] · C[128 x 0:512]      (latent output, fp32 in TMEM)
// O alone fills the 512 TMEM columns of an SM, so the work runs on clusters of two CTAs
// (an SM pair) that exchange only P:
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
//
// Each pair works through a list of pieces (decode_tc.cuh: one contiguous token range of
// one sequence each, written to its own partial-result slot). With the balanced schedule
// every pair gets the same number of 128-token tiles of the whole batch, so all SM pairs
// stay busy whatever the batch's shape, and a pair moves from one piece to the next
// without leaving the kernel: the next piece's query travels through the same load ring
// as the cache rows, and the value CTA drains O before it accumulates the next piece.
//
// The TMA engine spends a roughly fixed time per box row, so loads use 3D tensor maps
// (64 columns x rows x column chunks) that fetch several 128-byte chunks of each row
// per instruction; the shared-memory image is the same chunk-major 128B-swizzled
// layout as one 2D box per chunk. A tensor-core instruction costs at least ~64 cycles
// whatever N <= 128, so the score side uses N = 128 token tiles; the shared-memory link
// between the two SMs is narrow (~20 B/clk), so only P (16 KB per 64 tokens) crosses
// it, never fp32 scores.
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
#include "tmap.cuh"

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
constexpr int kFin = 128 * 2 * 4;          // final (m, l) of each head of a piece
constexpr int kEpiBuf = 4096;              // epilogue staging: 32 heads x 32 fp32 per TMA store
constexpr int kThreads = 320;              // warp 0 TMA, warp 1 MMA, warps 2..9 row warps
constexpr uint64_t kWaitNs = kDecodeWaitNs;
constexpr float kRescaleLog2 = 8.f;

constexpr uint32_t kQCol = 0;              // score CTA TMEM: Q as bf16 pairs (288 columns)
constexpr uint32_t kSCol = 288;            // score CTA TMEM: S (128 columns)
constexpr uint32_t kOCol = 0;              // value CTA TMEM: O (512 columns)

// Shared memory (offsets from the 1024-byte aligned dynamic base).
//   score CTA
constexpr int S_RING = 0;                              // kRing x 48 KB: query and cache groups
constexpr int S_PANEL = S_RING + kRing * kGroup;       // 2 x 16 KB P panels, send side
constexpr int S_HDR = S_PANEL + 2 * kPanel;            // rescale factors + flag sent with panel 0
constexpr int S_MX = S_HDR + kHdr;                     // [2 halves][128] fp32: tile maxima, then l halves
constexpr int S_END = S_MX + 2 * 128 * 4;
//   value CTA
constexpr int V_CST = 0;                               // kCStages x 64 KB
constexpr int V_PANEL = V_CST + kCStages * kCStage;    // 2 x 16 KB P panels, receive side
constexpr int V_HDR = V_PANEL + 2 * kPanel;
constexpr int V_FIN = V_HDR + kHdr;                    // 2 x final (m, l), by piece parity
constexpr int V_END = V_FIN + 2 * kFin;
//   both (same offset in both CTAs: remote arrivals and copies address it by offset)
constexpr int OFF_BAR = (S_END > V_END ? S_END : V_END);
enum Bar {
  SB_SLOT_FULL = 0,                       // [kRing] score: ring item landed
  SB_SLOT_EMPTY = SB_SLOT_FULL + kRing,   // [kRing] score: item consumed (QK MMAs, or the query copy)
  SB_QREADY = SB_SLOT_EMPTY + kRing,      // score: the piece's query copied into TMEM (256)
  SB_SFULL = SB_QREADY + 1,               // score: S written
  SB_SFREE = SB_SFULL + 1,                // score: S read by the softmax threads (256)
  SB_PFREE = SB_SFREE + 1,                // [2] score: the value CTA's PV finished with panel j (remote commit)
  SB_FLUSH = SB_PFREE + 2,                // score MMA warp: all MMAs done
  VB_CFULL = SB_FLUSH + 1,                // [kCStages] value: stage landed
  VB_CEMPTY = VB_CFULL + kCStages,        // [kCStages] value: PV done with the stage
  VB_PFULL = VB_CEMPTY + kCStages,        // [2] value: P panel j received (bulk copy bytes)
  VB_FIN = VB_PFULL + 2,                  // [2] value: a piece's final (m, l) stored (remote arrival)
  VB_FLUSH = VB_FIN + 2,                  // value MMA warp: all MMAs done
  VB_CREQ = VB_FLUSH + 1,                 // value: command for the row warps (1)
  VB_CDONE = VB_CREQ + 1,                 // value: row warps finished it (256)
  VB_GO = VB_CDONE + 1,                   // value: the score CTA holds its first query (remote arrival)
  VB_EPIFREE = VB_GO + 1,                 // value: an epilogue's stores finished reading their stage (8)
  B_COUNT = VB_EPIFREE + 1
};
constexpr int OFF_SCHED = OFF_BAR + B_COUNT * 8;           // SchedShared
constexpr int OFF_MISC = OFF_SCHED + (int)sizeof(SchedShared);   // tmem base, abort flag, command word, O-initialised flag
constexpr int kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(S_PANEL % 1024 == 0 && V_PANEL % 1024 == 0 && kGroup % 1024 == 0, "swizzle alignment");
static_assert(OFF_SCHED % 8 == 0 && V_FIN % 16 == 0, "alignment");
static_assert(8 * kEpiBuf * 2 <= kCStage, "epilogue staging fits in one value stage");
static_assert(8 * kEpiBuf * 6 <= kCStages * kCStage, "last epilogue staging fits in the value stages");
static_assert(16 * kThreads <= kRing * kGroup, "schedule scratch fits in the ring");

// Row-warp commands (the piece index travels in bits 8 and up for CMD_EPI)
enum Cmd { CMD_ZERO = 1, CMD_RESCALE = 2, CMD_EPI = 4, CMD_EXIT = 8 };

__device__ __forceinline__ void give_up(const DecodeParams& p, volatile int* abort_flag, unsigned char* smem,
                                        uint32_t peer) {
  record_status(p.status, MLA_ERR_TIMEOUT);
  *abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(smem + OFF_MISC + 4), peer), 1u);
}

__device__ __forceinline__ int piece_tiles(const Piece& pc) { return (pc.en - pc.st + kTile - 1) / kTile; }

// o_part / lse_part row of head 0 of slot `slot` of sequence b
__device__ __forceinline__ int64_t part_row(const DecodeParams& p, int b, int slot) {
  return ((int64_t)b * p.S + slot) * p.n_h;
}

// lse = -inf for slots from .. S - 1 of sequence b (threads tid0, tid0 + nthr, ...)
__device__ __forceinline__ void fill_unused_slots(const DecodeParams& p, int b, int from, int tid0, int nthr) {
  for (int i = tid0; i < (p.S - from) * p.n_h; i += nthr)
    p.lse_part[part_row(p, b, from) + i] = -INFINITY;
}

// kMulti = false: one piece per pair (the uniform schedule), the piece walk compiled out.
template <bool kMulti>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap smap,
                 const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
                 float scale_log2) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1;
  // waits an abort can end: the caller's limit (a test runs them out quickly); the drains
  // of copies and tensor-core work already in flight keep the long limit
  const uint64_t wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;
  griddep_launch_dependents();

  if (smem_u32(smem) & 1023u) {   // the 128B swizzle needs 1024-byte aligned slots (same in both CTAs)
    griddep_wait();
    if (threadIdx.x == 0) record_status(p.status, MLA_ERR_UNSUPPORTED);
    return;
  }
  // The pair's pieces (seq_lens is not written by the previous kernel of the step).
  SchedShared* sched = reinterpret_cast<SchedShared*>(smem + OFF_SCHED);
  if (kMulti) sched_init(p, pair, smem, sched);
  PieceCursor cur;
  cur.start(p, pair, *sched);
  auto next_piece = [&](Piece& pc) -> bool { return kMulti && cur.next(p, pc); };
  Piece first;
  const bool any = cur.next(p, first);
  if (!any || first.en <= first.st) {
    // no work for this pair: only the slot bookkeeping (no barrier or TMEM is set up)
    griddep_wait();   // o_part / lse_part may still be read by the previous kernel
    if (rank == 1) {
      mark_empty_sequences(p, pair, threadIdx.x, kThreads);
      if (any) {   // uniform schedule, empty split: o = 0, lse = -inf (and the unused slots after it)
        float* o = p.o_part + part_row(p, first.b, first.slot) * kLatent;
        for (int i = threadIdx.x; i < p.n_h * kLatent / 4; i += kThreads)
          reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        fill_unused_slots(p, first.b, first.slot, threadIdx.x, kThreads);
      }
    }
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
    mbar_init(&bars[VB_FIN + 1], 1);
    mbar_init(&bars[VB_FLUSH], 1);
    mbar_init(&bars[VB_CREQ], 1);
    mbar_init(&bars[VB_CDONE], 256);
    mbar_init(&bars[VB_GO], 1);
    mbar_init(&bars[VB_EPIFREE], 8);
    if (rank == 1) {   // the first tile's P panels may arrive any time after the cluster sync
      mbar_arrive_expect_tx(&bars[VB_PFULL], kPanel + kHdr);
      mbar_arrive_expect_tx(&bars[VB_PFULL + 1], kPanel);
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
  const int qrows = p.n_h < 128 ? p.n_h : 128;
  const bool paged = p.block_table != nullptr;

  if (rank == 0) {
    // =============================== score CTA =========================================
    if (warp == 0) {
      if (lane == 0) {
        // ---- TMA producer: per piece the query (three items), then three column slices
        // of a tile per item; item k goes to slot k % kRing ----
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();   // c_KV is read again by the value CTA
        prefetch_tmap(&smap);
        prefetch_tmap(&qmap);
        griddep_wait();   // q_lat comes from the previous kernel
        uint32_t k = 0;
        // test hook: no loads at all, so that every wait on them runs out
        const bool issue = !p.stall_loads;
        bool ok = true;
        Piece pc = first;
        auto slot_ready = [&](uint32_t item) -> bool {   // the slot's previous item was consumed
          if (item < kRing) return true;
          return mbar_wait(&bars[SB_SLOT_EMPTY + (int)(item % kRing)], (uint32_t)(((item / kRing) - 1) & 1), abort_flag,
                           wait_ns);
        };
        while (issue) {
          const int n_tiles = piece_tiles(pc);
          for (int g = 0; g < 3 && ok; ++g, ++k) {
            if (!(ok = slot_ready(k))) break;
            const int r = (int)(k % kRing);
            mbar_arrive_expect_tx(&bars[SB_SLOT_FULL + r], 3 * qrows * 128);
            tma_load_3d(smem + S_RING + r * kGroup, &qmap, &bars[SB_SLOT_FULL + r], 0, pc.b * p.n_h, 3 * g, pol_first);
          }
          HalfInfo h0{}, h1{};
          int pg0 = page_ahead(p, pc.b, pc.st, 0), pg1 = page_ahead(p, pc.b, pc.st, 1);   // one tile ahead
          for (int kk = 0; kk < 3 * n_tiles && ok && !*abort_flag; ++kk, ++k) {
            const int i = kk / 3, g = kk % 3;
            if (!(ok = slot_ready(k))) break;
            const int r = (int)(k % kRing);
            if (g == 0) {
              h0 = half_info(p, pc.b, pc.st, pc.en, 2 * i, true, pg0);
              h1 = half_info(p, pc.b, pc.st, pc.en, 2 * i + 1, true, pg1);
              pg0 = page_ahead(p, pc.b, pc.st, 2 * i + 2);
              pg1 = page_ahead(p, pc.b, pc.st, 2 * i + 3);
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
          }
          if (!(ok && !*abort_flag && next_piece(pc))) break;
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        // Loads still in flight land before the CTA may leave.
        const volatile int never = 0;
        for (uint32_t i = k > kRing ? k - kRing : 0; i < k; ++i)
          mbar_wait(&bars[SB_SLOT_FULL + (int)(i % kRing)], (uint32_t)((i / kRing) & 1), &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- S = Q · C^T, 36 MMAs of 128 x 128 x 16 per tile ----
        const uint32_t idq = idesc_f16(128, kTile, false, false, false);
        bool ok = true;
        uint32_t k = 0, tg = 0;   // ring item, tile of the pair
        int np = 0;              // piece of the pair
        Piece pc = first;
        do {
          const int n_tiles = piece_tiles(pc);
          k += 3;   // the query items (consumed by the softmax warps)
          if (!mbar_wait(&bars[SB_QREADY], (uint32_t)(np & 1), abort_flag, wait_ns)) {
            ok = false;
            break;
          }
          if (np == 0) mbar_arrive_remote(&bars[VB_GO], 1);   // the value CTA may start its loads
          for (int i = 0; ok && i < n_tiles; ++i, ++tg) {
            if (tg > 0 && !mbar_wait(&bars[SB_SFREE], (uint32_t)((tg - 1) & 1), abort_flag, wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int g = 0; g < 3; ++g, ++k) {
              const int r = (int)(k % kRing);
              if (!mbar_wait(&bars[SB_SLOT_FULL + r], (uint32_t)((k / kRing) & 1), abort_flag, wait_ns)) {
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
          ++np;
        } while (ok && next_piece(pc));
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
      float* mx = reinterpret_cast<float*>(smem + S_MX);
      const uint32_t panel_remote = mapa(smem_u32(smem + V_PANEL + j * kPanel), 1);
      const uint32_t hdr_remote = mapa(smem_u32(smem + V_HDR), 1);
      const uint32_t pfull_remote = mapa(smem_u32(&bars[VB_PFULL + j]), 1);
      uint32_t k = 0, tg = 0;
      int np = 0;
      Piece pc = first;
      // Every thread runs every iteration and every named barrier; after an abort the
      // waits return at once and the tiles are processed as fully masked.
      do {
        const int n_tiles = piece_tiles(pc);
        // The piece's query (items k .. k + 2) → TMEM as packed bf16 pairs; heads beyond
        // n_h are zero. The previous piece's QK MMAs are complete: this thread waited for
        // their S.
        bool qok = true;
        for (int g = 0; g < 3; ++g)
          qok = qok && warp_wait(&bars[SB_SLOT_FULL + (int)((k + g) % kRing)], (uint32_t)(((k + g) / kRing) & 1),
                                 abort_flag, wait_ns);
        if (qok) {
#pragma unroll 1
          for (int c = j; c < 9; c += 2) {
            uint32_t r[32];
            const unsigned char* row =
                smem + S_RING + (int)((k + c / 3) % kRing) * kGroup + (c % 3) * (qrows * 128) + h * 128;
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
        named_sync(1, 256);   // every thread has read the query items
        if (threadIdx.x == 64)
          for (int g = 0; g < 3; ++g) mbar_arrive(&bars[SB_SLOT_EMPTY + (int)((k + g) % kRing)]);
        tc_fence_before();
        mbar_arrive(&bars[SB_QREADY]);
        k += 3 + 3 * n_tiles;

        float m_run = -INFINITY, l_run = 0.f;
        int pg = page_ahead(p, pc.b, pc.st, j);   // this thread's half of the next tile, fetched ahead
        for (int i = 0; i < n_tiles; ++i, ++tg) {
          uint32_t sr[64];
          const bool got = warp_wait(&bars[SB_SFULL], (uint32_t)(tg & 1), abort_flag, wait_ns);
          if (got) {
            tc_fence_after();
            MLA_TMEM_LD32(trow + kSCol + 64 * j, sr);
            MLA_TMEM_LD32(trow + kSCol + 64 * j + 32, (sr + 32));
            tmem_wait_ld();
          }
          tc_fence_before();
          mbar_arrive(&bars[SB_SFREE]);
          const int nv = got ? half_info(p, pc.b, pc.st, pc.en, 2 * i + j, false, pg).nvalid : 0;
          pg = page_ahead(p, pc.b, pc.st, 2 * i + 2 + j);
          // Row maximum on the raw scores (the scale is positive); tokens past the piece
          // (ragged tiles only) become -inf so that their weight is exactly 0.
          if (nv < 64) {
#pragma unroll
            for (int t = 0; t < 64; ++t)
              if (t >= nv) sr[t] = __float_as_uint(-INFINITY);
          }
          float m8[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) m8[x] = __uint_as_float(sr[x]);
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
              const float2 xy =
                  ffma2(make_float2(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])), c2, nm2);
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
          if (tg > 0) mbar_wait<true>(&bars[SB_PFREE + j], (uint32_t)((tg - 1) & 1), abort_flag, wait_ns);
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
        // the piece's final (m, l) of each head → the value CTA, stored remotely
        named_sync(1, 256);
        mx[j * 128 + h] = l_run;
        named_sync(1, 256);
        if (j == 0) {
          st_cluster_v2_f32(mapa(smem_u32(smem + V_FIN + (np & 1) * kFin + 8 * h), 1), m_run, mx[h] + mx[128 + h]);
          fence_acq_rel_cluster();
          named_sync(2, 128);
          if (q == 0 && lane == 0 && !*abort_flag) mbar_arrive_remote(&bars[VB_FIN + (np & 1)], 1);
        }
        // mx is read above before the next piece's vote writes it; all 256 threads take
        // the same decision to go on, so no named barrier ever misses a thread
        const uint32_t stop = named_popc(1, 256, *abort_flag != 0);
        ++np;
        if (stop) break;
      } while (next_piece(pc));
    }
  } else {
    // =============================== value CTA =========================================
    if (warp == 0) {
      if (lane == 0) {
        // ---- TMA producer: c_KV of every 64-token step (evict-first: last reader) ----
        const uint64_t pol = l2_policy_evict_first();
        prefetch_tmap(&vmap);
        uint32_t u = 0;   // step of the pair
        int np = 0;
        bool ok = true;
        // The epilogue of piece n stages O in the stage of the piece's last step, s_n; a
        // load into s_n after that must wait until the epilogue's stores have read it
        // (VB_EPIFREE, one phase per epilogue, confirmed strictly in order).
        int prev_stage = -1;   // s_{np - 1}
        int epi_done = 0;      // epilogues confirmed
        auto wait_epi = [&](int n) -> bool {
          for (; epi_done <= n; ++epi_done)
            if (!mbar_wait(&bars[VB_EPIFREE], (uint32_t)(epi_done & 1), abort_flag, wait_ns)) return false;
          return true;
        };
        // Start once the score CTA has its first query: its query load goes first.
        if (!mbar_wait<true>(&bars[VB_GO], 0, abort_flag, wait_ns)) ok = false;
        Piece pc = first;
        while (ok && !*abort_flag) {
          const int n_halves = 2 * piece_tiles(pc);
          int pg = page_ahead(p, pc.b, pc.st, 0);
          // a piece has at least two steps, so piece np - 2's staging stage can only come
          // round again from piece np on
          if (np >= 2 && !wait_epi(np - 2)) ok = false;
          for (int ul = 0; ok && ul < n_halves && !*abort_flag; ++ul, ++u) {
            const int sg = (int)(u % kCStages);
            if (u >= kCStages &&
                !mbar_wait(&bars[VB_CEMPTY + sg], (uint32_t)(((u / kCStages) - 1) & 1), abort_flag, wait_ns)) {
              ok = false;
              break;
            }
            if (np >= 1 && sg == prev_stage && !wait_epi(np - 1)) {   // the previous epilogue's staging
              ok = false;
              break;
            }
            const HalfInfo hi = half_info(p, pc.b, pc.st, pc.en, ul, false, pg);
            pg = page_ahead(p, pc.b, pc.st, ul + 1);
            if (hi.load) {
              mbar_arrive_expect_tx(&bars[VB_CFULL + sg], kCStage);
              tma_load_3d(smem + V_CST + sg * kCStage, &vmap, &bars[VB_CFULL + sg], 0, hi.row0, 0, pol);
            } else {
              mbar_arrive(&bars[VB_CFULL + sg]);
            }
          }
          if (!ok || *abort_flag) break;
          prev_stage = (int)((u - 1) % kCStages);   // where this piece's epilogue stages O
          ++np;
          if (!next_piece(pc)) break;
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        const volatile int never = 0;
        for (uint32_t i = u > kCStages ? u - kCStages : 0; i < u; ++i)
          mbar_wait(&bars[VB_CFULL + (int)(i % kCStages)], (uint32_t)((i / kCStages) & 1), &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- O += P · V, 8 MMAs of 128 x 256 x 16 per 64-token step ----
        const uint32_t idv = idesc_f16(128, 256, false, false, true);
        int ncmd = 0, nflush = 0, np = 0;
        uint32_t u = 0, tg = 0;
        bool ok = true;
        const volatile int never = 0;
        Piece pc = first;
        auto command = [&](int c) -> bool {   // hand a command to the row warps and wait for it
          *cmd_word = c;
          mbar_arrive(&bars[VB_CREQ]);
          const bool done = mbar_wait(&bars[VB_CDONE], (uint32_t)(ncmd & 1), abort_flag, wait_ns);
          ++ncmd;
          return done;
        };
        do {
          const int n_halves = 2 * piece_tiles(pc);
          bool o_init = false;
          int pg = page_ahead(p, pc.b, pc.st, 0);
          for (int ul = 0; ul < n_halves; ++ul, ++u) {
            const int j = ul & 1, sg = (int)(u % kCStages);
            if (!mbar_wait(&bars[VB_CFULL + sg], (uint32_t)((u / kCStages) & 1), abort_flag, wait_ns) ||
                !mbar_wait<true>(&bars[VB_PFULL + j], (uint32_t)(tg & 1), abort_flag, wait_ns)) {
              ok = false;
              break;
            }
            // re-arm for the panel's next use (an arm that no copy ever completes is harmless)
            mbar_arrive_expect_tx(&bars[VB_PFULL + j], j == 0 ? kPanel + kHdr : kPanel);
            const HalfInfo hi = half_info(p, pc.b, pc.st, pc.en, ul, false, pg);
            pg = page_ahead(p, pc.b, pc.st, ul + 1);
            int c = 0;
            if (j == 0 && o_init && *reinterpret_cast<const volatile uint32_t*>(smem + V_HDR + 512) != 0u)
              c |= CMD_RESCALE;
            if (hi.nvalid > 0 && hi.nvalid < kHalf) c |= CMD_ZERO;
            if (c) {
              if (c & CMD_RESCALE) {   // O must be quiescent before its rows are rescaled
                mma_commit(&bars[VB_FLUSH]);
                if (!mbar_wait(&bars[VB_FLUSH], (uint32_t)(nflush & 1), &never, kWaitNs)) {
                  ok = false;
                  break;
                }
                ++nflush;
              }
              if (!command((int)((ul << 8) | c))) {
                ok = false;
                break;
              }
            }
            if (hi.nvalid > 0) {
              tc_fence_after();
              const uint32_t pb = smem_u32(smem + V_PANEL + j * kPanel);
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
            if (j == 1) ++tg;
          }
          if (!ok) break;
          // O final before the row warps read it; they acknowledge once O is drained
          mma_commit(&bars[VB_FLUSH]);
          if (!mbar_wait(&bars[VB_FLUSH], (uint32_t)(nflush & 1), &never, kWaitNs)) {
            ok = false;
            break;
          }
          ++nflush;
          *o_init_word = o_init ? 1 : 0;
          if (!command((np << 8) | CMD_EPI)) {
            ok = false;
            break;
          }
          ++np;
        } while (next_piece(pc));
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[VB_FLUSH]);   // nothing may be in flight when the CTA leaves
        mbar_wait(&bars[VB_FLUSH], (uint32_t)(nflush & 1), &never, kWaitNs);
        *cmd_word = CMD_EXIT;
        mbar_arrive(&bars[VB_CREQ]);
      }
    } else {
      // ---- row warps: commands from the PV issuer (ragged steps, rescales, epilogues) ----
      const int q = warp & 3;
      const int h = q * 32 + lane;
      const int j = (warp - 2) >> 2;
      const int tid = threadIdx.x - 64;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      griddep_wait();   // lse_part may still be read by the previous kernel of the stream
      mark_empty_sequences(p, pair, tid, 256);
      int k = 0, np = 0;
      uint32_t u_base = 0;   // first step of the current piece
      Piece pc = first;
      while (true) {
        if (!warp_wait(&bars[VB_CREQ], (uint32_t)(k & 1), abort_flag, wait_ns)) {
          give_up(p, abort_flag, smem, peer);
          break;
        }
        ++k;
        const int c = *cmd_word;
        if (c & CMD_EXIT) break;
        if (c & CMD_ZERO) {   // rows of a ragged step beyond the piece: zero V so that 0·V stays 0
          const int ul = c >> 8;
          const int nvalid = half_info(p, pc.b, pc.st, pc.en, ul, false).nvalid;
          unsigned char* cst = smem + V_CST + (int)((u_base + ul) % kCStages) * kCStage;
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
        if (!(c & CMD_EPI)) {
          mbar_arrive(&bars[VB_CDONE]);
          continue;
        }
        // ---- epilogue of piece np: o_part = O / l, lse_part = (m + log2 l) · ln 2 ----
        griddep_wait();   // o_part may still be read by the previous kernel of the stream
        const int f = np & 1;
        const bool fin_ok = warp_wait<true>(&bars[VB_FIN + f], (uint32_t)((np >> 1) & 1), abort_flag, wait_ns);
        tc_fence_after();
        const float* fin = reinterpret_cast<const float*>(smem + V_FIN + f * kFin);
        const float m = fin[2 * h];
        const float l = fin[2 * h + 1];
        const bool good = fin_ok && *o_init_word != 0 && l > 0.f;
        const float inv = good ? 1.f / l : 0.f;
        const int n_halves = 2 * piece_tiles(pc);
        Piece nxt;
        const bool more = next_piece(nxt);
        // Each row warp owns 32 heads x 256 columns: eight 32-column chunks, each scaled and
        // staged 128B-swizzled in a 4 KB buffer of the warp's own, then read back a row
        // per eight lanes and written with coalesced 16-byte stores (four 128-byte row
        // pieces per instruction): the SM's TMA store path moved o_part at ~64 GB/s and
        // paced this epilogue. Before another piece, the buffers lie in the stage of the
        // piece's last step, which the producer refills only after VB_EPIFREE; after the
        // pair's last piece every stage is idle.
        const int rows = p.n_h < 128 ? p.n_h : 128;
        const int wrows = rows < 32 ? rows : 32;
        const bool wlive = 32 * q < rows;
        unsigned char* wst = more ? smem + V_CST + (int)((u_base + n_halves - 1) % kCStages) * kCStage +
                                        (warp - 2) * 2 * kEpiBuf
                                  : smem + V_CST + (warp - 2) * 6 * kEpiBuf;
        const int64_t orow0 = part_row(p, pc.b, pc.slot) + 32 * q;
        uint32_t r[32];
        const int ux = lane & 7, usub = lane >> 3;   // read-back: 16-byte unit, row within four
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          const int chunk = 8 * j + cc;
          MLA_TMEM_LD32(trow + kOCol + 32 * chunk, r);
          tmem_wait_ld();
          if (cc == 7) {   // O is drained: the next piece may accumulate
            tc_fence_before();
            mbar_arrive(&bars[VB_CDONE]);
          }
          if (!wlive) continue;
          unsigned char* buf = wst + (cc & 1) * kEpiBuf;
          if (lane < wrows) {
            unsigned char* dst = buf + lane * 128;
#pragma unroll
            for (int x = 0; x < 8; ++x)
              *reinterpret_cast<float4*>(dst + ((x ^ (lane & 7)) << 4)) =
                  make_float4(__uint_as_float(r[4 * x]) * inv, __uint_as_float(r[4 * x + 1]) * inv,
                              __uint_as_float(r[4 * x + 2]) * inv, __uint_as_float(r[4 * x + 3]) * inv);
          }
          __syncwarp();
          // rows 4 k + usub: head 32 q + row of o_part, columns 32 chunk + 4 ux .. + 3
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int row = 4 * k + usub;
            if (row < wrows) {
              const float4 v = *reinterpret_cast<const float4*>(buf + row * 128 + ((ux ^ (row & 7)) << 4));
              *reinterpret_cast<float4*>(p.o_part + (orow0 + row) * kLatent + 32 * chunk + 4 * ux) = v;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[VB_EPIFREE]);   // this warp's staging is free again
        if (j == 0 && h < p.n_h)
          p.lse_part[part_row(p, pc.b, pc.slot) + h] = good ? (m + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
        if (pc.fill_from < p.S) fill_unused_slots(p, pc.b, pc.fill_from, tid, 256);
        u_base += n_halves;
        ++np;
        if (more) pc = nxt;
        else pc.en = pc.st;   // no further epilogue follows
      }
      if (lane == 0) bulk_wait_group0();   // the partial results are written before the CTA may leave
      tc_fence_before();
    }
  }

  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  cluster_sync();   // no CTA leaves while its peer may still touch its shared memory
}

// ------------------------------------ host side ---------------------------------------
// 3D map over rows of 576 bf16 seen as (64 columns, row, 64-column chunk), the chunk
// stride being 128 bytes; a box of `box_rows` rows x `box_chunks` chunks lands in
// shared memory chunk-major, each chunk a 128B-swizzled [box_rows][64] block.
bool make_row_map(const void* base, int64_t rows, int box_rows, int box_chunks, CUtensorMap* map) {
  const uint64_t dims[3] = {64, (uint64_t)rows, (uint64_t)(kRow / 64)};
  const uint64_t strides[2] = {(uint64_t)kRow * 2, 128};
  const uint32_t box[3] = {64, (uint32_t)box_rows, (uint32_t)box_chunks};
  return encode_tiled(tmap_desc(base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      map);
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
  CUtensorMap smap, vmap, qmap;
  if (!make_row_map(p.data, p.num_rows, p.block_table ? 64 : kTile, p.block_table ? 1 : 3, &smap) ||
      !make_row_map(p.data, p.num_rows, 64, 8, &vmap) ||
      !make_row_map(p.q_lat, (int64_t)p.B * p.n_h, p.n_h < 128 ? p.n_h : 128, 3, &qmap))
    return cudaErrorInvalidValue;
  static std::atomic<int> attr_multi[kMaxDevices], attr_single[kMaxDevices];
  const cudaError_t attr_err = p.balanced ? smem_attr_once(decode_tc_kernel<true>, kSmemBytes, attr_multi)
                                          : smem_attr_once(decode_tc_kernel<false>, kSmemBytes, attr_single);
  if (attr_err != cudaSuccess) return attr_err;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  if (p.balanced)
    return launch_overlapped(decode_tc_kernel<true>, dim3((unsigned)(2 * p.pairs)), dim3(kThreads), kSmemBytes, st, p,
                             smap, vmap, qmap, scale_log2);
  return launch_overlapped(decode_tc_kernel<false>, dim3((unsigned)(2 * (int64_t)p.B * p.S_used)), dim3(kThreads),
                           kSmemBytes, st, p, smap, vmap, qmap, scale_log2);
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

int decode_balanced_slots(int B, int max_seq_len, int pairs) {
  const int tmax = ceil_div(max_seq_len, kSchedTile);
  if (tmax <= 1) return 1;
  // enough slots that the quota rarely exceeds total / pairs: ceil(pairs / B) pieces of
  // a sequence plus two more for boundaries and length variation
  int S = ceil_div(pairs, B > 0 ? B : 1) + 2;
  if (S > tmax) S = tmax;
  if (S > MLA_MAX_SPLITS) S = MLA_MAX_SPLITS;
  return S;
}

}  // namespace mla
