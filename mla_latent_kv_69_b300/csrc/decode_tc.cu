// Tensor-core split-KV decode over the MLA latent cache (sm_103a: tcgen05 + TMEM + TMA).
//
// With W_UK folded into the query and W_UV applied after the latent-space sum
// ("DeepSeek-V2 机制拆解" (discosf.com), §长上下文推理的第一瓶颈), all n_h heads of one
// sequence attend over the same 576-wide cache rows, so per 64-token tile the work is
// two dense contractions with the heads as the M dimension:
//     S[128 x 64]  = Q[128 x 576] · C[64 x 576]^T        (scores, fp32 in TMEM)
//     O[128 x 512] += P[128 x 64] · C[64 x 0:512]        (latent output, fp32 in TMEM)
// O alone fills the 512 TMEM columns of an SM, so one work unit (sequence b, split s)
// runs on a cluster of two CTAs on two SMs:
//   CTA0  Q (bf16) lives in TMEM columns 0..287 and S in two 64-column buffers; it
//         issues S = Q·C^T with the A operand read from TMEM, runs the online softmax
//         (one thread per head, exp2 with a running maximum that is only raised when a
//         tile's maximum exceeds it by 2^8), and stores P (bf16) straight into CTA1's
//         shared memory over DSMEM.
//   CTA1  owns the 128 x 512 fp32 O accumulator (all of its TMEM) and issues O += P·V,
//         V being the same cache tile read as an MN-major operand. Its four row warps
//         rescale O rows when CTA0 raised a maximum, zero the unused rows of a ragged
//         last tile, and write the normalised o_part / lse_part at the end.
// Each cache tile is fetched from HBM once: the eight 8 KB boxes of c_KV (dims 0..511)
// are TMA-multicast into both CTAs (four issued by each), and the RoPE-key box (dims
// 512..575) goes to CTA0 only. A 3-stage ring of mbarriers paces the loads; a stage is
// refilled once both CTAs' tensor-core work on it has committed.
//
// Every wait is bounded (2 s); on expiry the CTA records MLA_ERR_TIMEOUT in the status
// word, tells the peer to stop, drains its own loads and MMAs, frees TMEM and returns.
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

constexpr int kTile = 64;                 // tokens per tile (= one page)
constexpr int kStages = 3;
constexpr int kBox = 64 * 64 * 2;         // one TMA box: 64 rows x 64 bf16 (128 B rows, 128B swizzle)
constexpr int kCStage = 8 * kBox;         // c_KV part of a tile: dims 0..511
constexpr int kPBytes = 128 * 64 * 2;     // P tile: 128 heads x 64 tokens bf16
constexpr int kThreads = 192;             // warp 0 TMA, warp 1 MMA, warps 2..5 row warps
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.f;       // raise the running max only when a tile exceeds it by 2^8

constexpr uint32_t kQCol = 0;             // CTA0 TMEM: Q as bf16 pairs (288 columns)
constexpr uint32_t kSCol = 288;           // CTA0 TMEM: S buffers, 2 x 64 columns
constexpr uint32_t kOCol = 0;             // CTA1 TMEM: O, 512 columns

// Shared memory map (offsets from the 1024-byte aligned dynamic base; same in both CTAs,
// which multicast requires).
constexpr int OFF_C = 0;                                // [3][64 KB] c_KV boxes 0..7
constexpr int OFF_X = kStages * kCStage;                // CTA0: [3][8 KB] RoPE-key box; CTA1: [2][16 KB] P
constexpr int OFF_FACT = OFF_X + 2 * kPBytes;           // CTA1: [2][128] fp32 rescale factors
constexpr int OFF_FLAGS = OFF_FACT + 2 * 128 * 4;       // CTA1: [2][4] int "some row of this quarter rescales"
constexpr int OFF_ML = OFF_FLAGS + 64;                  // CTA1: [128][2] fp32 final (max, sum) per head
constexpr int OFF_BAR = OFF_ML + 128 * 2 * 4;
enum Bar {
  B_FULL = 0,                // [3] tile landed (TMA transaction bytes)
  B_EMPTY = B_FULL + 3,      // [3] both CTAs' MMAs finished with the stage (2 arrivals)
  B_SFULL = B_EMPTY + 3,     // [2] CTA0: S buffer written by QK^T
  B_SFREE = B_SFULL + 2,     // [2] CTA0: S buffer read by the softmax threads (128)
  B_QREADY = B_SFREE + 2,    // CTA0: Q stored into TMEM (128)
  B_PFULL = B_QREADY + 1,    // [2] CTA1: P, factors and flags written by CTA0 (128 remote)
  B_PFREE = B_PFULL + 2,     // [2] CTA0: CTA1's PV MMA finished reading a P buffer (1 remote commit)
  B_FLUSH = B_PFREE + 2,     // MMA warp: all previously issued MMAs completed
  B_CREQ = B_FLUSH + 1,      // CTA1: command for the row warps (1)
  B_CDONE = B_CREQ + 1,      // CTA1: row warps finished the command (128)
  B_MLREADY = B_CDONE + 1,   // CTA1: final (max, sum) received (128 remote)
  B_COUNT = B_MLREADY + 1
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;         // tmem base, abort flag, command word
constexpr int kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

enum Cmd { CMD_ZERO = 1, CMD_RESCALE = 2, CMD_DONE = 4 };

struct TileInfo {
  int row0;     // first cache row of the tile (the TMA y coordinate)
  int nvalid;   // tokens of the tile that belong to the split
  bool valid;   // the tile's rows lie inside the caller's buffers
};

__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, int b, int t0, int en) {
  TileInfo ti;
  ti.nvalid = min(kTile, en - t0);
  ti.valid = true;
  ti.row0 = 0;
  if (p.block_table) {
    const int pi = t0 >> 6;
    const int page = pi < p.max_pages ? p.block_table[(int64_t)b * p.max_pages + pi] : -1;
    if (page < 0 || (int64_t)page * kTile >= p.num_rows) ti.valid = false;
    else ti.row0 = page * kTile;
  } else {
    const int64_t row = (int64_t)b * p.seq_stride + t0;
    if (t0 >= p.seq_stride || row >= p.num_rows) {
      ti.valid = false;
    } else {
      ti.row0 = (int)row;
      const int64_t room = (p.seq_stride - t0) < (p.num_rows - row) ? (p.seq_stride - t0) : (p.num_rows - row);
      if (room < ti.nvalid) ti.nvalid = (int)room;
    }
  }
  if (!ti.valid) {
    ti.nvalid = 0;
    ti.row0 = (int)(p.num_rows < (int64_t)(INT_MAX - kTile) ? p.num_rows : (int64_t)(INT_MAX - kTile));  // out of range: TMA fills zeros
  }
  return ti;
}

// A bounded wait taken by all 32 lanes of a warp together: every lane returns the same
// answer, so warp-collective code after it never runs with lanes missing.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort_flag, kWaitNs);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void give_up(const DecodeParams& p, volatile int* abort_flag, unsigned char* smem,
                                        uint32_t peer) {
  record_status(p.status, MLA_ERR_TIMEOUT);
  *abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(smem + OFF_MISC + 4), peer), 1u);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap, float scale_log2) {
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

  if (n_tiles == 0) {   // empty split: nothing crosses the cluster
    if (rank == 1) {
      float* o = p.o_part + ((int64_t)b * p.S + s) * p.n_h * kLatent;
      for (int i = threadIdx.x; i < p.n_h * kLatent / 4; i += kThreads)
        reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h = threadIdx.x; h < p.n_h; h += kThreads)
        p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] = -INFINITY;
    }
    return;
  }
  if (smem_u32(smem) & 1023u) {   // the 128B swizzle needs 1024-byte aligned stages
    if (threadIdx.x == 0) record_status(p.status, MLA_ERR_UNSUPPORTED);
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* cmd_word = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kStages; ++k) {
      mbar_init(&bars[B_FULL + k], 1);
      mbar_init(&bars[B_EMPTY + k], 2);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[B_SFULL + k], 1);
      mbar_init(&bars[B_SFREE + k], 128);
      mbar_init(&bars[B_PFULL + k], 128);
      mbar_init(&bars[B_PFREE + k], 1);
    }
    mbar_init(&bars[B_QREADY], 128);
    mbar_init(&bars[B_FLUSH], 1);
    mbar_init(&bars[B_CREQ], 1);
    mbar_init(&bars[B_CDONE], 128);
    mbar_init(&bars[B_MLREADY], 128);
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any multicast or remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      prefetch_tmap(&tmap);
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int stg = i % kStages;
        if (i >= kStages && !mbar_wait<true>(&bars[B_EMPTY + stg], ((i / kStages) - 1) & 1, abort_flag, kWaitNs)) {
          give_up(p, abort_flag, smem, peer);
          break;
        }
        const TileInfo ti = tile_info(p, b, st + i * kTile, en);
        if (!ti.valid && rank == 0) record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
        unsigned char* cst = smem + OFF_C + stg * kCStage;
        if (rank == 0) {
          mbar_arrive_expect_tx(&bars[B_FULL + stg], kCStage + kBox);
          for (int j = 0; j < 4; ++j) tma_load_2d_mc(cst + j * kBox, &tmap, &bars[B_FULL + stg], 64 * j, ti.row0, 0x3, pol);
          tma_load_2d(smem + OFF_X + stg * kBox, &tmap, &bars[B_FULL + stg], 512, ti.row0, pol);
        } else {
          mbar_arrive_expect_tx(&bars[B_FULL + stg], kCStage);
          for (int j = 4; j < 8; ++j) tma_load_2d_mc(cst + j * kBox, &tmap, &bars[B_FULL + stg], 64 * j, ti.row0, 0x3, pol);
        }
        issued = i + 1;
      }
      // Loads still in flight land before the CTA may leave.
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        const volatile int never = 0;
        mbar_wait<true>(&bars[B_FULL + i % kStages], (i / kStages) & 1, &never, kWaitNs / 4);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (rank == 0) {
        // ---------------------------- S = Q · C^T -----------------------------------
        const uint32_t idq = idesc_f16(128, 64, false, false, false);
        bool ok = mbar_wait(&bars[B_QREADY], 0, abort_flag, kWaitNs);
        tc_fence_after();
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int stg = i % kStages, sb = i & 1;
          if (!mbar_wait<true>(&bars[B_FULL + stg], (i / kStages) & 1, abort_flag, kWaitNs) ||
              (i >= 2 && !mbar_wait(&bars[B_SFREE + sb], ((i >> 1) - 1) & 1, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t cb = smem_u32(smem + OFF_C + stg * kCStage);
          const uint32_t kb = smem_u32(smem + OFF_X + stg * kBox);
          const uint32_t d = tmem + kSCol + 64 * sb;
#pragma unroll
          for (int k = 0; k < kRow / 16; ++k) {
            const int box = k >> 2;
            const uint32_t addr = (box < 8 ? cb + box * kBox : kb) + (k & 3) * 32;
            mma_ts(d, tmem + kQCol + 8 * k, sdesc_sw128(addr, 16, 1024), idq, k > 0);
          }
          mma_commit(&bars[B_SFULL + sb]);
          mma_commit_mc(&bars[B_EMPTY + stg], 0x3);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[B_FLUSH]);
        const volatile int never = 0;
        mbar_wait(&bars[B_FLUSH], 0, &never, kWaitNs);
      } else {
        // ---------------------------- O += P · V -------------------------------------
        const uint32_t idv = idesc_f16(128, 256, false, false, true);
        int ncmd = 0, nflush = 0;
        bool ok = true;
        const volatile int never = 0;
        for (int i = 0; i < n_tiles; ++i) {
          const int stg = i % kStages, sb = i & 1;
          if (!mbar_wait<true>(&bars[B_FULL + stg], (i / kStages) & 1, abort_flag, kWaitNs) ||
              !mbar_wait<true>(&bars[B_PFULL + sb], (i >> 1) & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          const TileInfo ti = tile_info(p, b, st + i * kTile, en);
          const volatile int* fl = reinterpret_cast<const volatile int*>(smem + OFF_FLAGS) + sb * 4;
          int c = 0;
          if (ti.nvalid < kTile) c |= CMD_ZERO;
          if (fl[0] | fl[1] | fl[2] | fl[3]) c |= CMD_RESCALE;
          if (c) {
            if (c & CMD_RESCALE) {   // O must be quiescent before its rows are rescaled
              mma_commit(&bars[B_FLUSH]);
              if (!mbar_wait(&bars[B_FLUSH], nflush & 1, &never, kWaitNs)) { ok = false; break; }
              ++nflush;
            }
            *cmd_word = (i << 8) | c;
            mbar_arrive(&bars[B_CREQ]);
            if (!mbar_wait(&bars[B_CDONE], ncmd & 1, abort_flag, kWaitNs)) { ok = false; break; }
            ++ncmd;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t pb = smem_u32(smem + OFF_X + sb * kPBytes);
          const uint32_t vb = smem_u32(smem + OFF_C + stg * kCStage);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t a = sdesc_sw128(pb + 32 * kk, 16, 1024);
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
              const uint64_t bd = sdesc_sw128(vb + 4 * nh * kBox + kk * 2048, kBox, 1024);
              mma_ss(tmem + kOCol + 256 * nh, a, bd, idv, (i > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit_mc(&bars[B_EMPTY + stg], 0x3);
          mma_commit_mc(&bars[B_PFREE + sb], 0x1);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[B_FLUSH]);                  // O final before the epilogue reads it
        mbar_wait(&bars[B_FLUSH], nflush & 1, &never, kWaitNs);
        *cmd_word = CMD_DONE;
        mbar_arrive(&bars[B_CREQ]);
      }
    }
  } else {
    // ------------------------------ row warps (2..5) ---------------------------------
    const int q = warp & 3;                       // TMEM lane quarter this warp may access
    const int h = q * 32 + lane;                  // head (= TMEM lane) owned by this thread
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    if (rank == 0) {
      // Q row h → TMEM (packed bf16 pairs; padded heads are zero)
      {
        const uint4* qrow = reinterpret_cast<const uint4*>(p.q_lat + ((int64_t)b * p.n_h + min(h, p.n_h - 1)) * kRow);
        uint32_t r[32];
#pragma unroll 1
        for (int c = 0; c < 9; ++c) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4 v = h < p.n_h ? __ldg(qrow + c * 8 + j) : make_uint4(0, 0, 0, 0);
            r[4 * j] = v.x; r[4 * j + 1] = v.y; r[4 * j + 2] = v.z; r[4 * j + 3] = v.w;
          }
          MLA_TMEM_ST32(trow + kQCol + 32 * c, r);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[B_QREADY]);
      }
      // online softmax
      float m_run = -INFINITY, l_run = 0.f;
      const uint32_t p_remote = mapa(smem_u32(smem + OFF_X), 1);
      const uint32_t fact_remote = mapa(smem_u32(smem + OFF_FACT), 1);
      const uint32_t flags_remote = mapa(smem_u32(smem + OFF_FLAGS), 1);
      for (int i = 0; i < n_tiles; ++i) {
        const int sb = i & 1;
        if (!warp_wait(&bars[B_SFULL + sb], (i >> 1) & 1, abort_flag)) {
          give_up(p, abort_flag, smem, peer);
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        MLA_TMEM_LD32(trow + kSCol + 64 * sb, sr);
        MLA_TMEM_LD32(trow + kSCol + 64 * sb + 32, (sr + 32));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[B_SFREE + sb]);
        const int nvalid = tile_info(p, b, st + i * kTile, en).nvalid;
        float x[64];
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          x[j] = j < nvalid ? __uint_as_float(sr[j]) * scale_log2 : -INFINITY;
          mt = fmaxf(mt, x[j]);
        }
        float factor = 1.f;
        bool need = false;
        if (m_run == -INFINITY) {
          m_run = mt;                              // nothing accumulated yet
        } else if (mt > m_run + kRescaleLog2) {
          factor = ex2(m_run - mt);
          l_run *= factor;
          m_run = mt;
          need = true;
        }
        const bool live = m_run != -INFINITY;
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float p0 = live ? ex2(x[2 * j] - m_run) : 0.f;
          const float p1 = live ? ex2(x[2 * j + 1] - m_run) : 0.f;
          const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
          const float2 back = __bfloat1622float2(v);
          lsum += back.x + back.y;                 // the sum of exactly the weights the MMA uses
          pk[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
        l_run += lsum;
        if (i >= 2 && !warp_wait<true>(&bars[B_PFREE + sb], ((i >> 1) - 1) & 1, abort_flag)) {
          give_up(p, abort_flag, smem, peer);
          break;
        }
        const uint32_t prow = p_remote + sb * kPBytes + h * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_cluster_v4(prow + ((c ^ (h & 7)) << 4), make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
        st_cluster_f32(fact_remote + (sb * 128 + h) * 4, factor);
        const unsigned any = __ballot_sync(0xffffffffu, need);
        if (lane == 0) st_cluster_u32(flags_remote + (sb * 4 + q) * 4, any != 0u);
        fence_proxy_async_cluster();
        mbar_arrive_remote(&bars[B_PFULL + sb], 1);
      }
      const uint32_t ml_remote = mapa(smem_u32(smem + OFF_ML), 1);
      st_cluster_f32(ml_remote + h * 8, m_run);
      st_cluster_f32(ml_remote + h * 8 + 4, l_run);
      mbar_arrive_remote(&bars[B_MLREADY], 1);
    } else {
      // CTA1: commands from the PV issuer, then the epilogue
      int k = 0;
      bool ok = true;
      while (true) {
        if (!warp_wait(&bars[B_CREQ], k & 1, abort_flag)) {
          ok = false;
          give_up(p, abort_flag, smem, peer);
          break;
        }
        ++k;
        const int c = *cmd_word;
        if (c & CMD_DONE) break;
        const int i = c >> 8;
        if (c & CMD_ZERO) {
          const int nvalid = tile_info(p, b, st + i * kTile, en).nvalid;
          unsigned char* cst = smem + OFF_C + (i % kStages) * kCStage;
          const int tid = threadIdx.x - 64;
          for (int idx = tid; idx < (kTile - nvalid) * 64; idx += 128) {
            const int row = nvalid + (idx >> 6), box = (idx >> 3) & 7, chunk = idx & 7;
            *reinterpret_cast<uint4*>(cst + box * kBox + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        if (c & CMD_RESCALE) {
          tc_fence_after();
          const float f = reinterpret_cast<const float*>(smem + OFF_FACT)[(i & 1) * 128 + h];
          if (__any_sync(0xffffffffu, f != 1.f)) {
            uint32_t r[32];
#pragma unroll 1
            for (int cc = 0; cc < 16; ++cc) {
              MLA_TMEM_LD32(trow + kOCol + 32 * cc, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
              MLA_TMEM_ST32(trow + kOCol + 32 * cc, r);
            }
            tmem_wait_st();
          }
          tc_fence_before();
        }
        mbar_arrive(&bars[B_CDONE]);
      }
      // epilogue: o_part = O / l, lse_part = (m + log2 l) · ln 2
      if (ok && !warp_wait<true>(&bars[B_MLREADY], 0, abort_flag)) {
        ok = false;
        give_up(p, abort_flag, smem, peer);
      }
      tc_fence_after();
      const float m = reinterpret_cast<const float*>(smem + OFF_ML)[2 * h];
      const float l = reinterpret_cast<const float*>(smem + OFF_ML)[2 * h + 1];
      const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
      float* orow = p.o_part + (((int64_t)b * p.S + s) * p.n_h + h) * kLatent;
      uint32_t r[32];
#pragma unroll 1
      for (int cc = 0; cc < 16; ++cc) {
        MLA_TMEM_LD32(trow + kOCol + 32 * cc, r);
        tmem_wait_ld();
        if (h < p.n_h) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(orow + 32 * cc)[j] =
                make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                            __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
        }
      }
      if (h < p.n_h)
        p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] =
            (ok && l > 0.f) ? (m + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
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

// One 2D map over the whole cache: rows of 576 bf16, boxes of 64 rows x 64 columns.
bool make_cache_map(const DecodeParams& p, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)p.num_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kRow * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.data), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool decode_tc_supported(const DecodeParams& p) {
  return p.kv_dtype == MLA_KV_BF16 && p.num_rows >= 1 && p.num_rows < (int64_t)INT_MAX - 2 * kTile;
}

cudaError_t launch_decode_tc(const DecodeParams& p, int max_seq_len, cudaStream_t st) {
  (void)max_seq_len;
  CUtensorMap map;
  if (!make_cache_map(p, &map)) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const float scale_log2 = p.scale * 1.4426950408889634f;
  const int64_t ctas = 2ll * p.B * p.S;
  decode_tc_kernel<<<(unsigned)ctas, kThreads, kSmemBytes, st>>>(p, map, scale_log2);
  return cudaGetLastError();
}

int decode_tc_num_splits(int B, int tiles, int n_h, int sms) {
  (void)n_h;
  const int pairs = sms / 2 > 0 ? sms / 2 : 1;
  int best = 1;
  double best_t = 1e30;
  for (int S = 1; S <= MLA_MAX_SPLITS && S <= tiles; ++S) {
    const int per = ceil_div(tiles, S);
    const int waves = ceil_div(B * S, pairs);
    // time in tile units: waves of `per` tiles, plus ~3.6 tile-equivalents of
    // partial-result traffic per unit (256 KB fp32 written, read back by the merge)
    const double t = waves * (per + 3.6) + 3.6 * (double)B * S / pairs;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  return best;
}

}  // namespace mla
