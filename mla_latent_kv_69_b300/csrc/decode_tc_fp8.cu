// Tensor-core split-KV decode over an e4m3 latent cache (sm_103a: tcgen05 + TMEM + TMA).
//
// The low-bit cache the pages report for serving ("DeepSeek-V2 机制拆解" (discosf.com),
// §推理参数与 128K 上下文的使用注意; "中文验证版", §方法适配) is stood in for by e4m3 codes
// with one fp32 scale per token. The work split is the bf16 kernel's (decode_tc.cu): a
// cluster of two CTAs per (sequence, split); the score CTA holds Q and S in TMEM and
// runs the softmax, the value CTA holds the 128 x 512 fp32 O accumulator.
//
// S = Q · code^T runs straight on the TMA-loaded codes (tcgen05 kind::f8f6f4, both
// operands e4m3): each head's query is multiplied by a power of two 2^k_h that puts its
// largest element in [2^7, 2^8) and split into two e4m3 parts, hi = e4m3(q) and
// lo = e4m3(q - hi), whose sum is the bf16 value exactly for every element within 2^-16
// of the head's largest (a bf16 value has 8 significant bits, e4m3 4); the two parts are
// two MMAs of K = 32 per step, which cost one f16 MMA of K = 16, so QK^T takes the bf16
// kernel's tensor time with no conversion of the cache. The score side loads its codes as
// 64B-swizzled [128 tokens][64 codes] chunks (the MMA's K-major operand layout).
// O += P' · V keeps f16 operands (an 8-bit P would not keep the error budget): every
// e4m3 code maps to the f16 of 2^-8 times its value, which is exact (see
// e4m3x16_to_f16); the value CTA's eight converter warps turn its TMA-loaded e4m3 rows
// into 128B-swizzled f16 tiles (its four row warps only rescale O and write it out):
//   value CTA  e4m3 ring of two 32 KB steps (64 tokens x 512 columns) → two 64 KB f16
//              stages → 8 MMAs of N = 256 per step (rows past the split are zeroed).
// The score CTA's four extra warps only stage each tile's per-token scales. 2^-k_h
// comes back in fp32 in the score scale, the value side's 2^8 in the output's 1/l.
// The per-token scale stays outside the MMAs. The score CTA multiplies each score column
// by it (x_t = scale_t · Q·code_t, log2 units) and runs the online softmax on the log2
// weight of the codes, y_t = x_t + log2 scale_t: the value CTA receives P'_t = 2^(y_t - m)
// in f16 and accumulates O += P'_t · code_t, and the normaliser sums
// 2^(x_t - m) = P'_t / scale_t in fp32. Since the running maximum m is taken over y, every
// P' that matters lies in f16's normal range (at most 2^8 under the lazy maximum) however
// small or large the tokens' scales are; folding scale_t into p instead would leave the
// top weight at amax/448, subnormal in f16 for rows of small magnitude. Every wait is
// bounded as in the bf16 kernel.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "decode_tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTile = 128;
constexpr int kHalf = kDecodeHalf;
constexpr int kThreads = 448;              // warp 0 TMA, 1 MMA, then per CTA role below
constexpr int kConvBase = 320;             // score CTA: warps 2..9 softmax, 10..13 scale staging
constexpr int kVRowWarps = 4;              // value CTA: warps 2..5 row warps (rescales, epilogue)
constexpr int kVConvWarp = 2 + kVRowWarps; // value CTA: warps 6..13 convert codes to f16
constexpr int kVConvWarps = kThreads / 32 - kVConvWarp;
constexpr uint64_t kWaitNs = kDecodeWaitNs;
constexpr float kRescaleLog2 = 8.f;

constexpr int kE4Chunk = 128 * 64;        // score operand chunk: 128 tokens x 64 codes, 64B swizzle (8 KB)
constexpr int kE4Group = 3 * kE4Chunk;     // score e4m3 group: three chunks (24 KB)
constexpr int kE4Ring = 7;
constexpr int kVE4 = 8 * 64 * 64;          // value e4m3 step: [8 chunks][64 rows][64 B]
constexpr int kVStage = 8 * 64 * 128;      // value f16 stage: [8 chunks][64 rows][128 B], 128B swizzle
constexpr int kPanel = 128 * 128;          // P for 64 tokens: 128 heads x 64 f16
constexpr int kHdr = 512 + 16;
constexpr int kFinBytes = 128 * 2 * 4;
constexpr int kQGroup = 3 * 128 * 128;     // Q staging: three chunk groups of up to 128 rows (bf16)

constexpr uint32_t kQCol = 0;              // score CTA TMEM: Q as e4m3, high parts (144 columns, 4 per column)
constexpr uint32_t kQLoCol = 144;          // score CTA TMEM: Q as e4m3, low parts (144 columns)
constexpr uint32_t kSCol = 288;            // score CTA TMEM: S (128 columns)
constexpr uint32_t kOCol = 0;              // value CTA TMEM: O (512 columns)

//   score CTA
constexpr int S_E4 = 0;
constexpr int S_PANEL = S_E4 + kE4Ring * kE4Group;
constexpr int S_HDR = S_PANEL + 2 * kPanel;
constexpr int S_MX = S_HDR + 1024;
constexpr int kSclBuf = 3 * 128;           // per tile: scale_t, log2 scale_t, 1 / scale_t (fp32)
constexpr int S_SCL = S_MX + 1024;         // [2 tiles][kSclBuf] fp32
constexpr int S_END = S_SCL + 2 * kSclBuf * 4;
//   value CTA
constexpr int V_E4 = 0;
constexpr int V_F16 = V_E4 + 2 * kVE4;
constexpr int V_PANEL = V_F16 + 2 * kVStage;
constexpr int V_HDR = V_PANEL + 2 * kPanel;
constexpr int V_END = V_HDR + 1024;
constexpr int OFF_BAR = (S_END > V_END ? S_END : V_END);
enum Bar {
  SB_E4FULL = 0,                          // [kE4Ring] e4m3 group landed
  SB_E4EMPTY = SB_E4FULL + kE4Ring,       // [kE4Ring] QK MMAs done with it
  SB_QFULL = SB_E4EMPTY + kE4Ring,
  SB_QREADY = SB_QFULL + 1,               // (256)
  SB_SFULL = SB_QREADY + 1,
  SB_SFREE = SB_SFULL + 1,                // (256)
  SB_PFREE = SB_SFREE + 1,                // [2] remote commit from the value CTA
  SB_FLUSH = SB_PFREE + 2,
  SB_SCLREADY = SB_FLUSH + 1,             // [2] tile scales stored (128)
  SB_SCLFREE = SB_SCLREADY + 2,           // [2] tile scales read (256)
  VB_E4FULL = SB_SCLFREE + 2,             // [2]
  VB_E4EMPTY = VB_E4FULL + 2,             // [2] (4 warps)
  VB_F16FULL = VB_E4EMPTY + 2,            // [2] (4 warps)
  VB_F16EMPTY = VB_F16FULL + 2,           // [2] PV MMAs done with the stage
  VB_PFULL = VB_F16EMPTY + 2,             // [2]
  VB_FIN = VB_PFULL + 2,
  VB_FLUSH = VB_FIN + 1,
  VB_CREQ = VB_FLUSH + 1,
  VB_CDONE = VB_CREQ + 1,                 // (256)
  VB_GO = VB_CDONE + 1,
  B_COUNT = VB_GO + 1
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
constexpr int kSmemBytes = OFF_MISC + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kE4Group % 1024 == 0 && S_PANEL % 1024 == 0 && V_F16 % 1024 == 0 && V_PANEL % 1024 == 0,
              "swizzle alignment");
static_assert(3 * kQGroup <= S_PANEL, "Q staging fits below the panels");

enum Cmd { CMD_RESCALE = 2, CMD_DONE = 4 };

__device__ __forceinline__ void give_up(const DecodeParams& p, volatile int* abort_flag, unsigned char* smem,
                                        uint32_t peer) {
  record_status(p.status, MLA_ERR_TIMEOUT);
  *abort_flag = 1;
  st_cluster_u32(mapa(smem_u32(smem + OFF_MISC + 4), peer), 1u);
}

// 16 e4m3 codes → 16 f16 values, each exactly 2^-8 times the code's value, as two
// 16-byte chunks. An e4m3 code s.eeee.mmm has exponent bias 7, f16 has 15; the f16 with
// sign s, exponent field eeee (top bit zero) and mantissa mmm0000000 is therefore the
// code's value times 2^-8, for normal codes (eeee > 0) and for subnormal ones alike
// (both sides subnormal, m · 2^-9 → m · 2^-17). So each code needs only its seven low
// bits moved up by 7 and its sign bit moved up by 8: two byte permutes and a shift-add
// per pair, where a conversion instruction per pair was the converters' bottleneck.
// The NaN codes (0x7F, 0xFF) map to ±480 · 2^-8; the cache holds none (the quantiser
// saturates at ±448).
__device__ __forceinline__ void e4m3x16_to_f16(uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t mag = w[k] & 0x7F7F7F7Fu, sgn = w[k] & 0x80808080u;
    o[2 * k] = (__byte_perm(mag, 0u, 0x4140) << 7) + __byte_perm(sgn, 0u, 0x1404);       // codes 0, 1
    o[2 * k + 1] = (__byte_perm(mag, 0u, 0x4342) << 7) + __byte_perm(sgn, 0u, 0x3424);   // codes 2, 3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Converts the 16 codes at `src` (columns 16 c16 .. 16 c16 + 15 of an e4m3 row) into
// 16-byte units 2 c16 and 2 c16 + 1 of the 128B-swizzled f16 row `row` at `dst_row`;
// zero when `valid` is false. The converters hand out units so that a warp reads 512
// contiguous bytes (eight 64-byte rows) per load and its stores hit each bank group
// four times: both are conflict-free.
__device__ __forceinline__ void convert_unit(const unsigned char* src, unsigned char* dst_row, int row, int c16,
                                             bool valid) {
  uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
  if (valid) e4m3x16_to_f16(*reinterpret_cast<const uint4*>(src), lo, hi);
  *reinterpret_cast<uint4*>(dst_row + (((2 * c16) ^ (row & 7)) << 4)) = lo;
  *reinterpret_cast<uint4*>(dst_row + (((2 * c16 + 1) ^ (row & 7)) << 4)) = hi;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_fp8_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap e4s_map,
                     const __grid_constant__ CUtensorMap e4v_map, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap omap, float scale_log2) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x >> 1;
  // uniform schedule: split s of S_used, written to slot s of S (slots S_used .. S - 1
  // are marked unused by the last split)
  const int b = unit / p.S_used, s = unit % p.S_used;
  const int L = max(p.seq_lens[b], 0);
  int st, en;
  split_range(L, p.S_used, s, &st, &en);
  const int n_tiles = (en - st + kTile - 1) / kTile;
  const int n_halves = 2 * n_tiles;
  griddep_launch_dependents();

  if (n_tiles == 0) {   // empty split: nothing crosses the cluster
    griddep_wait();
    if (rank == 1) {
      float* o = p.o_part + ((int64_t)b * p.S + s) * p.n_h * kLatent;
      for (int i = threadIdx.x; i < p.n_h * kLatent / 4; i += kThreads)
        reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int from = s == p.S_used - 1 ? s : p.S;   // this slot and the unused ones after it
      for (int i = threadIdx.x; i < p.n_h; i += kThreads) p.lse_part[((int64_t)b * p.S + s) * p.n_h + i] = -INFINITY;
      for (int i = threadIdx.x; i < (p.S - from - 1) * p.n_h && from < p.S; i += kThreads)
        p.lse_part[((int64_t)b * p.S + from + 1) * p.n_h + i] = -INFINITY;
    }
    return;
  }
  if (smem_u32(smem) & 1023u) {
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
    for (int k = 0; k < kE4Ring; ++k) {
      mbar_init(&bars[SB_E4FULL + k], 1);
      mbar_init(&bars[SB_E4EMPTY + k], 1);
    }
    mbar_init(&bars[SB_QFULL], 1);
    mbar_init(&bars[SB_QREADY], 256);
    mbar_init(&bars[SB_SFULL], 1);
    mbar_init(&bars[SB_SFREE], 256);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[SB_PFREE + k], 1);
      mbar_init(&bars[SB_SCLREADY + k], 128);
      mbar_init(&bars[SB_SCLFREE + k], 256);
      mbar_init(&bars[VB_E4FULL + k], 1);
      mbar_init(&bars[VB_E4EMPTY + k], kVConvWarps);
      mbar_init(&bars[VB_F16FULL + k], kVConvWarps);
      mbar_init(&bars[VB_F16EMPTY + k], 1);
      mbar_init(&bars[VB_PFULL + k], 1);
    }
    mbar_init(&bars[SB_FLUSH], 1);
    mbar_init(&bars[VB_FIN], 1);
    mbar_init(&bars[VB_FLUSH], 1);
    mbar_init(&bars[VB_CREQ], 1);
    mbar_init(&bars[VB_CDONE], 32 * kVRowWarps);
    mbar_init(&bars[VB_GO], 1);
    if (rank == 1) {
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
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (rank == 0) {
    // =============================== score CTA =========================================
    if (warp == 0) {
      if (lane == 0) {
        // ---- TMA producer: Q (bf16), then e4m3 groups of 128 tokens x 3 chunks, each
        // chunk a 64B-swizzled [128 tokens][64 codes] block: one box for a contiguous
        // cache, one per page and chunk (64 rows) for a paged one ----
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_norm = l2_policy_evict_normal();   // the value CTA reads the rows again
        prefetch_tmap(&e4s_map);
        prefetch_tmap(&qmap);
        const int qrows = p.n_h < 128 ? p.n_h : 128;
        griddep_wait();   // q_lat comes from the previous kernel
        mbar_arrive_expect_tx(&bars[SB_QFULL], 9 * qrows * 128);
        for (int g = 0; g < 3; ++g)
          tma_load_3d(smem + S_E4 + g * kQGroup, &qmap, &bars[SB_QFULL], 0, b * p.n_h, 3 * g, pol_first);
        // Q is staged over the e4m3 ring: the cache loads start once it sits in TMEM.
        int issued = 0;
        if (!mbar_wait(&bars[SB_QREADY], 0, abort_flag, kWaitNs)) give_up(p, abort_flag, smem, peer);
        HalfInfo h0{}, h1{};
        const bool paged = p.block_table != nullptr;
        for (int k = 0; k < 3 * n_tiles && !*abort_flag; ++k) {
          const int i = k / 3, g = k % 3, e = k % kE4Ring;
          if (k >= kE4Ring &&
              !mbar_wait(&bars[SB_E4EMPTY + e], ((k / kE4Ring) - 1) & 1, abort_flag, kWaitNs)) {
            give_up(p, abort_flag, smem, peer);
            break;
          }
          if (g == 0) {
            h0 = half_info(p, b, st, en, 2 * i, true);
            h1 = half_info(p, b, st, en, 2 * i + 1, true);
          }
          unsigned char* dst = smem + S_E4 + e * kE4Group;
          if (!paged) {   // 128 consecutive rows (those past the split are masked)
            if (h0.load) {
              mbar_arrive_expect_tx(&bars[SB_E4FULL + e], kE4Group);
              tma_load_3d(dst, &e4s_map, &bars[SB_E4FULL + e], 0, h0.row0, 3 * g, pol_norm);
            } else {
              mbar_arrive(&bars[SB_E4FULL + e]);
            }
          } else {        // page 0 → rows 0..63 of each chunk, page 1 → rows 64..127
            const uint32_t bytes = 3 * ((h0.load ? kE4Chunk / 2 : 0) + (h1.load ? kE4Chunk / 2 : 0));
            if (bytes) {
              mbar_arrive_expect_tx(&bars[SB_E4FULL + e], bytes);
              for (int c = 0; c < 3; ++c) {
                if (h0.load) tma_load_3d(dst + c * kE4Chunk, &e4s_map, &bars[SB_E4FULL + e], 0, h0.row0, 3 * g + c, pol_norm);
                if (h1.load)
                  tma_load_3d(dst + c * kE4Chunk + kE4Chunk / 2, &e4s_map, &bars[SB_E4FULL + e], 0, h1.row0, 3 * g + c,
                              pol_norm);
              }
            } else {
              mbar_arrive(&bars[SB_E4FULL + e]);
            }
          }
          issued = k + 1;
        }
        const volatile int never = 0;
        mbar_wait(&bars[SB_QFULL], 0, &never, kWaitNs / 4);
        for (int k = max(0, issued - kE4Ring); k < issued; ++k)
          mbar_wait(&bars[SB_E4FULL + k % kE4Ring], (k / kE4Ring) & 1, &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- S = (Q_hi + Q_lo) · code^T straight on the e4m3 codes: per 32-code step
        // two kind::f8f6f4 MMAs of 128 x 128 x 32, 36 per tile ----
        const uint32_t idq = idesc_e4m3(128, kTile);
        bool ok = mbar_wait(&bars[SB_QREADY], 0, abort_flag, kWaitNs);
        if (ok) mbar_arrive_remote(&bars[VB_GO], 1);
        for (int i = 0; ok && i < n_tiles; ++i) {
          if (i > 0 && !mbar_wait(&bars[SB_SFREE], (i - 1) & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          for (int g = 0; g < 3; ++g) {
            const int k = 3 * i + g, e = k % kE4Ring;
            if (!mbar_wait(&bars[SB_E4FULL + e], (k / kE4Ring) & 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t base = smem_u32(smem + S_E4 + e * kE4Group);
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                // codes 64 (3 g + c) + 32 ks .. + 31: TMEM column (that index) / 4
                const uint32_t col = 16 * (3 * g + c) + 8 * ks;
                const uint64_t bd = sdesc_sw64(base + c * kE4Chunk + 32 * ks, 512);
                mma_ts_f8(tmem + kSCol, tmem + kQCol + col, bd, idq, (g | c | ks) ? 1u : 0u);
                mma_ts_f8(tmem + kSCol, tmem + kQLoCol + col, bd, idq, 1u);
              }
            mma_commit(&bars[SB_E4EMPTY + e]);
          }
          if (!ok) break;
          mma_commit(&bars[SB_SFULL]);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[SB_FLUSH]);
        const volatile int never = 0;
        mbar_wait(&bars[SB_FLUSH], 0, &never, kWaitNs);
      }
    } else if (warp >= 10) {
      // ---- scale warps: each tile's per-token scales (the MMAs read the codes as they
      // are), one row per thread ----
      const int ct = threadIdx.x - kConvBase;
      const int r = ct, hh = r >> 6, rr = r & 63;
      float* scl = reinterpret_cast<float*>(smem + S_SCL);
      bool ok = true;
      // this row's scale, loaded one tile ahead by a predicated load (no select on the
      // loaded value), so that nothing waits for it before the next tile stores it
      auto row_scale = [&](int tile) -> float {
        if (tile >= n_tiles) return 0.f;
        const HalfInfo hi = half_info(p, b, st, en, 2 * tile + hh, false);
        return ld_global_nc_or_zero(p.scales + hi.row0 + rr, hi.load && rr < hi.nvalid);
      };
      float sc_next = row_scale(0);
      for (int i = 0; i < n_tiles && ok; ++i) {
        if (i >= 2 && !mbar_wait(&bars[SB_SCLFREE + (i & 1)], ((i >> 1) - 1) & 1, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        // rows past the split (scale 0) get log2 = -inf and 1/scale = 0; their scores
        // are masked to -inf anyway
        float* sb = scl + (i & 1) * kSclBuf;
        const bool pos = sc_next > 0.f;
        sb[r] = sc_next;
        sb[128 + r] = pos ? __log2f(sc_next) : -INFINITY;
        sb[256 + r] = pos ? __frcp_rn(sc_next) : 0.f;
        mbar_arrive(&bars[SB_SCLREADY + (i & 1)]);
        sc_next = row_scale(i + 1);
      }
      if (!ok) give_up(p, abort_flag, smem, peer);
    } else {
      // ---- softmax: thread (h, j) owns head h, tokens [64 j, 64 j + 64) of each tile ----
      const int q = warp & 3;
      const int h = q * 32 + lane;
      const int j = (warp - 2) >> 2;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      // Q rows → TMEM as two e4m3 parts. Each head's row is first multiplied by a power
      // of two 2^k_h that brings its largest magnitude into [2^7, 2^8); then hi = e4m3(q)
      // and lo = e4m3(q - hi). A bf16 value has 8 significant bits and e4m3 4, so
      // hi + lo is the value exactly down to 2^-9 (e4m3's subnormal step), i.e. for every
      // element within 2^-16 of the head's largest; 2^-k_h comes back in fp32 with the
      // scores (heads beyond n_h are zero).
      const int qrows = p.n_h < 128 ? p.n_h : 128;
      const bool qok = warp_wait(&bars[SB_QFULL], 0, abort_flag);
      uint32_t qmax = 0;   // largest |q| of this thread's chunks, as bf16 magnitude bits
      if (qok && h < p.n_h) {
#pragma unroll 1
        for (int c = j; c < 9; c += 2) {
          const unsigned char* row = smem + S_E4 + (c / 3) * kQGroup + (c % 3) * (qrows * 128) + h * 128;
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((x ^ (h & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) qmax = max(qmax, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
          }
        }
      }
      uint32_t* qmx = reinterpret_cast<uint32_t*>(smem + S_MX);
      qmx[j * 128 + h] = qmax;
      named_sync(1, 256);
      qmax = max(qmx[h], qmx[128 + h]);
      // later writes of this region come after the first tile's vote (a barrier of the
      // same 256 threads), so these reads cannot see them
      const int qexp = (int)((qmax >> 7) & 0xFFu);   // biased bf16 exponent of max |q|
      const int qk = qmax == 0u ? 0 : min(118, max(-126, 134 - qexp));
      const float qmul = __uint_as_float((uint32_t)(127 + qk) << 23);   // 2^k_h
      // 2^-k_h · scale · log2 e (scale_log2 carries the value side's 2^8, which the
      // scores, taken on the codes' own values, do not need)
      const float qsl = scalbnf(scale_log2, -qk - 8);
      if (qok) {
#pragma unroll 1
        for (int c = j; c < 9; c += 2) {
          // 64 elements of chunk c: codes of element 4 w + b in byte b of column 16 c + w
          uint32_t qh[16], ql[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) qh[w] = ql[w] = 0u;
          const unsigned char* row = smem + S_E4 + (c / 3) * kQGroup + (c % 3) * (qrows * 128) + h * 128;
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            uint4 v = h < p.n_h ? *reinterpret_cast<const uint4*>(row + ((x ^ (h & 7)) << 4))
                                : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
              const float2 y = make_float2(f2.x * qmul, f2.y * qmul);
              const __nv_fp8x2_storage_t hi2 = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
              const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi2, __NV_E4M3);
              const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
              const __nv_fp8x2_storage_t lo2 =
                  __nv_cvt_float2_to_fp8x2(make_float2(y.x - hf.x, y.y - hf.y), __NV_SATFINITE, __NV_E4M3);
              const int pi = 4 * x + e;   // elements 2 pi, 2 pi + 1
              qh[pi >> 1] |= (uint32_t)hi2 << (16 * (pi & 1));
              ql[pi >> 1] |= (uint32_t)lo2 << (16 * (pi & 1));
            }
          }
          MLA_TMEM_ST16(trow + kQCol + 16 * c, qh);
          MLA_TMEM_ST16(trow + kQLoCol + 16 * c, ql);
        }
        tmem_wait_st();
      } else {
        give_up(p, abort_flag, smem, peer);
      }
      tc_fence_before();
      mbar_arrive(&bars[SB_QREADY]);

      float m_run = -INFINITY, l_run = 0.f;
      float* mx = reinterpret_cast<float*>(smem + S_MX);
      const float* scl = reinterpret_cast<const float*>(smem + S_SCL);
      const uint32_t panel_remote = mapa(smem_u32(smem + V_PANEL + j * kPanel), 1);
      const uint32_t hdr_remote = mapa(smem_u32(smem + V_HDR), 1);
      const uint32_t pfull_remote = mapa(smem_u32(&bars[VB_PFULL + j]), 1);
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
        const bool sok = warp_wait(&bars[SB_SCLREADY + (i & 1)], (i >> 1) & 1, abort_flag);
        const int nv = (got && sok) ? half_info(p, b, st, en, 2 * i + j, false).nvalid : 0;
        const float* sb = scl + (i & 1) * kSclBuf;
        const float4* sc4 = reinterpret_cast<const float4*>(sb + 64 * j);
        const float4* ls4 = reinterpret_cast<const float4*>(sb + 128 + 64 * j);
        // x_t = s_t · scale_t · 2^-k_h · log2(e)/sqrt(d) is the log2 score of the
        // dequantised token; the softmax runs on y_t = x_t + log2 scale_t, the log2 of
        // its weight on the codes, so that P' = 2^(y_t - m) stays within f16's normal
        // range whatever the token's scale.
#pragma unroll
        for (int t4 = 0; t4 < 16; ++t4) {
          const float4 c4 = sc4[t4], l4 = ls4[t4];
          const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
          const float ll[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 4 * t4 + e;
            sr[t] = __float_as_uint(t < nv ? fmaf(__uint_as_float(sr[t]), cc[e] * qsl, ll[e]) : -INFINITY);
          }
        }
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int t = 8; t < 64; ++t) m8[t & 7] = fmaxf(m8[t & 7], __uint_as_float(sr[t]));
        const float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        float fac = 1.f;
        bool row_rescale = false;
        const uint32_t nneed = named_popc(1, 256, mt > m_run + kRescaleLog2);
        if (nneed) {
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
        // P' = 2^(y - m) goes to the value CTA (f16); the normaliser sums
        // 2^(x - m) = P' / scale_t in fp32.
        // Each 8-token slice is packed and stored at once (the panel must be free first:
        // the value CTA's PV on the previous tile has read it), which keeps the thread
        // within the register budget of a 14-warp CTA.
        if (i > 0) mbar_wait<true>(&bars[SB_PFREE + j], (i - 1) & 1, abort_flag, kWaitNs);
        unsigned char* stg = smem + S_PANEL + j * kPanel;
        unsigned char* hdr = smem + S_HDR;
        float lsum = 0.f;
        const bool live = m_run != -INFINITY;
        const float2 nm2 = make_float2(live ? -m_run : 0.f, live ? -m_run : 0.f);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 8 * c8 + 2 * e;
            const float2 is2 = reinterpret_cast<const float2*>(sb + 256 + 64 * j)[t >> 1];
            float2 pp = make_float2(0.f, 0.f);
            if (live) {
              const float2 xy = fadd2(make_float2(__uint_as_float(sr[t]), __uint_as_float(sr[t + 1])), nm2);
              pp = make_float2(ex2(xy.x), ex2(xy.y));
            }
            acc = ffma2(pp, is2, acc);
            const __half2 v = __floats2half2_rn(pp.x, pp.y);
            pk[e] = *reinterpret_cast<const uint32_t*>(&v);
          }
          *reinterpret_cast<uint4*>(stg + h * 128 + ((c8 ^ (h & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        lsum = acc.x + acc.y;
        l_run += lsum;
        mbar_arrive(&bars[SB_SCLFREE + (i & 1)]);
        if (j == 0) {
          reinterpret_cast<float*>(hdr)[h] = fac;
          if (h == 0) reinterpret_cast<uint32_t*>(hdr + 512)[0] = nres;
        }
        fence_proxy_async_smem();
        named_sync(2 + j, 128);
        if (q == 0 && lane == 0 && !*abort_flag) {
          bulk_copy_to_peer(panel_remote, stg, kPanel, pfull_remote);
          if (j == 0) bulk_copy_to_peer(hdr_remote, hdr, kHdr, pfull_remote);
        }
      }
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
        // ---- TMA producer: e4m3 c_KV of every 64-token step (evict-first: last reader) ----
        const uint64_t pol = l2_policy_evict_first();
        prefetch_tmap(&e4v_map);
        int issued = 0;
        if (!mbar_wait<true>(&bars[VB_GO], 0, abort_flag, kWaitNs)) give_up(p, abort_flag, smem, peer);
        for (int u = 0; u < n_halves && !*abort_flag; ++u) {
          const int e = u & 1;
          if (u >= 2 && !mbar_wait(&bars[VB_E4EMPTY + e], ((u >> 1) - 1) & 1, abort_flag, kWaitNs)) {
            give_up(p, abort_flag, smem, peer);
            break;
          }
          const HalfInfo hi = half_info(p, b, st, en, u, false);
          if (hi.load) {
            mbar_arrive_expect_tx(&bars[VB_E4FULL + e], kVE4);
            tma_load_3d(smem + V_E4 + e * kVE4, &e4v_map, &bars[VB_E4FULL + e], 0, hi.row0, 0, pol);
          } else {
            mbar_arrive(&bars[VB_E4FULL + e]);
          }
          issued = u + 1;
        }
        const volatile int never = 0;
        for (int u = max(0, issued - 2); u < issued; ++u)
          mbar_wait(&bars[VB_E4FULL + (u & 1)], (u >> 1) & 1, &never, kWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---- O += P' · code, 8 MMAs of 128 x 256 x 16 per 64-token step ----
        const uint32_t idv = idesc_f16(128, 256, /*fp16_inputs=*/true, false, true);
        int ncmd = 0, nflush = 0;
        bool ok = true, o_init = false;
        const volatile int never = 0;
        for (int u = 0; u < n_halves; ++u) {
          const int i = u >> 1, j = u & 1, sg = u & 1;
          if (!mbar_wait(&bars[VB_F16FULL + sg], (u >> 1) & 1, abort_flag, kWaitNs) ||
              !mbar_wait<true>(&bars[VB_PFULL + j], i & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          if (i + 1 < n_tiles) mbar_arrive_expect_tx(&bars[VB_PFULL + j], j == 0 ? kPanel + kHdr : kPanel);
          const HalfInfo hi = half_info(p, b, st, en, u, false);
          if (j == 0 && o_init && *reinterpret_cast<const volatile uint32_t*>(smem + V_HDR + 512) != 0u) {
            mma_commit(&bars[VB_FLUSH]);   // O must be quiescent before its rows are rescaled
            if (!mbar_wait(&bars[VB_FLUSH], nflush & 1, &never, kWaitNs)) {
              ok = false;
              break;
            }
            ++nflush;
            *cmd_word = (u << 8) | CMD_RESCALE;
            mbar_arrive(&bars[VB_CREQ]);
            if (!mbar_wait(&bars[VB_CDONE], ncmd & 1, abort_flag, kWaitNs)) {
              ok = false;
              break;
            }
            ++ncmd;
          }
          if (hi.nvalid > 0) {
            tc_fence_after();
            const uint32_t pb = smem_u32(smem + V_PANEL + j * kPanel);
            const uint32_t vb = smem_u32(smem + V_F16 + sg * kVStage);
#pragma unroll
            for (int kk = 0; kk < kHalf / 16; ++kk) {
              const uint64_t a = sdesc_sw128(pb + 32 * kk, 16, 1024);
#pragma unroll
              for (int nh = 0; nh < 2; ++nh) {
                const uint64_t bd = sdesc_sw128(vb + 4 * nh * (64 * 128) + kk * 2048, 64 * 128, 1024);
                mma_ss(tmem + kOCol + 256 * nh, a, bd, idv, (o_init || kk > 0) ? 1u : 0u);
              }
            }
            o_init = true;
          }
          mma_commit(&bars[VB_F16EMPTY + sg]);
          mma_commit_mc(&bars[SB_PFREE + j], 0x1);
        }
        if (!ok) give_up(p, abort_flag, smem, peer);
        mma_commit(&bars[VB_FLUSH]);
        mbar_wait(&bars[VB_FLUSH], nflush & 1, &never, kWaitNs);
        *o_init_word = o_init ? 1 : 0;
        *cmd_word = CMD_DONE;
        mbar_arrive(&bars[VB_CREQ]);
      }
    } else if (warp >= kVConvWarp) {
      // ---- converters: e4m3 step → f16 stage; rows past the split become zero ----
      const int ct = threadIdx.x - 32 * kVConvWarp;
      bool ok = true;
      for (int u = 0; u < n_halves && ok; ++u) {
        const int e = u & 1, sg = u & 1;
        if (!warp_wait(&bars[VB_E4FULL + e], (u >> 1) & 1, abort_flag) ||
            (u >= 2 && !warp_wait(&bars[VB_F16EMPTY + sg], ((u >> 1) - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        const HalfInfo hi = half_info(p, b, st, en, u, false);
        const unsigned char* vsrc = smem + V_E4 + e * kVE4;
        unsigned char* vdst = smem + V_F16 + sg * kVStage;
        // 8 chunks x 64 rows x 64 codes: unit f = 32 kVConvWarps k + ct is chunk f / 256,
        // row (f % 256) / 4
        static_assert(2048 % (32 * kVConvWarps) == 0, "units of a step split evenly over the converters");
#pragma unroll 4
        for (int kk = 0; kk < 2048 / (32 * kVConvWarps); ++kk) {
          const int f = 32 * kVConvWarps * kk + ct, chunk = f >> 8, row = (f & 255) >> 2, c16 = f & 3;
          convert_unit(vsrc + chunk * 4096 + row * 64 + 16 * c16, vdst + chunk * 8192 + row * 128, row, c16,
                       hi.load && row < hi.nvalid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[VB_F16FULL + sg]);
          mbar_arrive(&bars[VB_E4EMPTY + e]);
        }
      }
      if (!ok) give_up(p, abort_flag, smem, peer);
    } else {
      // ---- row warps: rescale commands, then the epilogue ----
      const int q = warp & 3;   // warps 2..5: each lane quarter once, all 512 columns
      const int h = q * 32 + lane;
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
        if (c & CMD_RESCALE) {
          tc_fence_after();
          const float f = reinterpret_cast<const float*>(smem + V_HDR)[h];
          if (__any_sync(0xffffffffu, f != 1.f)) {
            uint32_t rg[32];
#pragma unroll 1
            for (int cc = 0; cc < 16; ++cc) {
              const uint32_t col = kOCol + 32 * cc;
              MLA_TMEM_LD32(trow + col, rg);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) rg[x] = __float_as_uint(__uint_as_float(rg[x]) * f);
              MLA_TMEM_ST32(trow + col, rg);
            }
            tmem_wait_st();
          }
          tc_fence_before();
        }
        mbar_arrive(&bars[VB_CDONE]);
      }
      griddep_wait();   // o_part may still be read by the previous kernel of the stream
      const bool fin_ok = ok && warp_wait<true>(&bars[VB_FIN], 0, abort_flag);
      tc_fence_after();
      const float* fin = reinterpret_cast<const float*>(smem + V_PANEL);
      const float m = fin[2 * h];
      const float l = fin[2 * h + 1];
      const bool good = fin_ok && *o_init_word != 0 && l > 0.f;
      const float inv = good ? 256.f / l : 0.f;   // 2^8 undoes the operand scaling
      // Each row warp owns 32 heads x 512 columns: sixteen 32-column chunks, each scaled,
      // staged 128B-swizzled in a 4 KB buffer of the warp's own and written at once by a
      // TMA store that the warp issues; four buffers per warp rotate, so the stores
      // overlap the TMEM reads of the next chunks.
      const int rows = p.n_h < 128 ? p.n_h : 128;
      const int wrows = rows < 32 ? rows : 32;
      const bool wlive = 32 * q < rows;
      unsigned char* wst = smem + V_F16 + (warp - 2) * 16384;
      const int orow0 = (b * p.S + s) * p.n_h + 32 * q;
#pragma unroll 1
      for (int cc = 0; cc < 16; ++cc) {
        const int chunk = cc;
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
      if (h < p.n_h)
        p.lse_part[((int64_t)b * p.S + s) * p.n_h + h] =
            good ? (m + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
      if (s == p.S_used - 1)   // slots after the last split are unused
        for (int i = threadIdx.x - 64; i < (p.S - p.S_used) * p.n_h; i += 32 * kVRowWarps)
          p.lse_part[((int64_t)b * p.S + p.S_used) * p.n_h + i] = -INFINITY;
      tc_fence_before();
    }
  }

  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  cluster_sync();
}

// 3D map over rows of 576 e4m3 codes seen as (64 codes, row, 9 chunks of 64 codes); a
// box of `box_rows` rows x `box_chunks` chunks lands chunk-major, each chunk a
// [box_rows][64] block, 64B-swizzled for the score side's MMA operands or plain for the
// value side's converters.
bool make_code_map(const void* base, int64_t rows, int box_rows, int box_chunks, bool swizzle, CUtensorMap* map) {
  const uint64_t dims[3] = {64, (uint64_t)rows, (uint64_t)(kRow / 64)};
  const uint64_t strides[2] = {(uint64_t)kRow, 64};
  const uint32_t box[3] = {64, (uint32_t)box_rows, (uint32_t)box_chunks};
  return encode_tiled(tmap_desc(base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box,
                                swizzle ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      map);
}

bool make_q_map(const void* base, int64_t rows, int box_rows, CUtensorMap* map) {
  const uint64_t dims[3] = {64, (uint64_t)rows, (uint64_t)(kRow / 64)};
  const uint64_t strides[2] = {(uint64_t)kRow * 2, 128};
  const uint32_t box[3] = {64, (uint32_t)box_rows, 3};
  return encode_tiled(tmap_desc(base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B),
                      map);
}

// fp32 partial results [rows][512] as (32 values, row, 16 chunks of 32), 128B swizzle;
// a box is `box_rows` rows x one chunk (one row warp's store).
bool make_out_map(float* base, int64_t rows, int box_rows, CUtensorMap* map) {
  const uint64_t dims[3] = {32, (uint64_t)rows, (uint64_t)(kLatent / 32)};
  const uint64_t strides[2] = {(uint64_t)kLatent * 4, 128};
  const uint32_t box[3] = {32, (uint32_t)box_rows, 1};
  return encode_tiled(tmap_desc(base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE),
                      map);
}

}  // namespace

cudaError_t launch_decode_tc_fp8(const DecodeParams& p, cudaStream_t st) {
  const int rows = p.n_h < 128 ? p.n_h : 128;
  CUtensorMap e4s, e4v, qmap, omap;
  // score side: 128 rows x 3 chunks per box (contiguous) or 64 rows x 1 chunk (a page)
  const bool paged = p.block_table != nullptr;
  if (!make_code_map(p.data, p.num_rows, paged ? 64 : kTile, paged ? 1 : 3, true, &e4s) ||
      !make_code_map(p.data, p.num_rows, 64, 8, false, &e4v) ||
      !make_q_map(p.q_lat, (int64_t)p.B * p.n_h, rows, &qmap) ||
      !make_out_map(p.o_part, (int64_t)p.B * p.S * p.n_h, p.n_h < 32 ? p.n_h : 32, &omap))
    return cudaErrorInvalidValue;
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t attr_err = smem_attr_once(decode_tc_fp8_kernel, kSmemBytes, attr_done);
  if (attr_err != cudaSuccess) return attr_err;
  // 2^8: the f16 operands hold 2^-8 times the codes' values
  const float scale_log2 = p.scale * 1.4426950408889634f * 256.f;
  const int64_t ctas = 2ll * p.B * p.S_used;
  return launch_overlapped(decode_tc_fp8_kernel, dim3((unsigned)ctas), dim3(kThreads), kSmemBytes, st, p, e4s, e4v,
                           qmap, omap, scale_log2);
}

}  // namespace mla
