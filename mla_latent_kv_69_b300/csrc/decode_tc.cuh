// Tensor-core (tcgen05 + TMEM + TMA) split-KV decode: host-side entry points.
#pragma once
#include <climits>

#include "common.cuh"
#include "sm100.cuh"

namespace mla {

constexpr uint64_t kDecodeWaitNs = 2000000000ull;   // every mbarrier wait of the decode kernels
constexpr int kDecodeHalf = 64;                     // tokens per value step (= one page)

// 64-token half u of the split [st, en) of sequence b.
struct HalfInfo {
  int row0;     // first cache row (the TMA y coordinate)
  int nvalid;   // tokens of the half that belong to the split
  bool load;    // some token is valid and its rows lie inside the caller's buffers
};

// Block-table entry of half u of the split that starts at token st (-1 past the table;
// unused for contiguous caches). The predicated load writes its register by itself, so
// a role can fetch the next half's entry while it works on this one and only stall, if
// at all, when it uses it.
__device__ __forceinline__ int page_ahead(const DecodeParams& p, int b, int st, int u) {
  if (!p.block_table) return -1;
  const int pi = (st + kDecodeHalf * u) >> 6;
  return sm100::ld_global_nc_or(p.block_table + (int64_t)b * p.max_pages + pi, pi < p.max_pages, -1);
}

// `page` is half u's block-table entry (page_ahead), ignored for contiguous caches.
__device__ __forceinline__ HalfInfo half_info(const DecodeParams& p, int b, int st, int en, int u, bool record,
                                              int page) {
  HalfInfo hi;
  const int t0 = st + kDecodeHalf * u;
  hi.nvalid = max(0, min(kDecodeHalf, en - t0));
  hi.row0 = 0;
  hi.load = hi.nvalid > 0;
  if (!hi.load) return hi;
  bool valid = true;
  if (p.block_table) {
    if (page < 0 || (int64_t)page * kDecodeHalf >= p.num_rows) valid = false;
    else hi.row0 = page * kDecodeHalf;
  } else {
    const int64_t row = (int64_t)b * p.seq_stride + t0;
    if (t0 >= p.seq_stride || row >= p.num_rows) {
      valid = false;
    } else {
      hi.row0 = (int)row;
      const int64_t room = (p.seq_stride - t0) < (p.num_rows - row) ? (p.seq_stride - t0) : (p.num_rows - row);
      if (room < hi.nvalid) hi.nvalid = (int)room;
    }
  }
  if (!valid) {
    if (record) record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    hi.nvalid = 0;
    hi.load = false;
  }
  return hi;
}
__device__ __forceinline__ HalfInfo half_info(const DecodeParams& p, int b, int st, int en, int u, bool record) {
  return half_info(p, b, st, en, u, record, page_ahead(p, b, st, u));
}

// A bounded wait taken by all 32 lanes of a warp together: every lane returns the same
// answer, so warp-collective code after it never runs with lanes missing.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          uint64_t limit_ns = kDecodeWaitNs) {
  const bool ok = sm100::mbar_wait<kCluster>(bar, parity, abort_flag, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------ work schedule ----------------------------------------
// A decode launch assigns the batch's tokens to SM pairs (2-CTA clusters) in pieces; each
// piece is one contiguous token range of one sequence and writes one partial-result slot.
//   uniform  (balanced = 0): pair (b, s) takes split s of S_used uniform splits of b
//            (mla_split_range), slot s; the pair of split S_used - 1 marks the slots
//            S_used .. S - 1 unused.
//   balanced (balanced = 1): one launch of `pairs` persistent pairs. The kernel looks at
//            the batch's 128-token tile counts and takes the cheaper of two plans:
//     tiles  the batch's tiles are laid end to end (sequence by sequence) and pair p
//            takes tiles [p q, (p + 1) q). The quota q is at least ceil(T / pairs) (every
//            pair busy) and, unless S covers the longest sequence tile by tile, at least
//            ceil(T_max / (S - 1)), so that no sequence is cut into more than S pieces. A
//            piece's slot is the index of its pair minus the index of the pair holding
//            the sequence's first tile.
//     splits (only when every sequence has the same tile count) each sequence is cut into
//            n pieces of `per` tiles (the last one shorter), piece s in slot s; unit
//            u = b n + s goes to pair u mod pairs. Cuts then never cost a pair a second
//            piece where the tile plan would.
//   In both plans the pair holding a sequence's last piece marks the later slots unused,
//   and empty sequences are marked by pair b % pairs.
constexpr int kSchedTile = 128;
constexpr int64_t kSchedSwitchTiles = 3;   // a pair's cost of each piece after its first, in tiles

struct Piece {
  int b, st, en;   // sequence and token range [st, en)
  int slot;        // partial-result slot of sequence b
  int fill_from;   // slots fill_from .. S - 1 of b are unused and get lse = -inf (S: none)
};

struct SchedShared {   // the pair's share, computed once per CTA by sched_init
  int64_t c0;          // tile plan: global index of the first tile of sequence b0
  int64_t t_begin, t_end, q;
  int32_t b0;
  int32_t split;       // 0: tile plan; n > 0: split plan with n pieces of `per` tiles
  int32_t per;
  int32_t pad;
};

// Tiles per pair for T tiles in all, the longest sequence T_max tiles long, S slots per
// sequence and `pairs` SM pairs. A piece holds at least one tile, so S >= T_max needs no
// bound; otherwise the quota keeps every sequence within S pieces (with S == 1: one pair
// takes everything).
__host__ __device__ inline int64_t sched_quota(int64_t T, int Tmax, int S, int pairs) {
  int64_t q = (T + pairs - 1) / pairs;
  if (S < Tmax) {
    const int64_t qmin = S >= 2 ? (Tmax + S - 2) / (S - 1) : (T > 0 ? T : 1);
    q = q > qmin ? q : qmin;
  }
  return q < 1 ? 1 : q;
}

// Costs of the two plans for equal lengths (Tm tiles per sequence, B sequences), in
// tiles of the busiest pair plus kSchedSwitchTiles for each of its pieces after the first.
// Tile plan with quota q: a share of q tiles that is not a whole number of sequences
// straddles up to floor((q - 1) / Tm) + 1 sequence ends.
__host__ __device__ inline int64_t sched_tile_cost(int64_t q, int Tm) {
  const uint32_t qq = q > 0x3fffffff ? 0x3fffffffu : (uint32_t)q, t = (uint32_t)Tm;
  const uint32_t extra = qq % t == 0 ? qq / t - 1 : (qq - 1) / t + 1;
  return (int64_t)qq + kSchedSwitchTiles * extra;
}
// Split plan with n pieces per sequence (-1 when n gives the same cut as a smaller n, or
// is out of range).
__host__ __device__ inline int64_t sched_split_cost(int n, int B, int Tm, int S, int pairs) {
  if (n < 1 || n > S || n > Tm || B > (1 << 20)) return -1;
  const uint32_t t = (uint32_t)Tm, per = (t + n - 1) / n;
  if ((t + per - 1) / per != (uint32_t)n) return -1;
  const uint32_t waves = (uint32_t)(((uint64_t)B * n + pairs - 1) / (uint32_t)pairs);
  return (int64_t)waves * per + kSchedSwitchTiles * (int64_t)(waves - 1);
}

// The plan for T tiles in B sequences of Tmin .. Tmax tiles each; `split` is the best
// n of the split plan (the least cost, then the least n; 0 if none) and `split_cost` its
// cost. The fields c0 and b0 are left to the caller.
__host__ __device__ inline void sched_plan(int64_t T, int B, int Tmin, int Tmax, int S, int pairs, int pair,
                                           int split, int64_t split_cost, SchedShared* out) {
  const int64_t q = sched_quota(T, Tmax, S, pairs);
  out->q = q;
  out->t_begin = (int64_t)pair * q;
  out->t_end = (int64_t)(pair + 1) * q < T ? (int64_t)(pair + 1) * q : T;
  out->split = 0;
  out->per = 0;
  if (Tmin != Tmax || Tmin < 1 || split < 1 || split_cost >= sched_tile_cost(q, Tmax)) return;
  out->split = split;
  out->per = (Tmax + split - 1) / split;
}

// Host form of the search over n that the kernel spreads over one warp.
inline void sched_best_split(int B, int Tm, int S, int pairs, int* split, int64_t* cost) {
  *split = 0;
  *cost = -1;
  for (int n = 1; n <= S; ++n) {
    const int64_t c = sched_split_cost(n, B, Tm, S, pairs);
    if (c >= 0 && (*cost < 0 || c < *cost)) {
      *cost = c;
      *split = n;
    }
  }
}

// Block-wide: every thread of the CTA calls it with the same arguments. `scratch` holds
// 16 bytes per thread and is free for the call's duration; the result lands in `out`
// (visible to all threads on return).
__device__ inline void sched_init(const DecodeParams& p, int pair, unsigned char* scratch, SchedShared* out) {
  const int nthr = blockDim.x, tid = threadIdx.x;
  if (!p.balanced) {
    __syncthreads();
    return;
  }
  int64_t* sums = reinterpret_cast<int64_t*>(scratch);
  int* maxs = reinterpret_cast<int*>(scratch + 8 * nthr);
  int* mins = reinterpret_cast<int*>(scratch + 12 * nthr);
  const int K = (p.B + nthr - 1) / nthr;
  const int lo = min(p.B, tid * K), hi = min(p.B, lo + K);
  int64_t sum = 0;
  int mx = 0, mn = INT_MAX;
  for (int b = lo; b < hi; ++b) {
    const int T = (max(p.seq_lens[b], 0) + kSchedTile - 1) / kSchedTile;
    sum += T;
    mx = max(mx, T);
    mn = min(mn, T);
  }
  sums[tid] = sum;
  maxs[tid] = mx;
  mins[tid] = mn;
  __syncthreads();
  if (tid < 32) {   // exclusive prefix over the per-thread sums, total, maximum and minimum
    const int E = (nthr + 31) / 32;
    int64_t run = 0;
    int m = 0, n = INT_MAX;
    for (int i = tid * E; i < min(nthr, tid * E + E); ++i) {
      const int64_t v = sums[i];
      sums[i] = run;
      run += v;
      m = max(m, maxs[i]);
      n = min(n, mins[i]);
    }
    int64_t incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += o;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      n = min(n, __shfl_xor_sync(0xffffffffu, n, off));
    }
    const int64_t excl = incl - run;
    for (int i = tid * E; i < min(nthr, tid * E + E); ++i) sums[i] += excl;
    // split plan: lane l tries n = l + 1, l + 33, ...; the least (cost, n) wins
    int64_t best = -1;
    int bn = 0;
    if (n == m && m >= 1)
      for (int k = tid + 1; k <= p.S && k <= m; k += 32) {
        const int64_t c = sched_split_cost(k, p.B, m, p.S, p.pairs);
        if (c >= 0 && (best < 0 || c < best)) {
          best = c;
          bn = k;
        }
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const int64_t ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int on = __shfl_xor_sync(0xffffffffu, bn, off);
      if (ob >= 0 && (best < 0 || ob < best || (ob == best && on < bn))) {
        best = ob;
        bn = on;
      }
    }
    if (tid == 31) {
      sched_plan(incl, p.B, n, m, p.S, p.pairs, pair, bn, best, out);
      out->b0 = -1;
      out->c0 = 0;
    }
  }
  __syncthreads();
  const int64_t tb = out->t_begin;
  const int64_t ex = sums[tid];
  if (out->split == 0 && tb < out->t_end && ex <= tb && tb < ex + sum) {
    int64_t c = ex;
    for (int b = lo; b < hi; ++b) {
      const int T = (max(p.seq_lens[b], 0) + kSchedTile - 1) / kSchedTile;
      if (tb < c + T) {
        out->b0 = b;
        out->c0 = c;
        break;
      }
      c += T;
    }
  }
  __syncthreads();
}

// Walks the pieces of one pair in order; every role of both CTAs walks the same list.
struct PieceCursor {
  int64_t cb, tile, end, q;
  int b, split, per, step;
  bool done;

  __host__ __device__ void start(const DecodeParams& p, int pair, const SchedShared& sh) {
    split = 0;
    done = false;
    if (p.balanced && sh.split > 0) {
      split = sh.split;
      per = sh.per;
      tile = pair;            // the unit b n + s
      step = p.pairs;
    } else if (p.balanced) {
      b = sh.b0;
      cb = sh.c0;
      tile = sh.t_begin;
      end = sh.b0 >= 0 ? sh.t_end : sh.t_begin;
      q = sh.q;
    } else {
      b = pair / p.S_used;
      tile = pair % p.S_used;   // the split index
    }
  }

  __host__ __device__ bool next(const DecodeParams& p, Piece& pc) {
    if (!p.balanced) {
      if (done) return false;
      done = true;
      const int L = p.seq_lens[b] > 0 ? p.seq_lens[b] : 0;
      pc.b = b;
      pc.slot = (int)tile;
      split_range(L, p.S_used, pc.slot, &pc.st, &pc.en);
      pc.fill_from = pc.slot == p.S_used - 1 ? p.S_used : p.S;
      return true;
    }
    if (split > 0) {
      if (tile >= (int64_t)p.B * split) return false;
      pc.b = (int)((uint32_t)tile / (uint32_t)split);   // tile < B * split < 2^31
      pc.slot = (int)tile - pc.b * split;
      tile += step;
      const int L = p.seq_lens[pc.b] > 0 ? p.seq_lens[pc.b] : 0;
      const int64_t st = (int64_t)pc.slot * per * kSchedTile, en = st + (int64_t)per * kSchedTile;
      pc.st = (int)(st < L ? st : L);
      pc.en = (int)(en < L ? en : L);
      pc.fill_from = pc.slot == split - 1 ? split : p.S;
      if (pc.en <= pc.st || split > p.S) {   // only if seq_lens changed under the launch
#ifdef __CUDA_ARCH__
        record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
#endif
        tile = (int64_t)p.B * split;
        return false;
      }
      return true;
    }
    while (tile < end && b < p.B) {
      const int L = p.seq_lens[b] > 0 ? p.seq_lens[b] : 0;
      const int64_t Tb = (L + kSchedTile - 1) / kSchedTile;
      if (tile >= cb + Tb) {
        cb += Tb;
        ++b;
        continue;
      }
      const int64_t seg_end = end < cb + Tb ? end : cb + Tb;
      pc.b = b;
      pc.st = (int)((tile - cb) * kSchedTile);
      pc.en = (int)((seg_end - cb) * kSchedTile < L ? (seg_end - cb) * kSchedTile : L);
      pc.slot = (int)(tile / q - cb / q);
      pc.fill_from = seg_end == cb + Tb ? pc.slot + 1 : p.S;
      tile = seg_end;
      if (pc.slot >= p.S) {   // only if seq_lens changed under the launch: stop, consistently in every role
#ifdef __CUDA_ARCH__
        record_status(p.status, MLA_ERR_DEVICE_BOUNDS);
#endif
        tile = end;
        return false;
      }
      return true;
    }
    return false;
  }
};

// Balanced schedule: lse = -inf in every slot of the empty sequences b = pair (mod
// pairs), written by threads tid0, tid0 + nthr, ... (o_part is never read for such
// slots). Call it only after the previous kernel of the stream is complete.
__device__ inline void mark_empty_sequences(const DecodeParams& p, int pair, int tid0, int nthr) {
  if (!p.balanced) return;
  for (int b = pair; b < p.B; b += p.pairs) {
    if (p.seq_lens[b] > 0) continue;
    for (int i = tid0; i < p.S * p.n_h; i += nthr) p.lse_part[(int64_t)b * p.S * p.n_h + i] = -INFINITY;
  }
}

// True when the tcgen05 kernels handle this configuration.
bool decode_tc_supported(const DecodeParams& p);
// e4m3 cache: tcgen05 kernel with f16 operands (decode_tc_fp8.cu).
cudaError_t launch_decode_tc_fp8(const DecodeParams& p, cudaStream_t st);
// Launch; max_seq_len sizes nothing on the device side but is kept for heuristics.
cudaError_t launch_decode_tc(const DecodeParams& p, int max_seq_len, cudaStream_t st);
// Uniform split count for B sequences of up to `tiles` 64-token tiles.
int decode_tc_num_splits(int B, int tiles, int n_h, int sms);
// Slots per sequence of the balanced schedule (what num_splits = 0 resolves to).
int decode_balanced_slots(int B, int max_seq_len, int pairs);

}  // namespace mla
