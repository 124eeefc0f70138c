// Tensor-core (tcgen05 + TMEM + TMA) split-KV decode: host-side entry points.
#pragma once
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

// For a paged cache (the variable-length layout) and batches up to kLptMaxB, clusters are
// handed out longest sequence first: cluster r serves split r % S of the sequence whose
// rank in the order (length descending, index ascending) is r / S. The splits of one
// sequence are equal, so the longest units start first and the last wave holds the
// shortest ones. Contiguous caches and larger batches keep the index order (the ranking
// costs every unit ~1.5 us of start-up, measured, which uniform lengths do not repay).
// Returns the sequence and stores its
// length (clamped at 0) in *len. `scratch` is kLptMaxB + 1 ints of shared memory that
// nothing writes until the caller's next CTA barrier; every thread of the CTA calls
// this (it synchronises the CTA twice).
constexpr int kLptMaxB = 256;
__device__ __forceinline__ int lpt_sequence(const DecodeParams& p, int r, int* scratch, int* len) {
  const int seq_rank = r / p.S;
  if (p.B > kLptMaxB || !p.block_table) {
    *len = max(p.seq_lens[seq_rank], 0);
    return seq_rank;
  }
  for (int c = threadIdx.x; c < p.B; c += blockDim.x) scratch[c] = max(p.seq_lens[c], 0);
  __syncthreads();
  for (int c = threadIdx.x; c < p.B; c += blockDim.x) {
    const int lc = scratch[c];
    int rk = 0;
    for (int o = 0; o < p.B; ++o) rk += (scratch[o] > lc || (scratch[o] == lc && o < c)) ? 1 : 0;
    if (rk == seq_rank) scratch[kLptMaxB] = c;
  }
  __syncthreads();
  const int b = scratch[kLptMaxB];
  *len = scratch[b];
  return b;
}

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
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = sm100::mbar_wait<kCluster>(bar, parity, abort_flag, kDecodeWaitNs);
  return __all_sync(0xffffffffu, ok);
}

// True when the tcgen05 kernels handle this configuration.
bool decode_tc_supported(const DecodeParams& p);
// e4m3 cache: tcgen05 kernel with f16 operands (decode_tc_fp8.cu).
cudaError_t launch_decode_tc_fp8(const DecodeParams& p, cudaStream_t st);
// Launch; max_seq_len sizes nothing on the device side but is kept for heuristics.
cudaError_t launch_decode_tc(const DecodeParams& p, int max_seq_len, cudaStream_t st);
// Split count for B sequences of up to `tiles` 64-token tiles.
int decode_tc_num_splits(int B, int tiles, int n_h, int sms);

}  // namespace mla
