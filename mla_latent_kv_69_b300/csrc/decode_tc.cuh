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
