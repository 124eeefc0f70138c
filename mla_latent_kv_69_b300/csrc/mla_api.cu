// The library's extern "C" boundary: host-side validation, then one launch per call
// on the caller's stream. Validation touches no CUDA API, so a rejected call has no
// side effect and works without a GPU.
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "decode_tc.cuh"
#include "mla_test.h"

namespace {

using namespace mla;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_heads(int n_h) { return n_h == 16 || n_h == 32 || n_h == 64 || n_h == 128; }
inline mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

constexpr int kMaxBatch = 65535;   // grid dimensions carry B

// Per-device SM count, queried once per device.
int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 148;
  }
  std::lock_guard<std::mutex> g(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 148;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Uniform split count of the e4m3 decode (one SM pair per (sequence, split)). Its
// 128-token tile takes ~3.6 us on the score CTA's 8-bit MMAs and a unit ~15 us to start
// and drain (timestamps of the kernel at B = 128 x 8192), and every split adds an n_h x
// 2 KB partial that the merge reads back (~0.13 us per (sequence, split) at 128 heads
// over the GPU); the count minimises waves x unit time plus those reads.
int e4m3_num_splits(int B, int max_seq_len, int n_h, int pairs) {
  const int t = (max_seq_len + 127) / 128;
  if (t <= 1 || pairs < 1) return 1;
  int best = 1;
  double best_us = 1e30;
  for (int S = 1; S <= t && S <= MLA_MAX_SPLITS; ++S) {
    const int per = (t + S - 1) / S;
    const int waves = (B * S + pairs - 1) / pairs;
    const double us = waves * (per * 3.6 + 15.0) + 0.13 * (double)B * S * n_h / 128.0;
    if (us < best_us - 1e-9) {
      best_us = us;
      best = S;
    }
  }
  return best;
}

// A validated mla_rope: base > 1; plain (yarn_scale = 1) or YaRN with scale > 1,
// 0 <= alpha < beta and original_max_pos >= 1.
bool rope_spec(const mla_rope* r, RopeSpec* out) {
  if (!r || r->reserved != 0) return false;
  if (!(r->base > 1.f) || !std::isfinite(r->base)) return false;
  if (!(r->yarn_scale >= 1.f) || !std::isfinite(r->yarn_scale)) return false;
  if (r->yarn_scale > 1.f) {
    if (!(r->yarn_alpha >= 0.f) || !(r->yarn_beta > r->yarn_alpha) || !std::isfinite(r->yarn_beta)) return false;
    if (r->original_max_pos < 1) return false;
  }
  *out = RopeSpec{(double)r->base, (double)r->yarn_scale, (double)r->yarn_alpha, (double)r->yarn_beta,
                  r->original_max_pos};
  return true;
}

}  // namespace

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument (null, misaligned or out-of-range)";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: valid but unsupported configuration";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: caller buffer too small or a fixed limit exceeded";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: the CUDA runtime reported an error";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded device-side wait gave up";
    case MLA_ERR_DEVICE_BOUNDS: return "MLA_ERR_DEVICE_BOUNDS: a page id fell outside the cache pool";
    default: return "unknown mla_status";
  }
}

mla_status mla_split_range(int seq_len, int num_splits, int split, int* start, int* end) {
  if (!start || !end || seq_len < 0 || num_splits < 1 || num_splits > MLA_MAX_SPLITS || split < 0 ||
      split >= num_splits)
    return MLA_ERR_INVALID_ARG;
  split_range(seq_len, num_splits, split, start, end);
  return MLA_OK;
}

int mla_decode_kernel(int kv_dtype, int n_h) {
  if (!valid_heads(n_h) || (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)) return -1;
  DecodeParams p{};
  p.kv_dtype = kv_dtype;
  p.n_h = n_h;
  p.num_rows = 1;
  if (!decode_tc_supported(p)) return -1;
  return kv_dtype == MLA_KV_BF16 ? MLA_KERNEL_TC_BF16 : MLA_KERNEL_TC_E4M3;
}

int mla_num_splits(int B, int max_seq_len, int n_h) {
  if (B < 1 || max_seq_len < 0 || !valid_heads(n_h)) return 1;
  return decode_balanced_slots(B, max_seq_len, sm_count() / 2);
}

mla_status mla_absorb_q(const void* q, const void* w_uk, const int32_t* pos, int B, int n_h,
                        float rope_base, void* q_lat, cudaStream_t stream) {
  const mla_rope r = {rope_base, 1.f, 0.f, 0.f, 0, 0};
  return mla_absorb_q_ex(q, w_uk, pos, B, n_h, &r, q_lat, stream);
}

mla_status mla_absorb_q_ex(const void* q, const void* w_uk, const int32_t* pos, int B, int n_h,
                           const mla_rope* rope, void* q_lat, cudaStream_t stream) {
  if (!q || !w_uk || !pos || !q_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(w_uk) || !aligned16(q_lat) || !aligned16(pos)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(n_h)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  RopeSpec spec;
  if (!rope_spec(rope, &spec)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_absorb_q(static_cast<const __nv_bfloat16*>(q),
                                     static_cast<const __nv_bfloat16*>(w_uk), pos, B, n_h, spec,
                                     static_cast<__nv_bfloat16*>(q_lat), stream));
}

}  // extern "C"

namespace {

// mla_decode_fwd with the test hooks of DecodeParams (wait limit, withheld loads).
mla_status decode_fwd_impl(const void* q_lat, const mla_cache* cache, const int32_t* seq_lens, int B, int n_h,
                           int max_seq_len, float softmax_scale, int num_splits, float* o_part, float* lse_part,
                           int32_t* status, cudaStream_t stream, uint64_t wait_ns, int stall_loads) {
  if (!q_lat || !cache || !seq_lens || !o_part || !lse_part) return MLA_ERR_INVALID_ARG;
  if (!cache->data || cache->reserved != 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_lat) || !aligned16(cache->data) || !aligned16(o_part) || !aligned16(lse_part) ||
      !aligned16(seq_lens))
    return MLA_ERR_INVALID_ARG;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(n_h)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (max_seq_len < 0 || max_seq_len > (INT_MAX / 2)) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (cache->dtype == MLA_KV_BF16) {
    if (cache->scales) return MLA_ERR_INVALID_ARG;
  } else if (cache->dtype == MLA_KV_FP8_E4M3) {
    if (!cache->scales || !aligned16(cache->scales)) return MLA_ERR_INVALID_ARG;
  } else {
    return MLA_ERR_INVALID_ARG;
  }
  if (cache->num_rows < 0) return MLA_ERR_INVALID_ARG;
  if (cache->block_table) {
    if (cache->page_size != kPage) return cache->page_size > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    if (!aligned16(cache->block_table)) return MLA_ERR_INVALID_ARG;
    if (cache->max_pages < ceil_div(max_seq_len, kPage) || cache->max_pages < 1) return MLA_ERR_INVALID_ARG;
    if (cache->num_rows % kPage) return MLA_ERR_INVALID_ARG;
  } else {
    if (cache->seq_stride_tokens < max_seq_len) return MLA_ERR_INVALID_ARG;
    if (cache->num_rows < (int64_t)(B - 1) * cache->seq_stride_tokens + max_seq_len) return MLA_ERR_INVALID_ARG;
  }
  const int S = num_splits == 0 ? mla_num_splits(B, max_seq_len, n_h) : num_splits;

  DecodeParams p{};
  p.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
  p.data = cache->data;
  p.scales = cache->scales;
  p.block_table = cache->block_table;
  p.seq_lens = seq_lens;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.status = status;
  p.seq_stride = cache->seq_stride_tokens;
  p.num_rows = cache->num_rows;
  p.max_pages = cache->max_pages;
  p.kv_dtype = cache->dtype;
  p.B = B;
  p.n_h = n_h;
  p.S = S;
  p.S_used = S;
  p.balanced = 0;
  p.pairs = 0;
  if (num_splits == 0) {
    if (cache->dtype == MLA_KV_BF16 && cache->block_table) {
      // paged caches (ragged batches): the persistent kernel shares the batch's tiles out
      // evenly over all SM pairs
      p.balanced = 1;
      p.pairs = sm_count() / 2 > 0 ? sm_count() / 2 : 1;
    } else {
      // contiguous caches and e4m3: one pair per (sequence, split), uniform splits sized
      // for the longest sequence, within the slots
      const int tiles = ceil_div(max_seq_len, kPage);
      const int su = tiles <= 1                          ? 1
                     : cache->dtype == MLA_KV_FP8_E4M3 ? e4m3_num_splits(B, max_seq_len, n_h, sm_count() / 2)
                                                       : decode_tc_num_splits(B, tiles, n_h, sm_count());
      p.S_used = su < S ? su : S;
    }
  }
  p.scale = softmax_scale;
  p.wait_ns = wait_ns;
  p.stall_loads = stall_loads;
  // TMA coordinates are 32-bit: a cache of 2^31 rows (over 1 TB) is not served.
  if (!decode_tc_supported(p)) return MLA_ERR_UNSUPPORTED;
  return cuda_status(p.kv_dtype == MLA_KV_BF16 ? launch_decode_tc(p, max_seq_len, stream)
                                               : launch_decode_tc_fp8(p, stream));
}

}  // namespace

extern "C" {

mla_status mla_decode_fwd(const void* q_lat, const mla_cache* cache, const int32_t* seq_lens, int B,
                          int n_h, int max_seq_len, float softmax_scale, int num_splits, float* o_part,
                          float* lse_part, int32_t* status, cudaStream_t stream) {
  return decode_fwd_impl(q_lat, cache, seq_lens, B, n_h, max_seq_len, softmax_scale, num_splits, o_part, lse_part,
                         status, stream, 0, 0);
}

mla_status mla_test_decode_stalled(const void* q_lat, const mla_cache* cache, const int32_t* seq_lens, int B,
                                   int n_h, int max_seq_len, float softmax_scale, int num_splits, float* o_part,
                                   float* lse_part, int32_t* status, uint64_t wait_ns, cudaStream_t stream) {
  if (!cache || cache->dtype != MLA_KV_BF16 || !status) return MLA_ERR_INVALID_ARG;
  if (wait_ns < 1000 || wait_ns > kDecodeWaitNs) return MLA_ERR_INVALID_ARG;
  return decode_fwd_impl(q_lat, cache, seq_lens, B, n_h, max_seq_len, softmax_scale, num_splits, o_part, lse_part,
                         status, stream, wait_ns, 1);
}

mla_status mla_combine(const float* o_part, const float* lse_part, int B, int num_splits, int n_h,
                       float* o_lat, float* lse, cudaStream_t stream) {
  if (!o_part || !lse_part || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch || num_splits < 1 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(n_h)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  return cuda_status(launch_combine(o_part, lse_part, B, num_splits, n_h, o_lat, lse, stream));
}

mla_status mla_up_v(const float* o_lat, const void* w_uv, int B, int n_h, float* o, cudaStream_t stream) {
  if (!o_lat || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(n_h)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  return cuda_status(launch_up_v(o_lat, static_cast<const __nv_bfloat16*>(w_uv), B, n_h, o, stream));
}

mla_status mla_combine_up_v(const float* o_part, const float* lse_part, int B, int num_splits, int n_h,
                            const void* w_uv, float* o, float* o_lat, float* lse, cudaStream_t stream) {
  if (!o_part || !lse_part || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_part) || !aligned16(lse_part) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
  if (o_lat && !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch || num_splits < 1 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (!valid_heads(n_h)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  return cuda_status(launch_combine_up_v(o_part, lse_part, num_splits, static_cast<const __nv_bfloat16*>(w_uv), B,
                                         n_h, o, o_lat, lse, stream));
}

mla_status mla_cache_append(const void* h, const void* w_dkv, const void* w_kr, const int32_t* seq_ids,
                            const int32_t* pos, int T, int d_model, float rope_base, const mla_cache* cache,
                            int num_seqs, void* staging, int32_t* status, cudaStream_t stream) {
  const mla_rope r = {rope_base, 1.f, 0.f, 0.f, 0, 0};
  return mla_cache_append_ex(h, w_dkv, w_kr, seq_ids, pos, T, d_model, &r, cache, num_seqs, staging, status, stream);
}

mla_status mla_cache_append_ex(const void* h, const void* w_dkv, const void* w_kr, const int32_t* seq_ids,
                               const int32_t* pos, int T, int d_model, const mla_rope* rope, const mla_cache* cache,
                               int num_seqs, void* staging, int32_t* status, cudaStream_t stream) {
  if (!h || !w_dkv || !w_kr || !seq_ids || !pos || !cache || !cache->data) return MLA_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_dkv) || !aligned16(w_kr) || !aligned16(cache->data) || !aligned16(seq_ids) ||
      !aligned16(pos))
    return MLA_ERR_INVALID_ARG;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxBatch * 128) return MLA_ERR_INVALID_ARG;
  if (d_model < 512 || d_model > 32768 || d_model % 512) return d_model > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  RopeSpec spec;
  if (!rope_spec(rope, &spec)) return MLA_ERR_INVALID_ARG;
  if (num_seqs < 1 || cache->reserved != 0 || cache->num_rows < 1) return MLA_ERR_INVALID_ARG;
  if (cache->dtype == MLA_KV_BF16) {
    if (cache->scales) return MLA_ERR_INVALID_ARG;
  } else if (cache->dtype == MLA_KV_FP8_E4M3) {
    if (!cache->scales || !aligned16(cache->scales) || !staging || !aligned16(staging)) return MLA_ERR_INVALID_ARG;
  } else {
    return MLA_ERR_INVALID_ARG;
  }
  if (cache->block_table) {
    if (cache->page_size != kPage) return cache->page_size > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    if (!aligned16(cache->block_table) || cache->max_pages < 1 || cache->num_rows % kPage) return MLA_ERR_INVALID_ARG;
  } else if (cache->seq_stride_tokens < 1) {
    return MLA_ERR_INVALID_ARG;
  }
  if (T == 0) return MLA_OK;
  return cuda_status(launch_cache_append(static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(w_dkv),
                                         static_cast<const __nv_bfloat16*>(w_kr), seq_ids, pos, T, d_model, spec,
                                         *cache, num_seqs, static_cast<__nv_bfloat16*>(staging), status, stream));
}

mla_status mla_multi_token_view(const mla_cache* cache, const int32_t* seq_lens, int B, int T, int max_seq_len,
                                int32_t* view_seq_lens, int32_t* view_pos, int32_t* view_block_table,
                                int view_max_pages, mla_cache* view, cudaStream_t stream) {
  if (!cache || !cache->data || !seq_lens || !view_seq_lens || !view_pos || !view_block_table || !view)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(seq_lens) || !aligned16(view_seq_lens) || !aligned16(view_pos) || !aligned16(view_block_table))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || T < 1 || (int64_t)B * T > kMaxBatch || max_seq_len < 0) return MLA_ERR_INVALID_ARG;
  if (view_max_pages < ceil_div(max_seq_len, kPage) || view_max_pages < 1) return MLA_ERR_INVALID_ARG;
  if (cache->reserved != 0 || cache->num_rows < 1) return MLA_ERR_INVALID_ARG;
  if (cache->block_table) {
    if (cache->page_size != kPage) return cache->page_size > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    if (!aligned16(cache->block_table) || cache->max_pages < 1) return MLA_ERR_INVALID_ARG;
  } else {
    // the view pages a contiguous cache in place: whole 64-row pages per sequence
    if (cache->seq_stride_tokens < max_seq_len || cache->seq_stride_tokens < 1) return MLA_ERR_INVALID_ARG;
    if (cache->seq_stride_tokens % kPage || cache->num_rows % kPage) return MLA_ERR_UNSUPPORTED;
  }
  *view = *cache;
  view->block_table = view_block_table;
  view->page_size = kPage;
  view->max_pages = view_max_pages;
  view->seq_stride_tokens = 0;
  return cuda_status(launch_multi_token_view(seq_lens, B, T, *cache, view_max_pages, view_seq_lens, view_pos,
                                             view_block_table, stream));
}

mla_status mla_quantize_fp8(const void* rows, int64_t num_rows, uint8_t* codes, float* scales,
                            cudaStream_t stream) {
  if (!rows || !codes || !scales) return MLA_ERR_INVALID_ARG;
  if (!aligned16(rows) || !aligned16(codes) || !aligned16(scales)) return MLA_ERR_INVALID_ARG;
  if (num_rows < 0 || num_rows > ((int64_t)1 << 33)) return MLA_ERR_INVALID_ARG;
  if (num_rows == 0) return MLA_OK;
  return cuda_status(launch_quantize_fp8(static_cast<const __nv_bfloat16*>(rows), num_rows, codes, scales, stream));
}

}  // extern "C"
