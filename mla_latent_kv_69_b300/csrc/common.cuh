// Shared device/host helpers for the MLA decode library (sm_103a).
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mla.h"

namespace mla {

constexpr int kNope = MLA_D_NOPE;      // 128
constexpr int kRope = MLA_D_ROPE;      // 64
constexpr int kLatent = MLA_D_LATENT;  // 512
constexpr int kRow = MLA_D_ROW;        // 576
constexpr int kQ = MLA_D_Q;            // 192
constexpr int kPage = MLA_PAGE_SIZE;   // 64
constexpr int kMaxDevices = 64;

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Token range of split `s` (of S) of a sequence of L tokens: chunks are whole
// 64-token tiles, front-loaded; trailing splits may be empty.
__host__ __device__ inline void split_range(int L, int S, int s, int* start, int* end) {
  int tiles = ceil_div(L, kPage);
  int chunk = kPage * ceil_div(tiles, S);
  int64_t st = (int64_t)s * chunk;
  if (st > L) st = L;
  int64_t en = st + chunk;
  if (en > L) en = L;
  *start = (int)st;
  *end = (int)en;
}

// First device-side error wins.
__device__ inline void record_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Everything a decode kernel needs, resolved on the host.
struct DecodeParams {
  const __nv_bfloat16* q_lat;   // [B, n_h, 576]
  const void* data;             // cache rows
  const float* scales;          // fp8 per-row scales or nullptr
  const int32_t* block_table;   // [B, max_pages] or nullptr
  const int32_t* seq_lens;      // [B]
  float* o_part;                // [B, S, n_h, 512]
  float* lse_part;              // [B, S, n_h]
  int32_t* status;
  int64_t seq_stride;           // contiguous row stride between sequences
  int64_t num_rows;             // addressable rows
  int32_t max_pages;
  int32_t kv_dtype;             // mla_kv_dtype
  int32_t B, n_h, S;            // S: partial-result slots per sequence (the row stride of o_part)
  int32_t S_used;               // uniform schedule: splits per sequence (<= S)
  int32_t balanced;             // 1: balanced schedule over `pairs` SM pairs; 0: one pair per (b, split)
  int32_t pairs;                // balanced schedule: SM pairs sharing the batch
  float scale;                  // softmax scale (natural-log units)
  uint64_t wait_ns;             // limit of the waits that an abort can end (0: the default, 2 s)
  int32_t stall_loads;          // test hook: the score CTA issues no loads, so its consumers' waits run out
};

// Row index of token t (>= 0) of sequence b, or -1 when the token falls outside the
// caller's buffers (a page id outside the pool, or a length beyond the block table
// or the contiguous stride).
__device__ inline int64_t cache_row(const DecodeParams& p, int b, int t) {
  if (p.block_table == nullptr) {
    if (t >= p.seq_stride) return -1;
    const int64_t row = (int64_t)b * p.seq_stride + t;
    return row < p.num_rows ? row : -1;
  }
  if ((t >> 6) >= p.max_pages) return -1;
  const int32_t page = p.block_table[(int64_t)b * p.max_pages + (t >> 6)];
  const int64_t row = (int64_t)page * kPage + (t & (kPage - 1));
  if (page < 0 || row >= p.num_rows) return -1;
  return row;
}

// RoPE frequencies of the decoupled query/key (mla_rope in include/mla.h, validated).
struct RopeSpec {
  double base, yarn_scale, yarn_alpha, yarn_beta;
  int32_t original_max_pos;
};

// Host-side launchers (one per kernel family); each returns the launch error.
cudaError_t launch_absorb_q(const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const int32_t* pos,
                            int B, int n_h, const RopeSpec& rope, __nv_bfloat16* q_lat, cudaStream_t st);
cudaError_t launch_up_v(const float* o_lat, const __nv_bfloat16* w_uv, int B, int n_h, float* o,
                        cudaStream_t st);
cudaError_t launch_combine(const float* o_part, const float* lse_part, int B, int S, int n_h,
                           float* o_lat, float* lse, cudaStream_t st);
// combine and up_v in one kernel; o_lat and lse may be null (not written)
cudaError_t launch_combine_up_v(const float* o_part, const float* lse_part, int S, const __nv_bfloat16* w_uv, int B,
                                int n_h, float* o, float* o_lat, float* lse, cudaStream_t st);
cudaError_t launch_cache_append(const __nv_bfloat16* h, const __nv_bfloat16* w_dkv, const __nv_bfloat16* w_kr,
                                const int32_t* seq_ids, const int32_t* pos, int T, int d, const RopeSpec& rope,
                                const mla_cache& cache, int num_seqs, __nv_bfloat16* staging, int32_t* status,
                                cudaStream_t st);
cudaError_t launch_multi_token_view(const int32_t* seq_lens, int B, int T, const mla_cache& cache,
                                    int max_pages_out, int32_t* out_lens, int32_t* out_pos, int32_t* out_table,
                                    cudaStream_t st);
cudaError_t launch_quantize_fp8(const __nv_bfloat16* rows, int64_t n, uint8_t* codes, float* scales,
                                cudaStream_t st);

}  // namespace mla

namespace mla {

// Programmatic dependent launch. Every kernel of the decode step lets the next one in
// the stream start launching at its own entry (griddep_launch_dependents) and waits
// for the previous kernel's completion and memory (griddep_wait) only before it reads
// anything that kernel may write; each kernel waits before it finishes, so the order
// stays transitive along the stream. Without a programmatic predecessor the wait
// returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device (the attribute belongs to the device's copy of the kernel). `done` is the call
// site's own flag table.
template <typename... KArgs>
cudaError_t smem_attr_once(void (*kernel)(KArgs...), int bytes, std::atomic<int> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
  return e;
}

// Launch `kernel` so that it may overlap the tail of the previous kernel on `st`.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mla
