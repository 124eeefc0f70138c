// mla_multi_token_view: T new query tokens per sequence decoded as B*T sequences that
// share the cache. Query j of sequence b is sequence v = b T + j of the view; it sits at
// position L_b - T + j and sees the cache tokens 0 .. L_b - T + j ("DeepSeek-V2 机制拆解",
// §长上下文推理的第一瓶颈: each new token attends to every earlier one). The view is a
// paged cache over the same rows: sequence v's block-table row is sequence b's (a paged
// cache) or the 64-row pages of b's contiguous rows, so the decode kernels serve it as
// any paged batch; no cache byte is copied.
#include "common.cuh"

namespace mla {
namespace {

__global__ void multi_token_view_kernel(const int32_t* __restrict__ seq_lens, int B, int T,
                                        const int32_t* __restrict__ table_in, int max_pages_in,
                                        int64_t pages_per_seq, int max_pages_out, int32_t* __restrict__ out_lens,
                                        int32_t* __restrict__ out_pos, int32_t* __restrict__ out_table) {
  griddep_launch_dependents();
  griddep_wait();   // seq_lens may come from the previous kernel
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)B * T * max_pages_out) return;
  const int v = (int)(idx / max_pages_out), pg = (int)(idx % max_pages_out);
  const int b = v / T, j = v - b * T;
  if (pg == 0) {
    const int L = max(seq_lens[b], 0);
    const int seen = max(L - T + j + 1, 0);   // tokens query j sees
    out_lens[v] = seen;
    out_pos[v] = max(seen - 1, 0);
  }
  int32_t page;
  if (table_in)
    page = pg < max_pages_in ? table_in[(int64_t)b * max_pages_in + pg] : -1;
  else
    page = pg < pages_per_seq ? (int32_t)((int64_t)b * pages_per_seq + pg) : -1;
  out_table[idx] = page;
}

}  // namespace

cudaError_t launch_multi_token_view(const int32_t* seq_lens, int B, int T, const mla_cache& cache,
                                    int max_pages_out, int32_t* out_lens, int32_t* out_pos, int32_t* out_table,
                                    cudaStream_t st) {
  const int64_t n = (int64_t)B * T * max_pages_out;
  const int threads = 256;
  const int64_t pages_per_seq = cache.block_table ? 0 : cache.seq_stride_tokens / kPage;
  return launch_overlapped(multi_token_view_kernel, dim3((unsigned)ceil_div64(n, threads)), dim3(threads), 0, st,
                           seq_lens, B, T, cache.block_table, cache.max_pages, pages_per_seq, max_pages_out, out_lens,
                           out_pos, out_table);
}

}  // namespace mla
