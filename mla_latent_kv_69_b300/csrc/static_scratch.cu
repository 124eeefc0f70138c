// mla_decode_combine_static: the decode and the merge of its split partials in one
// call that allocates nothing.
//
// mla_decode_fwd writes per-split partial results that only mla_combine reads, and a
// normal caller allocates that buffer. Some callers cannot allocate device memory:
// an extension running under a host framework that has already reserved the GPU's
// memory for its own pools and hands the extension no allocator (a cudaMalloc there
// fails or fragments the framework's reservation), or latency-critical code that
// cannot take the device-wide synchronisation cudaMalloc may imply. For them the
// partials live in one fixed device array of this library, MLA_STATIC_SCRATCH_BYTES
// per GPU, which every GPU that loads the library holds until the process exits.
//
// On the host the array's name is only a stand-in symbol, not a device address, so
// the address is looked up with cudaGetSymbolAddress once per device (and again after a
// device reset has replaced the device's context), with that device current, by the
// first call made there; that first call should come before any stream capture. Every call uses the same array and leaves its partials there,
// so calls that overlap on the GPU (concurrent streams, or several host threads)
// race and must be serialised by the caller.
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"

namespace mla {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Unique id of the calling thread's current context (0 when it cannot be read). A
// device reset destroys the primary context; the next one reloads the module, and the
// array may then sit at another address, so the cached address is keyed on this id.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_static_scratch on the current device (nullptr on failure). It is
// looked up once per device and context; without a readable context id it is looked up
// on every call.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  static unsigned long long ctx_of[kMaxDevices] = {0};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  const unsigned long long ctx = current_context_id();   // 0 before the context exists
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {   // makes the context current
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
    ctx_of[dev] = current_context_id();
  }
  return addr[dev];
}

inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace mla

extern "C" {

mla_status mla_decode_combine_static(const void* q_lat, const mla_cache* cache, const int32_t* seq_lens, int B,
                                     int n_h, int max_seq_len, float softmax_scale, int num_splits, float* o_lat,
                                     float* lse, int32_t* status, cudaStream_t stream) {
  using namespace mla;
  if (!q_lat || !cache || !seq_lens || !o_lat) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o_lat) & 15u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || B > 65535 || num_splits < 0 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
  if (!(n_h == 16 || n_h == 32 || n_h == 64 || n_h == 128)) return n_h > 0 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (max_seq_len < 0) return MLA_ERR_INVALID_ARG;
  const int S = num_splits == 0 ? mla_num_splits(B, max_seq_len, n_h) : num_splits;
  const size_t part_bytes = round256((size_t)B * S * n_h * kLatent * sizeof(float));
  const size_t lse_bytes = round256((size_t)B * S * n_h * sizeof(float));
  if (part_bytes + lse_bytes > (size_t)MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_address());
  if (!scratch) return MLA_ERR_CUDA;
  float* o_part = reinterpret_cast<float*>(scratch);
  float* lse_part = reinterpret_cast<float*>(scratch + part_bytes);
  // Every (sequence, slot, head) lse entry is written by the decode before the merge
  // reads it (-inf for a slot without tokens, whose o_part the merge skips), so nothing
  // needs clearing.
  const mla_status st = mla_decode_fwd(q_lat, cache, seq_lens, B, n_h, max_seq_len, softmax_scale, num_splits,
                                       o_part, lse_part, status, stream);
  if (st != MLA_OK) return st;
  return mla_combine(o_part, lse_part, B, S, n_h, o_lat, lse, stream);
}

}  // extern "C"
