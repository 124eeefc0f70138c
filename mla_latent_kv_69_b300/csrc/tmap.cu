// Process-wide table of encoded tensor maps (see tmap.cuh).
#include "tmap.cuh"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

namespace mla {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult qr;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A step of one layer uses about eight maps; the table holds several layers' worth and
// replaces entries round robin.
constexpr int kEntries = 128;
struct Entry {
  TmapDesc desc;
  CUtensorMap map;
  bool used;
};
Entry g_table[kEntries];
int g_next = 0;
int g_last = 0;   // most recent hit or insert: consecutive calls mostly repeat a pattern
std::mutex g_mutex;

}  // namespace

TmapDesc tmap_desc(const void* base, CUtensorMapDataType dtype, uint32_t rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle,
                   CUtensorMapL2promotion l2promo) {
  TmapDesc d;
  std::memset(&d, 0, sizeof(d));
  d.base = base;
  d.dtype = (uint32_t)dtype;
  d.rank = rank;
  for (uint32_t i = 0; i < rank && i < 5; ++i) {
    d.dims[i] = dims[i];
    d.box[i] = box[i];
    if (i + 1 < rank) d.strides[i] = strides[i];
  }
  d.swizzle = (uint32_t)swizzle;
  d.l2promo = (uint32_t)l2promo;
  return d;
}

bool encode_tiled(const TmapDesc& d, CUtensorMap* out) {
  if (d.rank < 1 || d.rank > 5) return false;
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int k = 0; k < kEntries; ++k) {
    const int i = (g_last + k) % kEntries;
    if (g_table[i].used && std::memcmp(&g_table[i].desc, &d, sizeof(TmapDesc)) == 0) {
      *out = g_table[i].map;
      g_last = i + 1;
      return true;
    }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5];
  for (uint32_t i = 0; i < d.rank; ++i) {
    dims[i] = d.dims[i];
    box[i] = d.box[i];
    es[i] = 1;
    if (i + 1 < d.rank) strides[i] = d.strides[i];
  }
  CUtensorMap m;
  if (fn(&m, (CUtensorMapDataType)d.dtype, d.rank, const_cast<void*>(d.base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)d.swizzle, (CUtensorMapL2promotion)d.l2promo,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = g_table[g_next];
  e.desc = d;
  e.map = m;
  e.used = true;
  g_last = g_next + 1;
  g_next = (g_next + 1) % kEntries;
  *out = m;
  return true;
}

}  // namespace mla
