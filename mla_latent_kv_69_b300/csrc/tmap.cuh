// Tiled TMA tensor maps, encoded once per description and reused.
//
// Every launch of the library's kernels passes its tensor maps by value; encoding them
// through the driver costs host time on every call, while a serving loop reuses the same
// buffers step after step. A map depends only on its description (base address, element
// type, extents, strides, box, swizzle, L2 promotion), so equal descriptions reuse the
// encoded map from a small process-wide table.
#pragma once
#include <cuda.h>

#include <cstdint>

namespace mla {

struct TmapDesc {
  const void* base;
  uint32_t dtype;           // CUtensorMapDataType
  uint32_t rank;            // 1..5
  uint64_t dims[5];         // elements, innermost first
  uint64_t strides[4];      // bytes, of dims 1 .. rank - 1
  uint32_t box[5];
  uint32_t swizzle;         // CUtensorMapSwizzle
  uint32_t l2promo;         // CUtensorMapL2promotion
  uint32_t pad;
};

// A zero-filled description (the table compares descriptions byte for byte).
TmapDesc tmap_desc(const void* base, CUtensorMapDataType dtype, uint32_t rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle,
                   CUtensorMapL2promotion l2promo);

// Encode (or find) the map of `d`: element strides 1, no interleave, no OOB fill.
// False if the driver entry point is missing or rejects the description.
bool encode_tiled(const TmapDesc& d, CUtensorMap* out);

}  // namespace mla
