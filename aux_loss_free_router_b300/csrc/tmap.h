// Host-side creation of TMA tensor maps.  The driver entry point is fetched through
// the runtime, so the library has no link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

// 2-D row-major tensor [outer, inner] of `elem_bytes`-sized elements with rows
// `row_bytes` apart; box [box_outer, box_inner] with 128-byte swizzling
// (box_inner * elem_bytes must be 128).  Out-of-bounds elements read as zero.
// Returns false if the driver rejects the map (or the entry point is missing).
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

}  // namespace moe
