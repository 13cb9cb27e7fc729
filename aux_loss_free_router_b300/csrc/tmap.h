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

// The same row-major 2-byte-element tensor [rows, mn] seen as [mn/64 chunks][rows][64]:
// one box of box_chunks x box_rows x 64 lands in shared memory as box_chunks 128-byte
// swizzled [box_rows][64] blocks one after another, the MN-major operand layout of an
// MMA, in one copy instead of box_chunks.  mn must be a multiple of 64; false if not,
// or if the driver rejects the map.
// 3-D tensor [d2][d1][d0] (strides in bytes for dims 1 and 2), box [1][box1][box0] with
// 128-byte swizzling (box0 * element size must be 128).
bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1);

bool make_tmap_mn3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t mn,
                    uint64_t rows, uint64_t row_bytes, uint32_t box_rows, uint32_t box_chunks);

}  // namespace moe
