// tmap.cuh -- host-side TMA descriptor construction.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ssd {

// 4-D tensor map of 16-bit elements with 128-byte swizzle.  dims[0] is the contiguous
// dimension (elements); the row strides follow from the dense layout.
// Returns false if the driver entry point is unavailable or rejects the map.
// 16-bit elements (bfloat16 or float16; TMA copies the bits either way).
bool make_tmap_16b_4d(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint32_t box[4]);

}  // namespace ssd
