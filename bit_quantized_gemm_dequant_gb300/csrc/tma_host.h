// Host helper: a 2-D tiled TMA tensor map over a row-major matrix.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace wq {

// inner/outer: matrix extent in elements (inner = contiguous dimension);
// row_stride_bytes: distance between rows (multiple of 16); box_*: tile
// extent in elements.  Out-of-range box elements read as zero.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                         uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle);

}  // namespace wq
