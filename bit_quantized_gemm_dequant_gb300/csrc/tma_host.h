// Host helper: a 2-D tiled TMA tensor map over a row-major matrix.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace wq {

// inner/outer: matrix extent in elements (inner = contiguous dimension);
// row_stride_bytes: distance between rows (multiple of 16); box_*: tile
// extent in elements.  Out-of-range box elements read as zero.  promotion:
// the L2 fetch size for the box's rows (256 bytes unless the caller knows
// that the bytes next to its 128-byte rows are read by nobody soon).
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                         uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle,
                         CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

}  // namespace wq
