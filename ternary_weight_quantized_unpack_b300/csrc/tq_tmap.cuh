// Host-side creation of TMA tensor maps.  cuTensorMapEncodeTiled is a driver entry point; it is
// fetched through the runtime on first use, so libtq does not link libcuda and still loads on a
// machine without a GPU driver.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace tq {

// 2-D tiled map over a row-major [outer][inner] array with the given row stride (bytes, multiple of
// 16); box = [box_outer][box_inner] elements.  Out-of-range elements read as zero.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner, uint64_t outer,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

}  // namespace tq
