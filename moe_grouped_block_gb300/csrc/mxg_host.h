// mxg_host.h -- host-side helpers shared by the launchers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxg {

// 2-D tensor map over a row-major [rows, inner] matrix of `dtype` elements
// with `row_bytes` between rows; box [box_rows, box_inner]; the given
// swizzle.  Returns false if the driver entry point is missing or rejects
// the description.
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                  uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                  CUtensorMapSwizzle swizzle);

// 3-D tensor map without swizzle: dims[0] innermost (elements), byte strides
// of dims 1 and 2, box extents per dimension.
bool make_tmap_3d(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                  const uint64_t strides_bytes[2], const uint32_t box[3]);

}  // namespace mxg
