// tmap.h -- host-side TMA tensor-map encoding (see tmap.cu).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace hypic {

// Encode a tiled tensor map (unit element strides, no interleave, 256-byte
// L2 promotion, zero fill out of bounds).  dims/box have `rank` entries,
// strides rank-1 (bytes, dimensions 1..rank-1).
cudaError_t encode_tiled(CUtensorMap *map, CUtensorMapDataType type, cuuint32_t rank, const void *base,
                         const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                         CUtensorMapSwizzle swizzle);

}  // namespace hypic
