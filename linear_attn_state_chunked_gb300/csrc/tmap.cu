// tmap.cu -- host-side TMA tensor-map encoding shared by the kernels.  The
// driver's encoder is fetched through the runtime (no link-time dependency
// on the driver library), once per process.
#include <mutex>

#include "tmap.h"

namespace hypic {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;
std::once_flag g_encode_once;
}  // namespace

cudaError_t encode_tiled(CUtensorMap *map, CUtensorMapDataType type, cuuint32_t rank, const void *base,
                         const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                         CUtensorMapSwizzle swizzle)
{
    std::call_once(g_encode_once, []() {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn))
            g_encode_err = cudaErrorNotSupported;
        if (g_encode_err == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode_err != cudaSuccess) return g_encode_err;
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    const CUresult r = g_encode(map, type, rank, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace hypic
