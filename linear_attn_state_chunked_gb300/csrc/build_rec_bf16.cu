// build_rec_bf16.cu -- the bf16-input instantiations of the token-serial
// CUDA-core build (dispatched from build_rec.cu).
#include "build_rec.cuh"

namespace hypic {

cudaError_t launch_build_rec_bf16(const BuildArgs &a, const SegTable &tab, int n_items, cudaStream_t st)
{
    switch (a.dm.mode) {
    case HYPIC_GATED_DELTA: return launch_m<HYPIC_GATED_DELTA, __nv_bfloat16>(a, tab, n_items, st);
    case HYPIC_SCALAR_DECAY: return launch_m<HYPIC_SCALAR_DECAY, __nv_bfloat16>(a, tab, n_items, st);
    case HYPIC_KDA: return launch_m<HYPIC_KDA, __nv_bfloat16>(a, tab, n_items, st);
    default: return launch_m<HYPIC_DIAG_GATE, __nv_bfloat16>(a, tab, n_items, st);
    }
}

}  // namespace hypic
