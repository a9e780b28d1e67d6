// build_rec.cu -- dispatch of the token-serial CUDA-core build, and its fp32-
// input instantiations (the bf16 ones are compiled in build_rec_bf16.cu, so
// that the two compile in parallel).
#include "build_rec.cuh"

namespace hypic {

cudaError_t launch_build_rec_bf16(const BuildArgs &a, const SegTable &tab, int n_items, cudaStream_t st);

cudaError_t launch_build_rec(const BuildArgs &a, const SegTable &tab, cudaStream_t st)
{
    const int n_items = tab.n_seg * a.dm.L * a.dm.H;
    if (n_items == 0) return cudaSuccess;
    if (a.dm.dtype == HYPIC_BF16) return launch_build_rec_bf16(a, tab, n_items, st);
    switch (a.dm.mode) {
    case HYPIC_GATED_DELTA: return launch_m<HYPIC_GATED_DELTA, float>(a, tab, n_items, st);
    case HYPIC_SCALAR_DECAY: return launch_m<HYPIC_SCALAR_DECAY, float>(a, tab, n_items, st);
    case HYPIC_KDA: return launch_m<HYPIC_KDA, float>(a, tab, n_items, st);
    default: return launch_m<HYPIC_DIAG_GATE, float>(a, tab, n_items, st);
    }
}

}  // namespace hypic
