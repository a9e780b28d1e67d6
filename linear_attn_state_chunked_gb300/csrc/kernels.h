// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels.  Not installed; the public interface is include/hypic.h.
#pragma once

#include "common.cuh"

namespace hypic {

struct BuildArgs {
    Dims dm;
    TokPtrs tok;
    float *T_out;                // may be null (segment forward without the transition product)
    float *S_out;                // may be null (segment forward)
    float *o_out;                // per-token body outputs (segment forward), else null
    int *status;                 // device status word (0 = ok)
};

struct ComposeArgs {
    Dims dm;
    TokPtrs tok;
    const float *T;
    const float *S;
    const float *S_init;  // may be null (zero)
    float *S_prefix;      // may be null
    float *S_final;
    float *o_out;         // may be null when w == 0
    int *status;          // device word a kernel's bounded wait ORs 1 into when it gives up
};

struct SeamArgs {
    Dims dm;
    TokPtrs tok;
    const float *S_in;
    float *o_out;
    float *S_out;  // may be null; may alias S_in
    int *status;   // device word a kernel's bounded wait ORs 1 into when it gives up
};

cudaError_t launch_build_rec(const BuildArgs &a, const SegTable &tab, cudaStream_t st);
bool build_tc_supported(const Dims &dm);
cudaError_t launch_build_tc(const BuildArgs &a, const SegTable &tab, cudaStream_t st);
cudaError_t launch_compose(const ComposeArgs &a, const SegTable &tab, cudaStream_t st);
bool compose_tc_supported(const Dims &dm);
cudaError_t launch_compose_tc(const ComposeArgs &a, const SegTable &tab, cudaStream_t st);
cudaError_t launch_seam(const SeamArgs &a, const SegTable &tab, cudaStream_t st);
cudaError_t launch_seam_chunk(const SeamArgs &a, const SegTable &tab, cudaStream_t st);

}  // namespace hypic
