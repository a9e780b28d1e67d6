// common.cuh -- shared device-side definitions of the hypic CUDA library.
//
// Token inputs arrive packed as [L][N][H][d] (layer-major, token-major) in
// fp32 or bf16; states, pairs and outputs are fp32.  Kernels read their
// segment tables from kernel parameters (host offsets are validated and
// copied by the launch itself), so no call needs a host-to-device copy.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/hypic.h"

namespace hypic {

constexpr int kMaxSeg = HYPIC_MAX_SEGMENTS;
// Per-head L2 normalisation after the causal conv: x / sqrt(sum x^2 + eps).
constexpr float kL2Eps = 1e-6f;

struct Dims {
    int L, H, D, w, conv_k, mode, dtype, act;  // act: hypic_act after the conv
};

// SiLU, x sigma(x), applied after the causal conv when Dims::act says so.
__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

struct TokPtrs {
    const void *q, *k, *v, *alpha, *beta;
    const float *conv_w;  // [L][3][H][D][conv_k]
    int32_t N;
};

// Segment offsets plus a permutation of segment indices (build: longest body
// first; compose / seam: the request order).  Fits the kernel-parameter space.
struct SegTable {
    int32_t n_seg;
    int32_t n_perm;
    int32_t off[kMaxSeg + 1];
    int32_t perm[kMaxSeg];
};

template <typename T> __device__ __forceinline__ float ld_f(const T *p, size_t i);
template <> __device__ __forceinline__ float ld_f<float>(const float *p, size_t i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

// Index of token `tok` of layer l, head h, channel c in a [L][N][H][D] tensor.
__device__ __forceinline__ size_t tok_index(const Dims &dm, int32_t N, int l, int32_t tok, int h, int c) {
    return (((size_t)l * N + tok) * dm.H + h) * dm.D + c;
}
__device__ __forceinline__ size_t gate_index(const Dims &dm, int32_t N, int l, int32_t tok, int h) {
    return ((size_t)l * N + tok) * dm.H + h;
}

// Token index of the raw token `back` positions before stream position
// (entry e, offset j within its segment) in the request described by tab
// (perm = request order).  Returns -1 before the request start.
__device__ __forceinline__ int32_t stream_back(const SegTable &tab, int e, int j, int back) {
    int s = tab.perm[e];
    if (j - back >= 0) return tab.off[s] + j - back;
    int need = back - j;  // tokens needed before the start of entry e
    for (int ee = e - 1; ee >= 0; --ee) {
        int sp = tab.perm[ee];
        int len = tab.off[sp + 1] - tab.off[sp];
        if (need <= len) return tab.off[sp + 1] - need;
        need -= len;
    }
    return -1;
}

}  // namespace hypic
