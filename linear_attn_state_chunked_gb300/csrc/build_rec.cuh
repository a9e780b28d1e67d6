#pragma once
// build_rec.cuh -- segment build by the token-serial recurrence on CUDA cores
// (kernel and launch templates; instantiated per input dtype by build_rec.cu
// and build_rec_bf16.cu).
//
// Serves every mode, width and dtype; it is the exact-order fp32 path that
// the fp32-input workloads (1e-5 tolerance) use.  One CTA per work item
// (segment body, layer, head); items are launched longest body first, which
// the block scheduler dispatches in order -- the greedy longest-processing-
// time-first assignment of the HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, section
// "段并行"; article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, segment-parallelism paragraph).
//
// Gated delta keeps X = [T | S] (d_k x (d_k + d_v)) with one thread per
// column: for each token, u_c = sum_r k_r X_rc and
//     X_rc <- alpha (X_rc - beta k_r u_c) + beta k_r vbar_c ,
// where vbar is 0 on the T columns and v on the S columns -- the transition
// A_t = alpha (I - beta k k^T) applied on the left, plus the write
// beta k v^T on the S half (the pair (T_C, S(C|0)) of that article's "线性层").
// The two specialisations keep only S and form T as the product of gates.
//
// It also serves the segment forward: with an output buffer, each S-column
// thread emits o_t = S_t^T q_t for every body token (its column of S_t dotted
// with q_t, the segment's own zero-initial state); without a T buffer the
// gated delta and KDA CTAs carry the S columns only (TC = false), half the
// threads and registers, so that twice as many CTAs share an SM.
#include "common.cuh"
#include "kernels.h"

namespace hypic {

constexpr int kChunk = 16;

// Columns of the kept state and threads per CTA (at least one full warp;
// threads past the last column only help staging).
template <int D, int MODE, bool TC = true> struct RecGeom {
    static constexpr int NCOL = ((MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA) && TC ? 2 : 1) * D;
    static constexpr int NT = NCOL < 32 ? 32 : NCOL;
};

template <int D, int MODE, typename Tin, int CK, bool TC>
__global__ void __launch_bounds__(RecGeom<D, MODE, TC>::NT)
build_rec_kernel(const __grid_constant__ BuildArgs a, const __grid_constant__ SegTable tab)
{
    constexpr int NT = RecGeom<D, MODE, TC>::NT;
    constexpr int NCOL = RecGeom<D, MODE, TC>::NCOL;
    constexpr int AW = (MODE == HYPIC_DIAG_GATE || MODE == HYPIC_KDA) ? D : 1;
    constexpr bool DENSE_T = (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA);
    constexpr bool TCOLS = DENSE_T && TC;  // this CTA carries T columns 0 .. D-1
    __shared__ __align__(16) float ks[kChunk][D];
    __shared__ __align__(16) float vs[kChunk][D];
    __shared__ __align__(16) float qs[kChunk][D];  // forward outputs only
    __shared__ float as_[kChunk][AW];
    __shared__ float bs[kChunk];

    const Dims dm = a.dm;
    const int32_t N = a.tok.N;
    const int LH = dm.L * dm.H;
    const int item = blockIdx.x;
    const int s = tab.perm[item / LH];
    const int lh = item % LH;
    const int l = lh / dm.H, h = lh % dm.H;
    const int32_t seg0 = tab.off[s], seg1 = tab.off[s + 1];
    const int32_t b0 = seg0 + min(dm.w, seg1 - seg0);
    const int32_t n = seg1 - b0;
    const int c = threadIdx.x;

    const bool want_o = a.o_out != nullptr, want_t = a.T_out != nullptr, want_s = a.S_out != nullptr;
    // S columns emit the outputs (column sc of S); T columns exist only with TC
    const bool s_col = !TCOLS || c >= D;
    const int sc = TCOLS ? c - D : c;
    const bool active = c < NCOL;
    const Tin *qp = static_cast<const Tin *>(a.tok.q);
    const Tin *kp = static_cast<const Tin *>(a.tok.k);
    const Tin *vp = static_cast<const Tin *>(a.tok.v);
    const Tin *ap = static_cast<const Tin *>(a.tok.alpha);
    const Tin *bp = static_cast<const Tin *>(a.tok.beta);

    float x[D];
#pragma unroll
    for (int r = 0; r < D; ++r) x[r] = (TCOLS && r == c) ? 1.f : 0.f;

    float gamma = 1.f;
    if (MODE == HYPIC_SCALAR_DECAY) gamma = ld_f(ap, (size_t)l * dm.H + h);
    float tprod = 1.f;

    // conv taps of this head for the k and v channels: w[(l*3 + m)*H + h][ch][j]
    const float *wq = nullptr, *wk = nullptr, *wv = nullptr;
    if (CK > 0) {
        wq = a.tok.conv_w + (((size_t)l * 3 + 0) * dm.H + h) * D * CK;
        wk = a.tok.conv_w + (((size_t)l * 3 + 1) * dm.H + h) * D * CK;
        wv = a.tok.conv_w + (((size_t)l * 3 + 2) * dm.H + h) * D * CK;
    }

    for (int32_t t0 = 0; t0 < n; t0 += kChunk) {
        const int nc = min(kChunk, (int)(n - t0));
        __syncthreads();
        for (int e = c; e < nc * D; e += NT) {
            const int i = e / D, ch = e % D;
            const int32_t tok = b0 + t0 + i;
            if (CK == 0) {
                ks[i][ch] = ld_f(kp, tok_index(dm, N, l, tok, h, ch));
                vs[i][ch] = ld_f(vp, tok_index(dm, N, l, tok, h, ch));
                if (want_o) qs[i][ch] = ld_f(qp, tok_index(dm, N, l, tok, h, ch));
            } else {
                float qv = 0.f, kv = 0.f, vv = 0.f;
#pragma unroll
                for (int j = 0; j < CK; ++j) {
                    const int32_t tj = tok - j;
                    if (tj >= seg0) {
                        kv = fmaf(wk[ch * CK + j], ld_f(kp, tok_index(dm, N, l, tj, h, ch)), kv);
                        vv = fmaf(wv[ch * CK + j], ld_f(vp, tok_index(dm, N, l, tj, h, ch)), vv);
                        if (want_o) qv = fmaf(wq[ch * CK + j], ld_f(qp, tok_index(dm, N, l, tj, h, ch)), qv);
                    }
                }
                ks[i][ch] = dm.act ? silu(kv) : kv;
                vs[i][ch] = dm.act ? silu(vv) : vv;
                if (want_o) qs[i][ch] = dm.act ? silu(qv) : qv;
            }
            if (MODE == HYPIC_DIAG_GATE || MODE == HYPIC_KDA) as_[i][ch] = ld_f(ap, tok_index(dm, N, l, tok, h, ch));
        }
        if (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA) {
            for (int i = c; i < nc; i += NT) {
                const size_t gi = gate_index(dm, N, l, b0 + t0 + i, h);
                if (MODE == HYPIC_GATED_DELTA) as_[i][0] = ld_f(ap, gi);
                bs[i] = ld_f(bp, gi);
            }
        }
        __syncthreads();
        if (CK > 0) {
            // L2-normalise each convolved k row (and q row) over its D channels.
            const int warp = c / 32, lane = c % 32;
            for (int row = warp; row < (want_o ? 2 : 1) * nc; row += NT / 32) {
                float *xr = row < nc ? ks[row] : qs[row - nc];
                float ss = 0.f;
                for (int ch = lane; ch < D; ch += 32) ss = fmaf(xr[ch], xr[ch], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float inv = 1.f / sqrtf(ss + kL2Eps);
                for (int ch = lane; ch < D; ch += 32) xr[ch] *= inv;
            }
            __syncthreads();
        }
        for (int i = 0; i < nc && active; ++i) {
            if (MODE == HYPIC_GATED_DELTA) {
                const float al = as_[i][0], be = bs[i];
                float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&ks[i][r]);
                    u0 = fmaf(k4.x, x[r + 0], u0);
                    u1 = fmaf(k4.y, x[r + 1], u1);
                    u2 = fmaf(k4.z, x[r + 2], u2);
                    u3 = fmaf(k4.w, x[r + 3], u3);
                }
                const float u = (u0 + u1) + (u2 + u3);
                const float vt = s_col ? vs[i][sc] : 0.f;
                const float coef = be * (vt - al * u);
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&ks[i][r]);
                    x[r + 0] = fmaf(k4.x, coef, al * x[r + 0]);
                    x[r + 1] = fmaf(k4.y, coef, al * x[r + 1]);
                    x[r + 2] = fmaf(k4.z, coef, al * x[r + 2]);
                    x[r + 3] = fmaf(k4.w, coef, al * x[r + 3]);
                }
            } else if (MODE == HYPIC_KDA) {
                // decay the key channels, then erase along k and write:
                // y = diag(alpha) x,  x = y + k beta (v - k.y)
                const float be = bs[i];
                float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&ks[i][r]);
                    const float4 a4 = *reinterpret_cast<const float4 *>(&as_[i][r]);
                    x[r + 0] *= a4.x;
                    x[r + 1] *= a4.y;
                    x[r + 2] *= a4.z;
                    x[r + 3] *= a4.w;
                    u0 = fmaf(k4.x, x[r + 0], u0);
                    u1 = fmaf(k4.y, x[r + 1], u1);
                    u2 = fmaf(k4.z, x[r + 2], u2);
                    u3 = fmaf(k4.w, x[r + 3], u3);
                }
                const float u = (u0 + u1) + (u2 + u3);
                const float vt = s_col ? vs[i][sc] : 0.f;
                const float coef = be * (vt - u);
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&ks[i][r]);
                    x[r + 0] = fmaf(k4.x, coef, x[r + 0]);
                    x[r + 1] = fmaf(k4.y, coef, x[r + 1]);
                    x[r + 2] = fmaf(k4.z, coef, x[r + 2]);
                    x[r + 3] = fmaf(k4.w, coef, x[r + 3]);
                }
            } else {
                const float vc = vs[i][c];
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&ks[i][r]);
                    if (MODE == HYPIC_SCALAR_DECAY) {
                        x[r + 0] = fmaf(k4.x, vc, gamma * x[r + 0]);
                        x[r + 1] = fmaf(k4.y, vc, gamma * x[r + 1]);
                        x[r + 2] = fmaf(k4.z, vc, gamma * x[r + 2]);
                        x[r + 3] = fmaf(k4.w, vc, gamma * x[r + 3]);
                    } else {
                        x[r + 0] = fmaf(k4.x, vc, as_[i][r + 0] * x[r + 0]);
                        x[r + 1] = fmaf(k4.y, vc, as_[i][r + 1] * x[r + 1]);
                        x[r + 2] = fmaf(k4.z, vc, as_[i][r + 2] * x[r + 2]);
                        x[r + 3] = fmaf(k4.w, vc, as_[i][r + 3] * x[r + 3]);
                    }
                }
                if (MODE == HYPIC_DIAG_GATE) tprod *= as_[i][c];
            }
            if (want_o && s_col) {
                // o_t[c_s] = sum_r q_t[r] S_t[r][c_s]
                float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
                for (int r = 0; r < D; r += 4) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&qs[i][r]);
                    o0 = fmaf(q4.x, x[r + 0], o0);
                    o1 = fmaf(q4.y, x[r + 1], o1);
                    o2 = fmaf(q4.z, x[r + 2], o2);
                    o3 = fmaf(q4.w, x[r + 3], o3);
                }
                a.o_out[tok_index(dm, N, l, b0 + t0 + i, h, sc)] = (o0 + o1) + (o2 + o3);
            }
        }
    }

    const size_t pair = ((size_t)l * tab.n_seg + s) * dm.H + h;
    if (c >= NCOL) return;
    if (DENSE_T) {
        if (s_col ? !want_s : !want_t) return;
        float *dst = s_col ? a.S_out + pair * D * D + sc : a.T_out + pair * D * D + c;
#pragma unroll
        for (int r = 0; r < D; ++r) dst[(size_t)r * D] = x[r];
    } else {
        if (want_s) {
            float *dst = a.S_out + pair * D * D + c;
#pragma unroll
            for (int r = 0; r < D; ++r) dst[(size_t)r * D] = x[r];
        }
        if (MODE == HYPIC_DIAG_GATE && want_t) a.T_out[pair * D + c] = tprod;
        if (MODE == HYPIC_SCALAR_DECAY && c == 0 && want_t) {
            for (int32_t t = 0; t < n; ++t) tprod *= gamma;
            a.T_out[pair] = tprod;
        }
    }
}

template <int D, int MODE, typename Tin, bool TC>
static cudaError_t launch_tc(const BuildArgs &a, const SegTable &tab, int n_items, cudaStream_t st)
{
    constexpr int NT = RecGeom<D, MODE, TC>::NT;
    if (a.dm.conv_k == 0)
        build_rec_kernel<D, MODE, Tin, 0, TC><<<n_items, NT, 0, st>>>(a, tab);
    else if (a.dm.conv_k == 2)
        build_rec_kernel<D, MODE, Tin, 2, TC><<<n_items, NT, 0, st>>>(a, tab);
    else if (a.dm.conv_k == 3)
        build_rec_kernel<D, MODE, Tin, 3, TC><<<n_items, NT, 0, st>>>(a, tab);
    else
        build_rec_kernel<D, MODE, Tin, 4, TC><<<n_items, NT, 0, st>>>(a, tab);
    return cudaGetLastError();
}

template <int D, int MODE, typename Tin>
static cudaError_t launch_d(const BuildArgs &a, const SegTable &tab, int n_items, cudaStream_t st)
{
    // gated delta and KDA without T: the S columns only
    if constexpr (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA)
        if (a.T_out == nullptr) return launch_tc<D, MODE, Tin, false>(a, tab, n_items, st);
    return launch_tc<D, MODE, Tin, true>(a, tab, n_items, st);
}

template <int MODE, typename Tin>
static cudaError_t launch_m(const BuildArgs &a, const SegTable &tab, int n_items, cudaStream_t st)
{
    switch (a.dm.D) {
    case 16: return launch_d<16, MODE, Tin>(a, tab, n_items, st);
    case 32: return launch_d<32, MODE, Tin>(a, tab, n_items, st);
    case 64: return launch_d<64, MODE, Tin>(a, tab, n_items, st);
    default: return launch_d<128, MODE, Tin>(a, tab, n_items, st);
    }
}

}  // namespace hypic
