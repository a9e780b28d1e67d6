// compose.cu -- running-state composition with fused seams, and the
// standalone seam advance, on CUDA cores.
//
// HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, sections "线性层" and "全注意力层";
// article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, linear-layer and seam-window paragraphs): at reuse the
// running state is advanced entry by entry as S <- T_C S + S(C|0), and each
// segment's seam tokens are first re-run under the running state, emitting
// their per-token outputs.
//
// Columns of S evolve independently under both operations (T_C S acts on
// each column alone; a recurrence step's u = S^T k is per column), so a CTA
// owns one (layer, head) chain and a block of CB columns for the whole
// request.  The seam keeps each thread's slice of a column in registers; the
// T_C S product stages T_C in shared memory and accumulates a 4 x RPT
// register tile per thread.
#include "common.cuh"
#include "kernels.h"

namespace hypic {

template <int D> struct CompGeom {
    static constexpr int CB = D >= 32 ? 32 : D;                     // columns per CTA
    static constexpr int NT = (D * CB / 4 < 256) ? D * CB / 4 : 256; // threads
    static constexpr int CG = CB / 4;   // product: column groups of 4
    static constexpr int RG = NT / CG;  // product: row groups
    static constexpr int RPT = D / RG;  // product: rows per thread
    static constexpr int TPC = NT / CB; // seam: threads per column
    static constexpr int RPS = D / TPC; // seam: rows per thread
    static_assert(RPT >= 1 && RPS >= 1 && (32 % TPC) == 0, "geometry");
};

// Token staging area: q, k, v, alpha rows plus beta and two reduction slots.
template <int D> struct TokStage {
    float q[D], k[D], v[D], a[D];
    float beta, red[2], pad;
};

// Stage seam token j of request entry e into shared memory (all threads).
// With a causal conv, tap `lag` reads the raw token lag positions earlier in
// the request stream (crossing into previous entries: the conv warm-up),
// and q, k are then L2-normalised over the head's D channels.
template <int D, int MODE, typename Tin, int CK, int NT>
__device__ __forceinline__ void stage_token(const Dims &dm, const TokPtrs &tk, const SegTable &tab,
                                            int l, int h, int e, int j, TokStage<D> &st)
{
    const int tid = threadIdx.x;
    const int32_t N = tk.N;
    const int32_t tok = tab.off[tab.perm[e]] + j;
    const Tin *qp = static_cast<const Tin *>(tk.q);
    const Tin *kp = static_cast<const Tin *>(tk.k);
    const Tin *vp = static_cast<const Tin *>(tk.v);
    const Tin *ap = static_cast<const Tin *>(tk.alpha);
    for (int ch = tid; ch < D; ch += NT) {
        if (CK == 0) {
            const size_t ix = tok_index(dm, N, l, tok, h, ch);
            st.q[ch] = ld_f(qp, ix);
            st.k[ch] = ld_f(kp, ix);
            st.v[ch] = ld_f(vp, ix);
        } else {
            float qv = 0.f, kv = 0.f, vv = 0.f;
            const float *wq = tk.conv_w + (((size_t)l * 3 + 0) * dm.H + h) * D * CK + ch * CK;
            const float *wk = wq + (size_t)dm.H * D * CK;
            const float *wv = wk + (size_t)dm.H * D * CK;
#pragma unroll
            for (int lag = 0; lag < CK; ++lag) {
                const int32_t tb = stream_back(tab, e, j, lag);
                if (tb >= 0) {
                    const size_t ix = tok_index(dm, N, l, tb, h, ch);
                    qv = fmaf(wq[lag], ld_f(qp, ix), qv);
                    kv = fmaf(wk[lag], ld_f(kp, ix), kv);
                    vv = fmaf(wv[lag], ld_f(vp, ix), vv);
                }
            }
            st.q[ch] = dm.act ? silu(qv) : qv;
            st.k[ch] = dm.act ? silu(kv) : kv;
            st.v[ch] = dm.act ? silu(vv) : vv;
        }
        if (MODE == HYPIC_DIAG_GATE || MODE == HYPIC_KDA) st.a[ch] = ld_f(ap, tok_index(dm, N, l, tok, h, ch));
    }
    if (tid == 0) {
        if (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA) {
            const size_t gi = gate_index(dm, N, l, tok, h);
            if (MODE == HYPIC_GATED_DELTA) st.a[0] = ld_f(ap, gi);
            st.beta = ld_f(static_cast<const Tin *>(tk.beta), gi);
        } else if (MODE == HYPIC_SCALAR_DECAY) {
            st.a[0] = ld_f(ap, (size_t)l * dm.H + h);
        }
    }
    if (CK > 0) {
        __syncthreads();
        if (tid < 32) {
            float sq = 0.f, sk = 0.f;
            for (int ch = tid; ch < D; ch += 32) {
                sq = fmaf(st.q[ch], st.q[ch], sq);
                sk = fmaf(st.k[ch], st.k[ch], sk);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (tid == 0) {
                st.red[0] = 1.f / sqrtf(sq + kL2Eps);
                st.red[1] = 1.f / sqrtf(sk + kL2Eps);
            }
        }
        __syncthreads();
        for (int ch = tid; ch < D; ch += NT) {
            st.q[ch] *= st.red[0];
            st.k[ch] *= st.red[1];
        }
    }
}

template <int TPC> __device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = TPC / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Re-run the seam of request entry e for this thread's column slice xs
// (rows part + TPC*i of column c0 + col), writing o_out rows 0..w-1.
template <int D, int MODE, typename Tin, int CK>
__device__ void run_seam(float (&xs)[CompGeom<D>::RPS], const Dims &dm, const TokPtrs &tk,
                         const SegTable &tab, int l, int h, int e, int c0, float *o_out,
                         TokStage<D> &st)
{
    using G = CompGeom<D>;
    const int tid = threadIdx.x;
    const int col = tid / G::TPC, part = tid % G::TPC;
    const int s = tab.perm[e];
    const int sw = min(dm.w, tab.off[s + 1] - tab.off[s]);
    for (int j = 0; j < dm.w; ++j) {
        float o = 0.f;
        if (j < sw) {
            __syncthreads();
            stage_token<D, MODE, Tin, CK, G::NT>(dm, tk, tab, l, h, e, j, st);
            __syncthreads();
            const float vc = st.v[c0 + col];
            if (MODE == HYPIC_GATED_DELTA) {
                const float al = st.a[0], be = st.beta;
                float u = 0.f;
#pragma unroll
                for (int i = 0; i < G::RPS; ++i) u = fmaf(st.k[part + G::TPC * i], xs[i], u);
                u = group_sum<G::TPC>(u);
                const float coef = be * (vc - al * u);
#pragma unroll
                for (int i = 0; i < G::RPS; ++i) xs[i] = fmaf(st.k[part + G::TPC * i], coef, al * xs[i]);
            } else if (MODE == HYPIC_KDA) {
                // decay the key channels, then erase along k and write
                const float be = st.beta;
                float u = 0.f;
#pragma unroll
                for (int i = 0; i < G::RPS; ++i) {
                    const int r = part + G::TPC * i;
                    xs[i] *= st.a[r];
                    u = fmaf(st.k[r], xs[i], u);
                }
                u = group_sum<G::TPC>(u);
                const float coef = be * (vc - u);
#pragma unroll
                for (int i = 0; i < G::RPS; ++i) xs[i] = fmaf(st.k[part + G::TPC * i], coef, xs[i]);
            } else {
#pragma unroll
                for (int i = 0; i < G::RPS; ++i) {
                    const int r = part + G::TPC * i;
                    const float ar = (MODE == HYPIC_SCALAR_DECAY) ? st.a[0] : st.a[r];
                    xs[i] = fmaf(st.k[r], vc, ar * xs[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < G::RPS; ++i) o = fmaf(st.q[part + G::TPC * i], xs[i], o);
            o = group_sum<G::TPC>(o);
        }
        if (part == 0)
            o_out[(((size_t)l * tab.n_perm + e) * dm.w + j) * dm.H * D + (size_t)h * D + c0 + col] = o;
    }
}

template <int D, int MODE>
constexpr size_t compose_smem_bytes()
{
    using G = CompGeom<D>;
    return sizeof(float) * ((size_t)D * G::CB + (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA ? (size_t)D * (D + 1) : 0)) +
           sizeof(TokStage<D>);
}

template <int D, int MODE, typename Tin, int CK>
__global__ void __launch_bounds__(CompGeom<D>::NT)
compose_kernel(const __grid_constant__ ComposeArgs a, const __grid_constant__ SegTable tab)
{
    using G = CompGeom<D>;
    extern __shared__ __align__(16) float smem[];
    float *Sb = smem;                    // [D][CB] running-state block
    float *Ts = Sb + D * G::CB;          // [D][D+1] T_C (gated delta, KDA)
    TokStage<D> &st = *reinterpret_cast<TokStage<D> *>(
        Ts + (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA ? D * (D + 1) : 0));

    const Dims dm = a.dm;
    const int tid = threadIdx.x;
    constexpr int nblk = D / G::CB;
    const int lh = blockIdx.x / nblk, cb = blockIdx.x % nblk;
    const int l = lh / dm.H, h = lh % dm.H;
    const int c0 = cb * G::CB;
    const size_t st_base = ((size_t)l * dm.H + h) * D * D;

    for (int e = tid; e < D * G::CB; e += G::NT) {
        const int r = e / G::CB, cc = e % G::CB;
        Sb[e] = a.S_init ? a.S_init[st_base + (size_t)r * D + c0 + cc] : 0.f;
    }
    __syncthreads();

    const int col = tid / G::TPC, part = tid % G::TPC;
    const int cg = tid % G::CG, rg = tid / G::CG;

    for (int ent = 0; ent < tab.n_perm; ++ent) {
        const int s = tab.perm[ent];
        if (a.S_prefix) {
            float *dst = a.S_prefix + (((size_t)l * tab.n_perm + ent) * dm.H + h) * D * D + c0;
            for (int e = tid; e < D * G::CB; e += G::NT)
                dst[(size_t)(e / G::CB) * D + e % G::CB] = Sb[e];
        }
        if (dm.w > 0) {
            float xs[G::RPS];
#pragma unroll
            for (int i = 0; i < G::RPS; ++i) xs[i] = Sb[(part + G::TPC * i) * G::CB + col];
            run_seam<D, MODE, Tin, CK>(xs, dm, a.tok, tab, l, h, ent, c0, a.o_out, st);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < G::RPS; ++i) Sb[(part + G::TPC * i) * G::CB + col] = xs[i];
        }
        const size_t pair = ((size_t)l * tab.n_seg + s) * dm.H + h;
        const float *Sc = a.S + pair * D * D + c0;
        if (MODE == HYPIC_GATED_DELTA || MODE == HYPIC_KDA) {
            const float *Tg = a.T + pair * D * D;
            for (int e = tid; e < D * D; e += G::NT) Ts[(e / D) * (D + 1) + e % D] = Tg[e];
            __syncthreads();
            float acc[G::RPT][4];
#pragma unroll
            for (int i = 0; i < G::RPT; ++i) {
                const float4 c4 = *reinterpret_cast<const float4 *>(Sc + (size_t)(rg * G::RPT + i) * D + cg * 4);
                acc[i][0] = c4.x; acc[i][1] = c4.y; acc[i][2] = c4.z; acc[i][3] = c4.w;
            }
#pragma unroll 4
            for (int j = 0; j < D; ++j) {
                const float4 b4 = *reinterpret_cast<const float4 *>(Sb + j * G::CB + cg * 4);
#pragma unroll
                for (int i = 0; i < G::RPT; ++i) {
                    const float t = Ts[(rg * G::RPT + i) * (D + 1) + j];
                    acc[i][0] = fmaf(t, b4.x, acc[i][0]);
                    acc[i][1] = fmaf(t, b4.y, acc[i][1]);
                    acc[i][2] = fmaf(t, b4.z, acc[i][2]);
                    acc[i][3] = fmaf(t, b4.w, acc[i][3]);
                }
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < G::RPT; ++i)
                *reinterpret_cast<float4 *>(Sb + (rg * G::RPT + i) * G::CB + cg * 4) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            __syncthreads();
        } else {
            __syncthreads();
            for (int e = tid; e < D * G::CB; e += G::NT) {
                const int r = e / G::CB, cc = e % G::CB;
                const float t = (MODE == HYPIC_SCALAR_DECAY) ? a.T[pair] : a.T[pair * D + r];
                Sb[e] = fmaf(t, Sb[e], Sc[(size_t)r * D + cc]);
            }
            __syncthreads();
        }
    }
    for (int e = tid; e < D * G::CB; e += G::NT) {
        const int r = e / G::CB, cc = e % G::CB;
        a.S_final[st_base + (size_t)r * D + c0 + cc] = Sb[e];
    }
}

template <int D, int MODE, typename Tin, int CK>
__global__ void __launch_bounds__(CompGeom<D>::NT)
seam_kernel(const __grid_constant__ SeamArgs a, const __grid_constant__ SegTable tab)
{
    using G = CompGeom<D>;
    __shared__ __align__(16) TokStage<D> st;
    const Dims dm = a.dm;
    const int tid = threadIdx.x;
    constexpr int nblk = D / G::CB;
    const int LHB = dm.L * dm.H * nblk;
    const int ent = blockIdx.x / LHB;
    const int rem = blockIdx.x % LHB;
    const int lh = rem / nblk, cb = rem % nblk;
    const int l = lh / dm.H, h = lh % dm.H;
    const int c0 = cb * G::CB;
    const int col = tid / G::TPC, part = tid % G::TPC;
    const size_t base = (((size_t)l * tab.n_perm + ent) * dm.H + h) * D * D + c0 + col;
    float xs[G::RPS];
#pragma unroll
    for (int i = 0; i < G::RPS; ++i) xs[i] = a.S_in[base + (size_t)(part + G::TPC * i) * D];
    run_seam<D, MODE, Tin, CK>(xs, dm, a.tok, tab, l, h, ent, c0, a.o_out, st);
    if (a.S_out) {
#pragma unroll
        for (int i = 0; i < G::RPS; ++i) a.S_out[base + (size_t)(part + G::TPC * i) * D] = xs[i];
    }
}

// ---------------------------------------------------------------------------
// launch plumbing

template <int D, int MODE, typename Tin, int CK>
static cudaError_t launch_compose_t(const ComposeArgs &a, const SegTable &tab, cudaStream_t st)
{
    using G = CompGeom<D>;
    const size_t smem = compose_smem_bytes<D, MODE>();
    auto kern = compose_kernel<D, MODE, Tin, CK>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int grid = a.dm.L * a.dm.H * (D / G::CB);
    kern<<<grid, G::NT, smem, st>>>(a, tab);
    return cudaGetLastError();
}

template <int D, int MODE, typename Tin, int CK>
static cudaError_t launch_seam_t(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    using G = CompGeom<D>;
    const long long grid = (long long)tab.n_perm * a.dm.L * a.dm.H * (D / G::CB);
    if (grid == 0) return cudaSuccess;
    seam_kernel<D, MODE, Tin, CK><<<(unsigned)grid, G::NT, 0, st>>>(a, tab);
    return cudaGetLastError();
}


#define HYPIC_DISPATCH(FN, ARGS)                                                              \
    template <int D, int MODE, typename Tin>                                                  \
    static cudaError_t FN##_ck(const ARGS &a, const SegTable &tab, cudaStream_t st)            \
    {                                                                                         \
        switch (a.dm.conv_k) {                                                                \
        case 0: return FN##_t<D, MODE, Tin, 0>(a, tab, st);                                    \
        case 2: return FN##_t<D, MODE, Tin, 2>(a, tab, st);                                    \
        case 3: return FN##_t<D, MODE, Tin, 3>(a, tab, st);                                    \
        default: return FN##_t<D, MODE, Tin, 4>(a, tab, st);                                   \
        }                                                                                     \
    }                                                                                         \
    template <int MODE, typename Tin>                                                         \
    static cudaError_t FN##_d(const ARGS &a, const SegTable &tab, cudaStream_t st)             \
    {                                                                                         \
        switch (a.dm.D) {                                                                     \
        case 16: return FN##_ck<16, MODE, Tin>(a, tab, st);                                    \
        case 32: return FN##_ck<32, MODE, Tin>(a, tab, st);                                    \
        case 64: return FN##_ck<64, MODE, Tin>(a, tab, st);                                    \
        default: return FN##_ck<128, MODE, Tin>(a, tab, st);                                   \
        }                                                                                     \
    }                                                                                         \
    template <typename Tin>                                                                   \
    static cudaError_t FN##_m(const ARGS &a, const SegTable &tab, cudaStream_t st)             \
    {                                                                                         \
        switch (a.dm.mode) {                                                                  \
        case HYPIC_GATED_DELTA: return FN##_d<HYPIC_GATED_DELTA, Tin>(a, tab, st);             \
        case HYPIC_SCALAR_DECAY: return FN##_d<HYPIC_SCALAR_DECAY, Tin>(a, tab, st);           \
        case HYPIC_KDA: return FN##_d<HYPIC_KDA, Tin>(a, tab, st);                             \
        default: return FN##_d<HYPIC_DIAG_GATE, Tin>(a, tab, st);                              \
        }                                                                                     \
    }

HYPIC_DISPATCH(launch_compose, ComposeArgs)
HYPIC_DISPATCH(launch_seam, SeamArgs)
#undef HYPIC_DISPATCH

cudaError_t launch_compose(const ComposeArgs &a, const SegTable &tab, cudaStream_t st)
{
    // Gated delta at d = 128 with bf16 inputs composes on the tensor cores
    // (tf32 T_C S, 2e-3 class); fp32-input requests (1e-5 class) and the other
    // modes and widths use the CUDA-core kernel below.
    // (its TMA row coordinate, pair x 128, must fit 31 bits)
    const long long pair_rows = (long long)a.dm.L * (tab.n_seg > 0 ? tab.n_seg : 1) * a.dm.H * a.dm.D;
    if (compose_tc_supported(a.dm) && pair_rows < (1LL << 31)) return launch_compose_tc(a, tab, st);
    return a.dm.dtype == HYPIC_BF16 ? launch_compose_m<__nv_bfloat16>(a, tab, st)
                                    : launch_compose_m<float>(a, tab, st);
}

cudaError_t launch_seam(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    // Gated delta seams (DeltaNet included) run all their tokens in one pass
    // over the prefix state; the other modes re-run them token by token.
    if (a.dm.mode == HYPIC_GATED_DELTA) return launch_seam_chunk(a, tab, st);
    return a.dm.dtype == HYPIC_BF16 ? launch_seam_m<__nv_bfloat16>(a, tab, st)
                                    : launch_seam_m<float>(a, tab, st);
}

}  // namespace hypic
