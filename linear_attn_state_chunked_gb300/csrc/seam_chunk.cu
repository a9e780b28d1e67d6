// seam_chunk.cu -- standalone seam advance for the gated delta rule: every
// seam of a request re-run in parallel from its prefix state, all tokens of
// a seam in one pass over that state.
//
// HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, section "线性层";
// article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, linear-layer and seam-window paragraphs): a segment's
// first w tokens are re-run under the state left by the segments before it,
// emitting their per-token outputs and advancing that state.
//
// Algebra.  With prefix state S0 (rows: key channels, columns: value
// channels), one gated delta step is S_t = a_t S_{t-1} + k_t d_t^T with
// d_t = b_t (v_t - a_t S_{t-1}^T k_t).  Unrolling over a pass of n <= 8
// tokens with G_t = a_0 ... a_t and g(t, i) = a_{i+1} ... a_t (g(t, t) = 1):
//   d_t = b_t (v_t - G_t S0^T k_t) - sum_{i<t} b_t g(t, i) (k_t . k_i) d_i
//   o_t = S_t^T q_t = G_t S0^T q_t + sum_{i<=t} g(t, i) (q_t . k_i) d_i
//   S_n = G_{n-1} S0 + sum_i g(n-1, i) k_i d_i^T
// so S0 is read once, for the 2n column products S0^T k_t and S0^T q_t, and
// the rest is n x n algebra per column.  The decay ratios are products of
// gates, never quotients, so a gate of 0 stays exact.  Seams longer than 8
// tokens take several passes, the state carried in registers between them.
//
// Two forms, both fp32 on CUDA cores (2 x 8 x d^2 multiply-adds per pass):
// d = 128 with seams of at most 8 tokens runs the persistent pipelined form
// at the end of this file; the other widths and longer seams run one CTA per
// (layer, request entry, head) seam with 2 d threads: thread (cp, rq) holds
// columns 2cp, 2cp + 1 of rows [rq d/4, (rq + 1) d/4) of S0 in registers
// (loaded first, so that the state read overlaps the token staging),
// accumulates the 16 partial column products for those rows with [k; q]
// broadcast from shared memory, the four row quarters are summed through
// shared memory, and thread c < d solves its column's triangular system and
// writes the outputs.
#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace hypic {

namespace {

constexpr int WC = 8;       // seam tokens per pass
constexpr int MR = 2 * WC;  // rows of [k_0..k_7; q_0..q_7]

template <int D> struct ChunkGeom {
    static constexpr int NT = 2 * D;      // threads
    static constexpr int NW = NT / 32;    // warps
    static constexpr int CP = D / 2;      // column pairs
    static constexpr int RQ = NT / CP;    // row quarters (4)
    static constexpr int RPT = D / RQ;    // state rows per thread
    static constexpr int WS = MR + 4;     // [k; q]^T row stride: 16-byte rows, conflict-free 16-byte stores
    static constexpr int HW = D >= 32 ? D / 32 : 1;  // warps per token half (staging)
    static constexpr int RL = D >= 32 ? 32 : D;      // lanes of one token half within a warp
    static_assert(RQ == 4 && RPT * RQ == D && NW >= 1, "geometry");
};

template <int D> struct ChunkSmem {
    float wt[D][ChunkGeom<D>::WS];  // [channel][k_0..k_7, q_0..q_7, pad]
    float kq[MR][D];                // k_0..k_7, q_0..q_7 token-major (dot products)
    float v[WC][D];
    float red[4][MR][D];            // partial column products per row quarter
    float dl[WC][D];                // g(n-1, t) d_t, for the state update
    float nrm[2][ChunkGeom<D>::HW][2 * 4];
    float dots[2][WC][WC];          // k_t . k_i and q_t . k_i
    float ck[WC][WC], cq[WC][WC];   // b_t g(t, i) k_t . k_i (i < t); g(t, i) q_t . k_i (i <= t)
    float alpha[WC], beta[WC], gam[WC], glast[WC];
    int32_t tok0, sw, prev[4];
};

// Stage seam tokens [b WC, b WC + WC) of the CTA's seam: causal conv (if
// any), L2 normalisation after the conv, transposed and token-major copies
// of k and q, v, and the gates (tokens past the seam end: zero k, q, v,
// gate 1, beta 0, so that they drop out of every sum).
template <int D, typename Tin, int CK>
__device__ __forceinline__ void stage_pass(ChunkSmem<D> &sm, const Dims &dm, const TokPtrs &tk, int l, int h,
                                           int b)
{
    using G = ChunkGeom<D>;
    const int tid = threadIdx.x;
    const int ch = tid % D, th = tid / D;
    const int sw = sm.sw, tok0 = sm.tok0;
    const int jb = b * WC + th * 4;
    const Tin *qp = static_cast<const Tin *>(tk.q);
    const Tin *kp = static_cast<const Tin *>(tk.k);
    const Tin *vp = static_cast<const Tin *>(tk.v);
    float qq[4], kk[4], vv[4];
    if constexpr (CK == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = jb + u;
            qq[u] = kk[u] = vv[u] = 0.f;
            if (j < sw) {
                const size_t ix = tok_index(dm, tk.N, l, tok0 + j, h, ch);
                qq[u] = ld_f(qp, ix);
                kk[u] = ld_f(kp, ix);
                vv[u] = ld_f(vp, ix);
            }
        }
    } else {
        constexpr int NWIN = CK - 1 + 4;
        float wq[CK], wk[CK], wv[CK];
        {
            const float *w0 = tk.conv_w + (((size_t)l * 3) * dm.H + h) * D * CK + (size_t)ch * CK;
            const size_t step = (size_t)dm.H * D * CK;
#pragma unroll
            for (int g = 0; g < CK; ++g) {
                wq[g] = __ldg(w0 + g);
                wk[g] = __ldg(w0 + step + g);
                wv[g] = __ldg(w0 + 2 * step + g);
            }
        }
        float rq[NWIN], rk[NWIN], rv[NWIN];
#pragma unroll
        for (int x = 0; x < NWIN; ++x) {
            const int p = jb - (CK - 1) + x;  // seam position of this raw token
            const int32_t t = p >= 0 ? (p < sw ? tok0 + p : -1) : sm.prev[-p];
            rq[x] = rk[x] = rv[x] = 0.f;
            if (t >= 0) {
                const size_t ix = tok_index(dm, tk.N, l, t, h, ch);
                rq[x] = ld_f(qp, ix);
                rk[x] = ld_f(kp, ix);
                rv[x] = ld_f(vp, ix);
            }
        }
        float ss[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float a = 0.f, c = 0.f, e = 0.f;
#pragma unroll
            for (int lag = 0; lag < CK; ++lag) {
                a = fmaf(wq[lag], rq[u + CK - 1 - lag], a);
                c = fmaf(wk[lag], rk[u + CK - 1 - lag], c);
                e = fmaf(wv[lag], rv[u + CK - 1 - lag], e);
            }
            if (dm.act) {
                a = silu(a);
                c = silu(c);
                e = silu(e);
            }
            const bool live = jb + u < sw;
            qq[u] = live ? a : 0.f;
            kk[u] = live ? c : 0.f;
            vv[u] = live ? e : 0.f;
            ss[u] = qq[u] * qq[u];
            ss[4 + u] = kk[u] * kk[u];
        }
#pragma unroll
        for (int o = G::RL / 2; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 8; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
        if (ch % 32 == 0) {
#pragma unroll
            for (int u = 0; u < 8; ++u) sm.nrm[th][ch / 32][u] = ss[u];
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int w = 0; w < G::HW; ++w) {
                sq += sm.nrm[th][w][u];
                sk += sm.nrm[th][w][4 + u];
            }
            qq[u] *= 1.f / sqrtf(sq + kL2Eps);
            kk[u] *= 1.f / sqrtf(sk + kL2Eps);
        }
    }
    *reinterpret_cast<float4 *>(&sm.wt[ch][th * 4]) = make_float4(kk[0], kk[1], kk[2], kk[3]);
    *reinterpret_cast<float4 *>(&sm.wt[ch][WC + th * 4]) = make_float4(qq[0], qq[1], qq[2], qq[3]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        sm.kq[th * 4 + u][ch] = kk[u];
        sm.kq[WC + th * 4 + u][ch] = qq[u];
        sm.v[th * 4 + u][ch] = vv[u];
    }
    if (tid < 2 * WC) {
        const int u = tid % WC, j = b * WC + u;
        const bool live = j < sw;
        const size_t gi = live ? gate_index(dm, tk.N, l, tok0 + j, h) : 0;
        if (tid < WC) sm.alpha[u] = live ? ld_f(static_cast<const Tin *>(tk.alpha), gi) : 1.f;
        else sm.beta[u] = live ? ld_f(static_cast<const Tin *>(tk.beta), gi) : 0.f;
    }
}

template <int D, typename Tin, int CK>
__global__ void __launch_bounds__(ChunkGeom<D>::NT, 2)
seam_chunk_kernel(const __grid_constant__ SeamArgs a, const __grid_constant__ SegTable tab)
{
    using G = ChunkGeom<D>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ChunkSmem<D> &sm = *reinterpret_cast<ChunkSmem<D> *>(smem_raw);
    const Dims dm = a.dm;
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int h = blockIdx.x % dm.H;
    const int le = blockIdx.x / dm.H;
    const int ent = le % tab.n_perm, l = le / tab.n_perm;

    // Segment lookups (kernel-parameter table) first, off the critical path
    // of the state read below.
    if (tid == 0) {
        const int s = tab.perm[ent];
        const int32_t t0 = tab.off[s];
        sm.tok0 = t0;
        sm.sw = min(dm.w, tab.off[s + 1] - t0);
    } else if (tid < 4) {
        sm.prev[tid] = tid < CK ? stream_back(tab, ent, 0, tid) : -1;
    }

    // The prefix state: columns 2cp, 2cp + 1 of this thread's row quarter.
    const int cp = tid % G::CP, rq = tid / G::CP;
    const size_t sbase = (((size_t)l * tab.n_perm + ent) * dm.H + h) * D * D;
    float2 xs[G::RPT];
#pragma unroll
    for (int i = 0; i < G::RPT; ++i)
        xs[i] = __ldg(reinterpret_cast<const float2 *>(a.S_in + sbase + (size_t)(rq * G::RPT + i) * D) + cp);

    __syncthreads();

    const int sw = sm.sw;
    const int n_pass = (dm.w + WC - 1) / WC;
    float *o_base = a.o_out + ((size_t)l * tab.n_perm + ent) * dm.w * dm.H * D + (size_t)h * D;
    const size_t o_row = (size_t)dm.H * D;

    for (int b = 0; b < n_pass; ++b) {
        const bool more = b + 1 < n_pass && (b + 1) * WC < sw;
        const bool need_state = more || a.S_out != nullptr;
        if (b * WC >= sw) {
            // nothing left of the seam: zero outputs for the remaining rows
            for (int e = tid; e < WC * D; e += G::NT) {
                const int j = b * WC + e / D;
                if (j < dm.w) o_base[(size_t)j * o_row + e % D] = 0.f;
            }
            continue;
        }
        if (b > 0) __syncthreads();  // previous pass done with the staging area
        stage_pass<D, Tin, CK>(sm, dm, a.tok, l, h, b);
        __syncthreads();

        // dot products k_t . k_i and q_t . k_i (2 x 64 of them)
        for (int d = warp; d < 2 * WC * WC; d += G::NW) {
            const int which = d / (WC * WC), t = (d / WC) % WC, i = d % WC;
            const float *x = sm.kq[which * WC + t];
            const float *y = sm.kq[i];
            float s = 0.f;
            for (int c = lane; c < D; c += 32) s = fmaf(x[c], y[c], s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) sm.dots[which][t][i] = s;
        }

        // partial column products [k; q] S0 over this thread's rows
        float acc[MR][2];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = 0.f;
#pragma unroll
        for (int i = 0; i < G::RPT; ++i) {
            const float4 *wr = reinterpret_cast<const float4 *>(sm.wt[rq * G::RPT + i]);
#pragma unroll
            for (int m4 = 0; m4 < MR / 4; ++m4) {
                const float4 w4 = wr[m4];
                acc[4 * m4 + 0][0] = fmaf(w4.x, xs[i].x, acc[4 * m4 + 0][0]);
                acc[4 * m4 + 0][1] = fmaf(w4.x, xs[i].y, acc[4 * m4 + 0][1]);
                acc[4 * m4 + 1][0] = fmaf(w4.y, xs[i].x, acc[4 * m4 + 1][0]);
                acc[4 * m4 + 1][1] = fmaf(w4.y, xs[i].y, acc[4 * m4 + 1][1]);
                acc[4 * m4 + 2][0] = fmaf(w4.z, xs[i].x, acc[4 * m4 + 2][0]);
                acc[4 * m4 + 2][1] = fmaf(w4.z, xs[i].y, acc[4 * m4 + 2][1]);
                acc[4 * m4 + 3][0] = fmaf(w4.w, xs[i].x, acc[4 * m4 + 3][0]);
                acc[4 * m4 + 3][1] = fmaf(w4.w, xs[i].y, acc[4 * m4 + 3][1]);
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m)
            *reinterpret_cast<float2 *>(&sm.red[rq][m][2 * cp]) = make_float2(acc[m][0], acc[m][1]);
        __syncthreads();

        // decay products and the coefficients of the triangular system
        for (int e = tid; e < WC * WC; e += G::NT) {
            const int t = e / WC, i = e % WC;
            float g = 1.f;
            for (int j = i + 1; j <= t; ++j) g *= sm.alpha[j];
            sm.ck[t][i] = i < t ? sm.beta[t] * g * sm.dots[0][t][i] : 0.f;
            sm.cq[t][i] = i <= t ? g * sm.dots[1][t][i] : 0.f;
            if (i == 0) {
                float gt = 1.f, gl = 1.f;
                for (int j = 0; j <= t; ++j) gt *= sm.alpha[j];
                for (int j = t + 1; j < WC; ++j) gl *= sm.alpha[j];
                sm.gam[t] = gt;
                sm.glast[t] = gl;
            }
        }
        __syncthreads();

        // per column: solve for d_t, emit o_t
        if (tid < D) {
            const int c = tid;
            float pk[WC], pq[WC];
#pragma unroll
            for (int t = 0; t < WC; ++t) {
                pk[t] = sm.red[0][t][c] + sm.red[1][t][c] + sm.red[2][t][c] + sm.red[3][t][c];
                pq[t] = sm.red[0][WC + t][c] + sm.red[1][WC + t][c] + sm.red[2][WC + t][c] +
                        sm.red[3][WC + t][c];
            }
            float dt[WC];
#pragma unroll
            for (int t = 0; t < WC; ++t) {
                float r = sm.beta[t] * (sm.v[t][c] - sm.gam[t] * pk[t]);
#pragma unroll
                for (int i = 0; i < t; ++i) r = fmaf(-sm.ck[t][i], dt[i], r);
                dt[t] = r;
                float o = sm.gam[t] * pq[t];
#pragma unroll
                for (int i = 0; i <= t; ++i) o = fmaf(sm.cq[t][i], dt[i], o);
                const int j = b * WC + t;
                if (j < dm.w) o_base[(size_t)j * o_row + c] = o;
            }
            if (need_state) {
#pragma unroll
                for (int t = 0; t < WC; ++t) sm.dl[t][c] = sm.glast[t] * dt[t];
            }
        }
        if (need_state) {
            __syncthreads();
            // S <- G_{n-1} S + sum_t k_t (g(n-1, t) d_t)^T on this thread's rows
            float2 dd[WC];
#pragma unroll
            for (int t = 0; t < WC; ++t) dd[t] = *reinterpret_cast<const float2 *>(&sm.dl[t][2 * cp]);
            const float gn = sm.gam[WC - 1];
#pragma unroll
            for (int i = 0; i < G::RPT; ++i) {
                const float4 *wr = reinterpret_cast<const float4 *>(sm.wt[rq * G::RPT + i]);
                const float4 k0 = wr[0], k1 = wr[1];
                const float kr[WC] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                float x0 = gn * xs[i].x, x1 = gn * xs[i].y;
#pragma unroll
                for (int t = 0; t < WC; ++t) {
                    x0 = fmaf(kr[t], dd[t].x, x0);
                    x1 = fmaf(kr[t], dd[t].y, x1);
                }
                xs[i] = make_float2(x0, x1);
            }
        }
        if (!more) {
            // the remaining passes (if any) only zero their output rows
            for (int bb = b + 1; bb < n_pass; ++bb)
                for (int e = tid; e < WC * D; e += G::NT) {
                    const int j = bb * WC + e / D;
                    if (j < dm.w) o_base[(size_t)j * o_row + e % D] = 0.f;
                }
            break;
        }
    }
    if (a.S_out) {
#pragma unroll
        for (int i = 0; i < G::RPT; ++i)
            reinterpret_cast<float2 *>(a.S_out + sbase + (size_t)(rq * G::RPT + i) * D)[cp] = xs[i];
    }
}

// ---------------------------------------------------------------------------
// Persistent pipelined form for d = 128 and seams of at most 8 tokens: one
// CTA per SM walks a contiguous range of seams u = ((l n_order) + e) H + h,
// so that the H heads of one request entry follow each other (the entry's
// request-table lookups, slow in the constant bank, are made once per H
// seams, and its gate and token lines stay in cache).  Four warp roles run
// one seam apart:
//   row producer (warp 12): looks the seam up and bulk-copies its raw q, k, v
//     rows (the seam plus its conv history) into a two-stage ring;
//   state producer (warp 13): bulk-copies the prefix state (64 KB) into a
//     two-stage ring and prefetches the state two seams ahead into L2;
//   prep (warps 8-11): the gates, conv, L2 normalisation, [k; q] transposed,
//     v, and the dot products and decay products of the triangular system,
//     into one of two buffers;
//   compute (warps 0-7): the column products [k; q] S0 (packed fp32 FMAs),
//     the per-column solve for d_t and the outputs o_t (and S_n).
// So the state read of seam u + 1 and the staging of seam u + 1 both
// overlap the column products of seam u.  What bounds it: two latency chains
// of about equal length per seam, the compute warps' (column products on the
// FMA pipe with broadcast shared-memory reads of [k; q], then the
// per-column solve) and the prep warps' (conv, norms, dots), coupled through
// the double-buffered hand-off.

namespace pipe {

constexpr int D = 128;
constexpr int NC = 256;            // compute threads (warps 0-7)
constexpr int NP = 128;            // prep threads (warps 8-11), one per channel
constexpr int NT = NC + NP + 64;   // + the two producer warps
constexpr int HIST = 3;            // conv history slots (taps - 1, taps <= 4)
constexpr int NPOS = HIST + WC;    // raw token slots of one seam
constexpr int BAR_C = 1, BAR_P = 2;  // named barriers of the compute and prep warps
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds

struct Info {
    int32_t t0;     // first token of the segment
    int32_t sw;     // seam length
    uint32_t mask;  // raw slots present (slot x = seam position x - HIST)
    int32_t pad;
};

// Written by the prep warps, read by the compute warps (two buffers).
struct PrepOut {
    float wt[D][MR + 4];   // [channel][k_0..k_7, q_0..q_7, pad]: 16-byte rows, conflict-free 16-byte stores
    float v[WC][D];
    float ck[WC][WC], cq[WC][WC];  // b_t g(t, i) k_t . k_i (i < t); g(t, i) q_t . k_i (i <= t)
    float gam[WC], glast[WC];      // G_t, g(7, t)
    float beta[WC];
    float pad[WC];
};
struct PrepScratch {
    float kq[MR][D];       // k_0..k_7, q_0..q_7 token-major (dot products)
    float nrm[NP / 32][MR];
    float alpha[WC], beta[WC];
};
// RS slots of partial column products: four (one per row quarter, summed by
// the readers after one barrier) when the shared memory allows it, else two
// (quarters 2, 3 added into quarters 0, 1 first, a second barrier).
template <int RS> struct CompScratch {
    float2 red[RS][MR / 2][D];  // two rows m per entry
    float dl[WC][D];           // g(7, t) d_t (state update)
};

enum { B_FULLR = 0, B_EMPTYR = 2, B_FULLS = 4, B_EMPTYS = 6, B_PREPPED = 8, B_PFREE = 10, B_COUNT = 12 };

template <typename Tin> struct Layout {
    static constexpr uint32_t S_STAGE = D * D * 4;
    static constexpr uint32_t ROW = D * sizeof(Tin);
    static constexpr uint32_t RAW_STAGE = 3 * NPOS * ROW;
    static constexpr uint32_t S = 0;
    static constexpr uint32_t RAW = S + 2 * S_STAGE;
    static constexpr uint32_t INFO = RAW + 2 * RAW_STAGE;
    static constexpr uint32_t POUT = INFO + 2 * sizeof(Info);
    static constexpr uint32_t PSCR = POUT + 2 * sizeof(PrepOut);
    static constexpr uint32_t CSCR = PSCR + sizeof(PrepScratch);
    static constexpr int RS = sizeof(Tin) == 2 ? 4 : 2;  // fp32 raw rows leave room for two slots only
    static constexpr uint32_t BAR = (CSCR + sizeof(CompScratch<RS>) + 15) / 16 * 16;
    static constexpr uint32_t BYTES = BAR + 8 * B_COUNT + 16;
    static_assert(BYTES <= 232448, "shared memory budget");
    static_assert(RAW % 16 == 0 && ROW % 16 == 0 && POUT % 16 == 0 && sizeof(PrepOut) % 16 == 0 &&
                  PSCR % 16 == 0 && CSCR % 16 == 0, "alignment");
};

__device__ __forceinline__ bool wait_bar(uint32_t mbar, uint32_t parity, volatile int *abort_flag, int *status)
{
    return tc::wait_bounded(mbar, parity, abort_flag, kWaitCycles, status);
}

// Plain (generic-address) read of a staged raw element as fp32.
__device__ __forceinline__ float raw_f(const float *p, int i) { return p[i]; }
__device__ __forceinline__ float raw_f(const __nv_bfloat16 *p, int i) { return __bfloat162float(p[i]); }

// (layer, request entry, head) of seam u = (l n_perm + e) H + h, stepped
// along u without divisions.
struct Cursor {
    int l, ent, h;
    __device__ __forceinline__ void init(long long u, const Dims &dm, int n_perm)
    {
        h = (int)(u % dm.H);
        const long long le = u / dm.H;
        ent = (int)(le % n_perm);
        l = (int)(le / n_perm);
    }
    __device__ __forceinline__ void next(const Dims &dm, int n_perm)
    {
        if (++h == dm.H) {
            h = 0;
            if (++ent == n_perm) {
                ent = 0;
                ++l;
            }
        }
    }
};

// Butterfly sum of N values (N = 8, 16 or 32) over the 32 lanes of a warp:
// each step hands half the values to the partner lane, so after log2(N)
// steps lane bits 4, 3, ... select which sum a lane carries; the remaining
// lane bits are summed plainly.  Returns the sum of value index
// (lane >> (5 - log2 N)) as laid out by those bits.
template <int N> __device__ __forceinline__ float butterfly_sum(float (&v)[N], int lane)
{
    constexpr int LOGN = N == 32 ? 5 : N == 16 ? 4 : 3;
    static_assert(N == (1 << LOGN), "8, 16 or 32 values");
#pragma unroll
    for (int st = 0; st < LOGN; ++st) {
        const int half = N >> (st + 1), bit = 16 >> st;
        const bool up = lane & bit;
#pragma unroll
        for (int x = 0; x < half; ++x) {
            const float send = up ? v[x] : v[x + half];
            const float keep = up ? v[x + half] : v[x];
            v[x] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = v[0];
#pragma unroll
    for (int st = LOGN; st < 5; ++st) r += __shfl_xor_sync(0xffffffffu, r, 16 >> st);
    return r;
}

}  // namespace pipe

template <typename Tin, int CK>
__global__ void __launch_bounds__(pipe::NT, 1)
seam_pipe_kernel(const __grid_constant__ SeamArgs a, const __grid_constant__ SegTable tab)
{
    using namespace pipe;
    using LY = Layout<Tin>;
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sb = tc::smem_u32(smem);
    auto bar = [&](int i) { return sb + LY::BAR + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + LY::BAR + 8 * B_COUNT);
    auto info = [&](int stg) -> Info & { return reinterpret_cast<Info *>(smem + LY::INFO)[stg]; };
    auto pout = [&](int b) -> PrepOut & { return reinterpret_cast<PrepOut *>(smem + LY::POUT)[b]; };
    PrepScratch &ps = *reinterpret_cast<PrepScratch *>(smem + LY::PSCR);
    constexpr int RS = LY::RS;
    CompScratch<RS> &cs = *reinterpret_cast<CompScratch<RS> *>(smem + LY::CSCR);
    const Dims dm = a.dm;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const long long n_units = (long long)dm.L * tab.n_perm * dm.H;
    const long long u_beg = n_units * blockIdx.x / gridDim.x;
    const long long u_end = n_units * (blockIdx.x + 1) / gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < B_COUNT; ++i) tc::mbar_init(bar(i), 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();

    if (warp == (NC + NP) / 32 + 1) {
        // ================================================ state producer
        if (lane != 0) return;
        int i = 0;
        for (long long u = u_beg; u < u_end; ++u, ++i) {
            const int stg = i & 1;
            if (i >= 2 && !wait_bar(bar(B_EMPTYS + stg), ((i - 2) >> 1) & 1, abort_flag, a.status)) break;
            tc::mbar_arrive_expect_tx(bar(B_FULLS + stg), LY::S_STAGE);
            tc::bulk_load(sb + LY::S + stg * LY::S_STAGE, a.S_in + u * (D * D), LY::S_STAGE, bar(B_FULLS + stg));
            if (u + 2 < u_end) tc::bulk_prefetch_l2(a.S_in + (u + 2) * (D * D), LY::S_STAGE);
        }
        // let the copies of the last two stages land before the CTA can exit
        const long long t0c = clock64();
        for (int k = i - 2; k < i; ++k) {
            if (k < 0) continue;
            while (!tc::mbar_test(bar(B_FULLS + (k & 1)), (k >> 1) & 1) && clock64() - t0c < kWaitCycles) {
            }
        }
        return;
    }

    if (warp == (NC + NP) / 32) {
        // ================================================== row producer
        const Tin *src[3] = {static_cast<const Tin *>(a.tok.q), static_cast<const Tin *>(a.tok.k),
                             static_cast<const Tin *>(a.tok.v)};
        int i = 0, cur_ent = -1, sw = 0;
        int32_t t0 = 0, tok = -1;
        uint32_t mask = 0;
        Cursor pc;
        pc.init(u_beg, dm, tab.n_perm);
        for (long long u = u_beg; u < u_end; ++u, ++i, pc.next(dm, tab.n_perm)) {
            const int stg = i & 1;
            bool ok = true;
            if (i >= 2 && lane == 0) ok = wait_bar(bar(B_EMPTYR + stg), ((i - 2) >> 1) & 1, abort_flag, a.status);
            if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
            const int l = pc.l, ent = pc.ent, h = pc.h;
            if (ent != cur_ent) {
                // request-table lookups: lane 0 the segment, lanes 1..3 the conv history
                cur_ent = ent;
                int32_t len = 0, pv = -1;
                if (lane == 0) {
                    const int s = tab.perm[ent];
                    t0 = tab.off[s];
                    len = tab.off[s + 1] - t0;
                } else if (lane < CK) {
                    pv = stream_back(tab, ent, 0, lane);
                }
                t0 = __shfl_sync(0xffffffffu, t0, 0);
                len = __shfl_sync(0xffffffffu, len, 0);
                sw = min(dm.w, len);
                const int p = lane - HIST;  // seam position of raw slot `lane`
                const int32_t pvx = __shfl_sync(0xffffffffu, pv, p < 0 ? -p : 0);
                tok = -1;
                if (lane < NPOS) tok = p >= 0 ? (p < sw ? t0 + p : -1) : (-p < CK ? pvx : -1);
                mask = __ballot_sync(0xffffffffu, tok >= 0);
            }
            if (lane == 0) {
                Info &inf = info(stg);
                inf.t0 = t0;
                inf.sw = sw;
                inf.mask = mask;
                tc::mbar_arrive_expect_tx(bar(B_FULLR + stg), (uint32_t)__popc(mask) * 3u * LY::ROW);
            }
            __syncwarp();
            if (tok >= 0) {
                const size_t ix = tok_index(dm, a.tok.N, l, tok, h, 0);
#pragma unroll
                for (int c = 0; c < 3; ++c)
                    tc::bulk_load(sb + LY::RAW + stg * LY::RAW_STAGE + (uint32_t)(c * NPOS + lane) * LY::ROW,
                                  src[c] + ix, LY::ROW, bar(B_FULLR + stg));
            }
        }
        // let the copies of the last two stages land before the CTA can exit
        if (lane == 0) {
            const long long t0c = clock64();
            for (int k = i - 2; k < i; ++k) {
                if (k < 0) continue;
                while (!tc::mbar_test(bar(B_FULLR + (k & 1)), (k >> 1) & 1) && clock64() - t0c < kWaitCycles) {
                }
            }
        }
        return;
    }

    if (warp >= NC / 32) {
        // ================================================= prep warps
        constexpr int NL = CK > 0 ? CK : 1;
        const int ch = tid - NC, pw = warp - NC / 32;
        Cursor cc;
        cc.init(u_beg, dm, tab.n_perm);
        // conv weights of channel ch, loaded one seam ahead of use
        float wq[NL], wk[NL], wv[NL];
        auto load_w = [&](const Cursor &cw) {
            if (CK > 0) {
                const float *w0 = a.tok.conv_w + (((size_t)cw.l * 3) * dm.H + cw.h) * D * NL + (size_t)ch * NL;
                const size_t step = (size_t)dm.H * D * NL;
#pragma unroll
                for (int g = 0; g < NL; ++g) {
                    wq[g] = __ldg(w0 + g);
                    wk[g] = __ldg(w0 + step + g);
                    wv[g] = __ldg(w0 + 2 * step + g);
                }
            }
        };
        load_w(cc);
        int i = 0;
        for (long long u = u_beg; u < u_end; ++u, ++i, cc.next(dm, tab.n_perm)) {
            const int stg = i & 1, b = i & 1;
            bool ok = true;
            if (ch == 0) {
                if (i >= 2) ok = wait_bar(bar(B_PFREE + b), ((i - 2) >> 1) & 1, abort_flag, a.status);
                if (ok) ok = wait_bar(bar(B_FULLR + stg), (i >> 1) & 1, abort_flag, a.status);
            }
            if (!tc::bar_and(BAR_P, NP, ok)) break;
            PrepOut &po = pout(b);
            const Info &inf = info(stg);
            const int sw = inf.sw;
            const int32_t t0 = inf.t0;
            const uint32_t mask = inf.mask;
            const Tin *raw = reinterpret_cast<const Tin *>(smem + LY::RAW + stg * LY::RAW_STAGE);
            // gates (alpha 1, beta 0 past the seam end): loaded now, stored
            // to shared memory at the end of the staging, read in the dot products
            float gate = 0.f;
            if (pw == 0 && lane < 2 * WC) {
                const int j = lane % WC;
                const Tin *gp = static_cast<const Tin *>(lane < WC ? a.tok.alpha : a.tok.beta);
                gate = j < sw ? ld_f(gp, gate_index(dm, a.tok.N, cc.l, t0 + j, cc.h)) : (lane < WC ? 1.f : 0.f);
            }

            // ---- the seam's 8 tokens for channel ch: conv, then L2 norms
            float qq[WC], kk[WC], vv[WC];
            if constexpr (CK == 0) {
#pragma unroll
                for (int j = 0; j < WC; ++j) {
                    const int x = j + HIST;
                    const bool pres = (mask >> x) & 1u;
                    qq[j] = pres ? raw_f(raw, (0 * NPOS + x) * D + ch) : 0.f;
                    kk[j] = pres ? raw_f(raw, (1 * NPOS + x) * D + ch) : 0.f;
                    vv[j] = pres ? raw_f(raw, (2 * NPOS + x) * D + ch) : 0.f;
                }
            } else {
                constexpr int NWIN = CK - 1 + WC;
                float rq_[NWIN], rk_[NWIN], rv_[NWIN];
#pragma unroll
                for (int x = 0; x < NWIN; ++x) {
                    const int slot = HIST - (CK - 1) + x;
                    const bool pres = (mask >> slot) & 1u;
                    rq_[x] = pres ? raw_f(raw, (0 * NPOS + slot) * D + ch) : 0.f;
                    rk_[x] = pres ? raw_f(raw, (1 * NPOS + slot) * D + ch) : 0.f;
                    rv_[x] = pres ? raw_f(raw, (2 * NPOS + slot) * D + ch) : 0.f;
                }
                float ss[2 * WC];
#pragma unroll
                for (int j = 0; j < WC; ++j) {
                    float q_ = 0.f, k_ = 0.f, v_ = 0.f;
#pragma unroll
                    for (int lag = 0; lag < CK; ++lag) {
                        q_ = fmaf(wq[lag], rq_[j + CK - 1 - lag], q_);
                        k_ = fmaf(wk[lag], rk_[j + CK - 1 - lag], k_);
                        v_ = fmaf(wv[lag], rv_[j + CK - 1 - lag], v_);
                    }
                    if (dm.act) {
                        q_ = silu(q_);
                        k_ = silu(k_);
                        v_ = silu(v_);
                    }
                    const bool live = j < sw;
                    qq[j] = live ? q_ : 0.f;
                    kk[j] = live ? k_ : 0.f;
                    vv[j] = live ? v_ : 0.f;
                    ss[j] = qq[j] * qq[j];
                    ss[WC + j] = kk[j] * kk[j];
                }
                // sums of squares over the warp's 32 channels: lane bits 4..1
                // select the sum index (q of token x < 8, k of token x - 8)
                const float r = butterfly_sum<2 * WC>(ss, lane);
                if ((lane & 1) == 0) ps.nrm[pw][lane >> 1] = r;
                tc::bar_sync(BAR_P, NP);
                float n[2 * WC];
#pragma unroll
                for (int x = 0; x < 2 * WC; ++x) n[x] = 0.f;
#pragma unroll
                for (int w4 = 0; w4 < NP / 32; ++w4) {
#pragma unroll
                    for (int x4 = 0; x4 < WC / 2; ++x4) {
                        const float4 t4 = reinterpret_cast<const float4 *>(ps.nrm[w4])[x4];
                        n[4 * x4 + 0] += t4.x;
                        n[4 * x4 + 1] += t4.y;
                        n[4 * x4 + 2] += t4.z;
                        n[4 * x4 + 3] += t4.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < WC; ++j) {
                    qq[j] *= rsqrtf(n[j] + kL2Eps);
                    kk[j] *= rsqrtf(n[WC + j] + kL2Eps);
                }
            }
            float4 *wr = reinterpret_cast<float4 *>(po.wt[ch]);
            wr[0] = make_float4(kk[0], kk[1], kk[2], kk[3]);
            wr[1] = make_float4(kk[4], kk[5], kk[6], kk[7]);
            wr[2] = make_float4(qq[0], qq[1], qq[2], qq[3]);
            wr[3] = make_float4(qq[4], qq[5], qq[6], qq[7]);
#pragma unroll
            for (int j = 0; j < WC; ++j) {
                ps.kq[j][ch] = kk[j];
                ps.kq[WC + j][ch] = qq[j];
                po.v[j][ch] = vv[j];
            }
            if (pw == 0 && lane < 2 * WC) {
                if (lane < WC) ps.alpha[lane] = gate;
                else ps.beta[lane - WC] = gate;
            }
            {
                Cursor cn = cc;
                cn.next(dm, tab.n_perm);
                if (u + 1 < u_end) load_w(cn);
            }
            tc::bar_sync(BAR_P, NP);
            if (ch == 0) tc::mbar_arrive(bar(B_EMPTYR + stg));  // raw rows consumed
            float al[WC], be[WC];
#pragma unroll
            for (int j = 0; j < WC; ++j) {
                al[j] = ps.alpha[j];
                be[j] = ps.beta[j];
            }
            if (pw == 0 && lane < WC) {
                float gt = 1.f, gl = 1.f, bl = 0.f;
#pragma unroll
                for (int j = 0; j < WC; ++j) {
                    if (j <= lane) gt *= al[j];
                    else gl *= al[j];
                    if (j == lane) bl = be[j];
                }
                po.gam[lane] = gt;
                po.glast[lane] = gl;
                po.beta[lane] = bl;
            }

            // ---- dot products k_t . k_i (warps 0, 1) and q_t . k_i (warps 2,
            // 3), four rows t per warp, four channels per lane, and the
            // coefficients of the triangular system
            {
                float4 kr[WC];
#pragma unroll
                for (int i2 = 0; i2 < WC; ++i2) kr[i2] = reinterpret_cast<const float4 *>(ps.kq[i2])[lane];
                const int which = pw / 2;
                // the warp's 32 partial dots (rows t = 4 (pw % 2) + g4, columns
                // i2) reduced in one reduce-scatter: lane L ends with dot
                // (g4, i2) = (L >> 3, L & 7)
                float sv[4 * WC];
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    const float4 x4 = reinterpret_cast<const float4 *>(ps.kq[which * WC + 4 * (pw % 2) + g4])[lane];
#pragma unroll
                    for (int i2 = 0; i2 < WC; ++i2) {
                        float sdot = x4.x * kr[i2].x;
                        sdot = fmaf(x4.y, kr[i2].y, sdot);
                        sdot = fmaf(x4.z, kr[i2].z, sdot);
                        sv[g4 * WC + i2] = fmaf(x4.w, kr[i2].w, sdot);
                    }
                }
                const float r = butterfly_sum<4 * WC>(sv, lane);
                const int t = 4 * (pw % 2) + (lane >> 3), i2 = lane & 7;
                float g = 1.f, bt = 0.f;
#pragma unroll
                for (int j = 0; j < WC; ++j) {
                    if (j > i2 && j <= t) g *= al[j];
                    if (j == t) bt = be[j];
                }
                if (which == 0) po.ck[t][i2] = i2 < t ? bt * g * r : 0.f;
                else po.cq[t][i2] = i2 <= t ? g * r : 0.f;
            }
            tc::bar_sync(BAR_P, NP);
            if (ch == 0) tc::mbar_arrive(bar(B_PREPPED + b));
        }
        return;
    }

    // ===================================================== compute warps
    const int cp = tid % (D / 2), rq = tid / (D / 2);
    Cursor cc;
    cc.init(u_beg, dm, tab.n_perm);
    int i = 0;
    for (long long u = u_beg; u < u_end; ++u, ++i, cc.next(dm, tab.n_perm)) {
        const int stg = i & 1, b = i & 1;
        bool ok = true;
        if (tid == 0) {
            ok = wait_bar(bar(B_PREPPED + b), (i >> 1) & 1, abort_flag, a.status);
            if (ok) ok = wait_bar(bar(B_FULLS + stg), (i >> 1) & 1, abort_flag, a.status);
        }
        if (!tc::bar_and(BAR_C, NC, ok)) break;
        const PrepOut &po = pout(b);
        const float *S0 = reinterpret_cast<const float *>(smem + LY::S + stg * LY::S_STAGE);

        // ---- partial column products [k; q] S0 over this thread's 32 rows:
        // acc[mp][j] = (P[2 mp][c_j], P[2 mp + 1][c_j]) by paired FMAs, the
        // next row's operands loaded while this row's are used
        float2 acc[MR / 2][2];
#pragma unroll
        for (int mp = 0; mp < MR / 2; ++mp) acc[mp][0] = acc[mp][1] = make_float2(0.f, 0.f);
        {
            const int r0 = rq * (D / 4);
            float2 xn = *reinterpret_cast<const float2 *>(S0 + r0 * D + 2 * cp);
            float4 wn[MR / 4];
#pragma unroll
            for (int m4 = 0; m4 < MR / 4; ++m4) wn[m4] = reinterpret_cast<const float4 *>(po.wt[r0])[m4];
#pragma unroll 4
            for (int r8 = 0; r8 < D / 4; ++r8) {
                const float2 x2 = xn;
                float4 w[MR / 4];
#pragma unroll
                for (int m4 = 0; m4 < MR / 4; ++m4) w[m4] = wn[m4];
                if (r8 + 1 < D / 4) {
                    const int r = r0 + r8 + 1;
                    xn = *reinterpret_cast<const float2 *>(S0 + r * D + 2 * cp);
#pragma unroll
                    for (int m4 = 0; m4 < MR / 4; ++m4) wn[m4] = reinterpret_cast<const float4 *>(po.wt[r])[m4];
                }
                const float2 xx = make_float2(x2.x, x2.x), yy = make_float2(x2.y, x2.y);
#pragma unroll
                for (int m4 = 0; m4 < MR / 4; ++m4) {
                    const float2 wa = make_float2(w[m4].x, w[m4].y), wb = make_float2(w[m4].z, w[m4].w);
                    acc[2 * m4][0] = __ffma2_rn(wa, xx, acc[2 * m4][0]);
                    acc[2 * m4][1] = __ffma2_rn(wa, yy, acc[2 * m4][1]);
                    acc[2 * m4 + 1][0] = __ffma2_rn(wb, xx, acc[2 * m4 + 1][0]);
                    acc[2 * m4 + 1][1] = __ffma2_rn(wb, yy, acc[2 * m4 + 1][1]);
                }
            }
        }
        // the row quarters hand their partial sums over: each into its own
        // slot (one barrier), or quarters 2, 3 into quarters 0, 1 (two)
        if (RS == 4 || rq >= 2) {
#pragma unroll
            for (int mp = 0; mp < MR / 2; ++mp) {
                cs.red[rq % RS][mp][2 * cp] = acc[mp][0];
                cs.red[rq % RS][mp][2 * cp + 1] = acc[mp][1];
            }
        }
        tc::bar_sync(BAR_C, NC);
        // without a state to write, the state stage is consumed: hand it back
        if (a.S_out == nullptr && tid == 0) tc::mbar_arrive(bar(B_EMPTYS + stg));
        if (RS == 2) {
            if (rq < 2) {
#pragma unroll
                for (int mp = 0; mp < MR / 2; ++mp) {
                    float2 &e0 = cs.red[rq][mp][2 * cp], &e1 = cs.red[rq][mp][2 * cp + 1];
                    e0 = make_float2(e0.x + acc[mp][0].x, e0.y + acc[mp][0].y);
                    e1 = make_float2(e1.x + acc[mp][1].x, e1.y + acc[mp][1].y);
                }
            }
            tc::bar_sync(BAR_C, NC);
        }

        // ---- per column: d_t, then o_t
        if (tid < D) {
            const int c = tid;
            float pk[WC], pq[WC], dt[WC];
#pragma unroll
            for (int mp = 0; mp < WC / 2; ++mp) {
                float2 k2 = cs.red[0][mp][c], q2 = cs.red[0][WC / 2 + mp][c];
#pragma unroll
                for (int qq = 1; qq < RS; ++qq) {
                    const float2 kx = cs.red[qq][mp][c], qx = cs.red[qq][WC / 2 + mp][c];
                    k2 = make_float2(k2.x + kx.x, k2.y + kx.y);
                    q2 = make_float2(q2.x + qx.x, q2.y + qx.y);
                }
                pk[2 * mp] = k2.x;
                pk[2 * mp + 1] = k2.y;
                pq[2 * mp] = q2.x;
                pq[2 * mp + 1] = q2.y;
            }
            float *o_base = a.o_out + (((size_t)cc.l * tab.n_perm + cc.ent) * dm.w * dm.H + cc.h) * D + c;
#pragma unroll
            for (int t = 0; t < WC; ++t) {
                float r = po.beta[t] * (po.v[t][c] - po.gam[t] * pk[t]);
#pragma unroll
                for (int i2 = 0; i2 < t; ++i2) r = fmaf(-po.ck[t][i2], dt[i2], r);
                dt[t] = r;
                float o = po.gam[t] * pq[t];
#pragma unroll
                for (int i2 = 0; i2 <= t; ++i2) o = fmaf(po.cq[t][i2], dt[i2], o);
                if (t < dm.w) o_base[(size_t)t * dm.H * D] = o;
            }
            if (a.S_out) {
#pragma unroll
                for (int t = 0; t < WC; ++t) cs.dl[t][c] = po.glast[t] * dt[t];
            }
        }
        if (a.S_out) {
            tc::bar_sync(BAR_C, NC);
            float2 d2[WC];
#pragma unroll
            for (int t = 0; t < WC; ++t) d2[t] = *reinterpret_cast<const float2 *>(&cs.dl[t][2 * cp]);
            const float gn = po.gam[WC - 1];
            float *so = a.S_out + u * (D * D) + 2 * cp;
#pragma unroll 4
            for (int r8 = 0; r8 < D / 4; ++r8) {
                const int r = rq * (D / 4) + r8;
                const float2 x2 = *reinterpret_cast<const float2 *>(S0 + r * D + 2 * cp);
                const float4 *wr = reinterpret_cast<const float4 *>(po.wt[r]);
                const float4 k0 = wr[0], k1 = wr[1];
                const float kr[WC] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                float x0 = gn * x2.x, x1 = gn * x2.y;
#pragma unroll
                for (int t = 0; t < WC; ++t) {
                    x0 = fmaf(kr[t], d2[t].x, x0);
                    x1 = fmaf(kr[t], d2[t].y, x1);
                }
                *reinterpret_cast<float2 *>(so + (size_t)r * D) = make_float2(x0, x1);
            }
        }
        tc::bar_sync(BAR_C, NC);
        if (tid == 0) {
            if (a.S_out) tc::mbar_arrive(bar(B_EMPTYS + stg));
            tc::mbar_arrive(bar(B_PFREE + b));
        }
    }
}

template <int D, typename Tin, int CK>
cudaError_t launch_t(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    using G = ChunkGeom<D>;
    const long long grid = (long long)tab.n_perm * a.dm.L * a.dm.H;
    if (grid == 0) return cudaSuccess;
    auto kern = seam_chunk_kernel<D, Tin, CK>;
    const int smem = (int)sizeof(ChunkSmem<D>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<(unsigned)grid, G::NT, smem, st>>>(a, tab);
    return cudaGetLastError();
}

template <int D, typename Tin> cudaError_t launch_ck(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    switch (a.dm.conv_k) {
    case 0: return launch_t<D, Tin, 0>(a, tab, st);
    case 2: return launch_t<D, Tin, 2>(a, tab, st);
    case 3: return launch_t<D, Tin, 3>(a, tab, st);
    default: return launch_t<D, Tin, 4>(a, tab, st);
    }
}

template <typename Tin> cudaError_t launch_d(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    switch (a.dm.D) {
    case 16: return launch_ck<16, Tin>(a, tab, st);
    case 32: return launch_ck<32, Tin>(a, tab, st);
    case 64: return launch_ck<64, Tin>(a, tab, st);
    default: return launch_ck<128, Tin>(a, tab, st);
    }
}

template <typename Tin, int CK> cudaError_t launch_pipe_t(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    // the SM count of the device this launch runs on (a cheap query; nothing is
    // cached across calls, which may come from several devices and threads)
    int n_sm = 0, dev = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    const long long units = (long long)tab.n_perm * a.dm.L * a.dm.H;
    if (units == 0) return cudaSuccess;
    auto kern = seam_pipe_kernel<Tin, CK>;
    const int smem = (int)pipe::Layout<Tin>::BYTES;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return err;
    const int grid = units < n_sm ? (int)units : n_sm;
    kern<<<grid, pipe::NT, smem, st>>>(a, tab);
    return cudaGetLastError();
}

template <typename Tin> cudaError_t launch_pipe(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    switch (a.dm.conv_k) {
    case 0: return launch_pipe_t<Tin, 0>(a, tab, st);
    case 2: return launch_pipe_t<Tin, 2>(a, tab, st);
    case 3: return launch_pipe_t<Tin, 3>(a, tab, st);
    default: return launch_pipe_t<Tin, 4>(a, tab, st);
    }
}

}  // namespace

cudaError_t launch_seam_chunk(const SeamArgs &a, const SegTable &tab, cudaStream_t st)
{
    // d = 128 with seams of at most 8 tokens: the persistent pipelined form;
    // otherwise one CTA per seam.
    if (a.dm.D == pipe::D && a.dm.w <= WC)
        return a.dm.dtype == HYPIC_BF16 ? launch_pipe<__nv_bfloat16>(a, tab, st) : launch_pipe<float>(a, tab, st);
    return a.dm.dtype == HYPIC_BF16 ? launch_d<__nv_bfloat16>(a, tab, st) : launch_d<float>(a, tab, st);
}

}  // namespace hypic
