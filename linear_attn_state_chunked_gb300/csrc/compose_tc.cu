// compose_tc.cu -- running-state composition with fused seams on the tcgen05
// tensor core, for gated delta with bf16 inputs at d_k = d_v = 128.
//
// HYPIC pages (codernav.top summary, sections "线性层" and "全注意力层";
// xix.ai article, linear-layer and seam-window paragraphs): at reuse the
// running state advances entry by entry as S <- T_C S + S(C|0), each segment's
// seam tokens first re-run under the running state, emitting their outputs.
//
// One CTA per (layer, head) chain.  Per request entry e:
//   * T_C and S(C|0) of the entry stream into shared memory by TMA
//     (128-byte swizzle, the tensor core's operand layout) and D = T_C S runs
//     as 16 tf32 MMAs (A = T_C, B = S^T from shared memory, D in tensor
//     memory), both driven by thread 0;
//   * the 8 warps run the seam column-parallel (a pair of threads owns column
//     j of S in registers, so u_j = k.S[:, j] needs one shuffle), write the
//     tf32-rounded state as the MMA's B operand, and after the MMA form
//     S_new = D + S(C|0) row-parallel (tensor-memory lanes), transposing it
//     through shared memory back to columns for the next seam.
// The next entry's T_C loads while this entry's epilogue and the next seam
// run; its S(C|0) loads while the seam and the MMA run.  The next entry's
// seam tokens (with their conv warm-up) are staged while the MMA runs.
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace hypic {
namespace {

constexpr int D = 128;
constexpr int WMAX = 8;     // seam window served by this kernel
constexpr int NMAIN = 256;  // 8 warps: seams, epilogue, outputs; thread 0 also drives TMA and the MMA
constexpr int NT = NMAIN;
constexpr int BAR_MAIN = 1;
constexpr long long kWaitCycles = 4000000000LL;

constexpr uint32_t SM_T = 0;           // T_C   [128][128] fp32, sw128 (A)
constexpr uint32_t SM_SC = 65536;      // S(C|0) [128][128] fp32, sw128
constexpr uint32_t SM_ST = 131072;     // S^T  [128][128] fp32, sw128 (B; also the transpose buffer)
constexpr int TOK_F = 3 * D + 4;       // q, k, v, alpha, beta (+pad) per token
constexpr uint32_t SM_TOK = 196608;    // [WMAX][TOK_F] fp32: the staged seam tokens
constexpr int HIST = 3;                // conv history rows (taps - 1, taps <= 4)
constexpr int RAW_ROWS = HIST + WMAX;  // per tensor: history rows, then the seam rows
constexpr uint32_t RAW_T = RAW_ROWS * D * 2;           // bytes per tensor (bf16)
constexpr uint32_t SM_RAW = SM_TOK + WMAX * TOK_F * 4;  // 2 buffers x {q, k, v} raw rows (TMA)
constexpr uint32_t SM_RED = SM_RAW + 2 * 3 * RAW_T;     // [8 warps][WMAX][2] partial sums
constexpr uint32_t SM_BAR = SM_RED + 8 * WMAX * 2 * 4;
constexpr uint32_t SM_MISC = SM_BAR + 8 * 8;
constexpr uint32_t SM_BYTES = SM_MISC + 64;
constexpr uint32_t SMEM_DYN = SM_BYTES + 1024;
static_assert(SMEM_DYN <= 232448, "shared memory budget");
static_assert(SM_RAW % 128 == 0 && RAW_T % 128 == 0 && (HIST * D * 2) % 128 == 0, "TMA alignment");

enum { B_FULLT = 0, B_FULLSC, B_MMADONE, B_FULLR0, B_FULLR1, B_COUNT };

__device__ __forceinline__ bool wait_bar(uint32_t mbar, uint32_t parity, volatile int *abort_flag)
{
    const long long t0 = clock64();
    while (!tc::mbar_try(mbar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

struct TokMaps {
    CUtensorMap rows8[3];  // q, k, v: boxes of WMAX token rows
    CUtensorMap rows3[3];  // q, k, v: boxes of HIST token rows (conv history)
};

// Whether the conv history of entry e's seam is the previous entry's last
// HIST tokens, fetched by TMA (otherwise the history crosses several short
// segments or precedes the request, and the staging reads it directly).
__device__ __forceinline__ bool hist_by_tma(const SegTable &tab, int e)
{
    if (e == 0) return false;
    const int sp = tab.perm[e - 1];
    return tab.off[sp + 1] - tab.off[sp] >= HIST;
}

// Stage seam tokens t < sw of request entry e from the raw rows the TMA
// brought in (the 256 main threads; thread = channel c of tokens
// th*WMAX/2 .. th*WMAX/2 + WMAX/2 - 1): q, k, v (convolved along the request
// stream when CK > 0, then q and k L2-normalised per token).  alpha and beta
// come in registers from threads 0 .. 2*WMAX-1 (gab: thread t < WMAX holds
// alpha of token t, thread WMAX + t beta).
template <int CK>
__device__ void stage_seam(float *tok, float *red, const uint8_t *raw, const Dims &dm, const TokPtrs &tk,
                           const SegTable &tab, int l, int h, int e, int sw, int tid, float gab)
{
    constexpr int TH = WMAX / 2;
    constexpr int NL = CK > 0 ? CK : 1;
    const int c = tid & (D - 1), th = tid >> 7;
    const bool htma = CK > 0 && hist_by_tma(tab, e);
    float wq[NL], wk[NL], wv[NL];
    if (CK > 0) {
        const float *w0 = tk.conv_w + (((size_t)l * 3 + 0) * dm.H + h) * D * CK + c * CK;
#pragma unroll
        for (int j = 0; j < NL; ++j) {
            wq[j] = __ldg(w0 + j);
            wk[j] = __ldg(w0 + (size_t)dm.H * D * CK + j);
            wv[j] = __ldg(w0 + 2 * (size_t)dm.H * D * CK + j);
        }
    }
    auto raw_at = [&](int tensor, int row) {
        const uint16_t u = *reinterpret_cast<const uint16_t *>(raw + tensor * RAW_T + (row * D + c) * 2);
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    };
    float sq[TH], sk[TH];
#pragma unroll
    for (int tt = 0; tt < TH; ++tt) {
        const int t = th * TH + tt;
        sq[tt] = sk[tt] = 0.f;
        if (t >= sw) continue;
        float qv = 0.f, kv = 0.f, vv = 0.f;
#pragma unroll
        for (int lag = 0; lag < NL; ++lag) {
            float rq, rk, rv;
            if (t - lag >= 0 || htma) {
                const int row = HIST + t - lag;
                rq = raw_at(0, row);
                rk = raw_at(1, row);
                rv = raw_at(2, row);
            } else {
                // history across short segments or before the request start
                const int32_t tb = stream_back(tab, e, t, lag);
                rq = rk = rv = 0.f;
                if (tb >= 0) {
                    const size_t ix = tok_index(dm, tk.N, l, tb, h, c);
                    rq = __bfloat162float(static_cast<const __nv_bfloat16 *>(tk.q)[ix]);
                    rk = __bfloat162float(static_cast<const __nv_bfloat16 *>(tk.k)[ix]);
                    rv = __bfloat162float(static_cast<const __nv_bfloat16 *>(tk.v)[ix]);
                }
            }
            if (CK == 0) {
                qv = rq; kv = rk; vv = rv;
            } else {
                qv = fmaf(wq[lag], rq, qv);
                kv = fmaf(wk[lag], rk, kv);
                vv = fmaf(wv[lag], rv, vv);
            }
        }
        float *row = tok + t * TOK_F;
        row[c] = qv;
        row[D + c] = kv;
        row[2 * D + c] = vv;
        sq[tt] = qv * qv;
        sk[tt] = kv * kv;
    }
    if (tid < 2 * WMAX && (tid & (WMAX - 1)) < sw) tok[(tid & (WMAX - 1)) * TOK_F + 3 * D + (tid >= WMAX)] = gab;
    if (CK > 0) {
        const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
        for (int tt = 0; tt < TH; ++tt) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq[tt] += __shfl_xor_sync(0xffffffffu, sq[tt], o);
                sk[tt] += __shfl_xor_sync(0xffffffffu, sk[tt], o);
            }
            if (lane == 0) {
                red[(warp * WMAX + tt) * 2] = sq[tt];
                red[(warp * WMAX + tt) * 2 + 1] = sk[tt];
            }
        }
        tc::bar_sync(BAR_MAIN, NMAIN);
#pragma unroll
        for (int tt = 0; tt < TH; ++tt) {
            const int t = th * TH + tt;
            if (t >= sw) continue;
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                a += red[((4 * th + w) * WMAX + tt) * 2];
                b += red[((4 * th + w) * WMAX + tt) * 2 + 1];
            }
            float *row = tok + t * TOK_F;
            row[c] *= 1.f / sqrtf(a + kL2Eps);
            row[D + c] *= 1.f / sqrtf(b + kL2Eps);
        }
    }
}

template <int CK>
__global__ void __launch_bounds__(NT, 1)
compose_tc_kernel(const __grid_constant__ ComposeArgs a, const __grid_constant__ SegTable tab,
                  const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmS,
                  const __grid_constant__ TokMaps tmX)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = tc::smem_u32(sm);
    auto bar = [&](int i) { return s_base + SM_BAR + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM_MISC);
    uint32_t *tmem_base_sh = reinterpret_cast<uint32_t *>(sm + SM_MISC + 16);
    float *red = reinterpret_cast<float *>(sm + SM_RED);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Dims dm = a.dm;
    const int l = blockIdx.x / dm.H, h = blockIdx.x % dm.H;
    const int n_ent = tab.n_perm;
    const int w = dm.w;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i) tc::mbar_init(bar(i), 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_base_sh), 128);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = *tmem_base_sh;

    {
        // ------------------------------------------------ main warps: seams, epilogue, outputs
        // Seam / state layout: the thread pair (tid, tid ^ 1) owns column
        // j = tid / 2; thread hf = tid % 2 holds rows 8m + 4hf .. 8m + 4hf + 3
        // (m = 0..15) in x[4m .. 4m + 3], so a warp's 16-byte reads of k and q
        // hit two adjacent chunks (no bank conflict); the pair's partial dot
        // products meet by a shuffle.  Epilogue layout: tensor-memory lane
        // i = 32 (warp % 4) + lane, columns 64 (warp / 4) .. + 63.
        constexpr int HR = D / 2;
        const int j = tid >> 1, hf = tid & 1;
        auto RW = [&](int r) { return 8 * (r >> 2) + 4 * hf + (r & 3); };
        const int lane_i = 32 * (warp & 3) + lane, cbase = 64 * (warp >> 2);
        const uint32_t my = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const size_t st_base = ((size_t)l * dm.H + h) * D * D;
        float *toks = reinterpret_cast<float *>(sm + SM_TOK);
        // thread 0 drives the copies and the MMA
        auto pair_row = [&](int e) {
            return (int)((((size_t)l * tab.n_seg + tab.perm[e]) * dm.H + h) * D);
        };
        auto load_T = [&](int e) {
            tc::mbar_arrive_expect_tx(bar(B_FULLT), D * D * 4);
#pragma unroll
            for (int at = 0; at < 4; ++at)
                tc::tma_load_2d(s_base + SM_T + at * 16384, &tmT, 32 * at, pair_row(e), bar(B_FULLT));
        };
        auto load_SC = [&](int e) {
            tc::mbar_arrive_expect_tx(bar(B_FULLSC), D * D * 4);
#pragma unroll
            for (int at = 0; at < 4; ++at)
                tc::tma_load_2d(s_base + SM_SC + at * 16384, &tmS, 32 * at, pair_row(e), bar(B_FULLSC));
        };
        // raw seam rows of entry e (and the conv history rows when they are the
        // previous entry's last tokens) into raw buffer e & 1
        auto load_raw = [&](int e) {
            const int s = tab.perm[e];
            const uint32_t fb = bar(B_FULLR0 + (e & 1));
            const int sw = min(w, tab.off[s + 1] - tab.off[s]);
            if (sw == 0) {
                tc::mbar_arrive(fb);
                return;
            }
            const bool htma = CK > 0 && hist_by_tma(tab, e);
            tc::mbar_arrive_expect_tx(fb, 3 * WMAX * D * 2 + (htma ? 3 * HIST * D * 2 : 0));
            const uint32_t rb = s_base + SM_RAW + (e & 1) * 3 * RAW_T;
#pragma unroll
            for (int x3 = 0; x3 < 3; ++x3) {
                tc::tma_load_4d(rb + x3 * RAW_T + HIST * D * 2, &tmX.rows8[x3], 0, h, tab.off[s], l, fb);
                if (htma)
                    tc::tma_load_4d(rb + x3 * RAW_T, &tmX.rows3[x3], 0, h, tab.off[tab.perm[e - 1] + 1] - HIST, l, fb);
            }
        };
        auto load_gates = [&](int e) {  // threads 0 .. 2*WMAX-1: alpha / beta of token tid % WMAX
            float v = 0.f;
            const int s = tab.perm[e];
            const int t = tid & (WMAX - 1);
            if (tid < 2 * WMAX && t < min(w, tab.off[s + 1] - tab.off[s])) {
                const size_t gi = gate_index(dm, a.tok.N, l, tab.off[s] + t, h);
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(tid < WMAX ? a.tok.alpha : a.tok.beta);
                v = __bfloat162float(src[gi]);
            }
            return v;
        };
        auto stage = [&](int e, float gab) -> bool {
            bool wr = true;
            if (tid == 0) wr = wait_bar(bar(B_FULLR0 + (e & 1)), (e >> 1) & 1, abort_flag);
            if (!tc::bar_and(BAR_MAIN, NMAIN, wr)) return false;
            const int s = tab.perm[e];
            stage_seam<CK>(toks, red, sm + SM_RAW + (e & 1) * 3 * RAW_T, dm, a.tok, tab, l, h, e,
                           min(w, tab.off[s + 1] - tab.off[s]), tid, gab);
            return true;
        };
        int armed = 0;  // entries whose copies were issued
        if (tid == 0 && n_ent > 0) {
            load_T(0);
            load_SC(0);
            armed = 1;
            if (w > 0) load_raw(0);
        }
        float x[HR];
#pragma unroll
        for (int r = 0; r < HR; ++r) x[r] = a.S_init ? a.S_init[st_base + (size_t)RW(r) * D + j] : 0.f;
        bool ok = true;
        if (w > 0 && n_ent > 0) ok = stage(0, load_gates(0));
        for (int e = 0; e < n_ent && ok; ++e) {
            const int s = tab.perm[e];
            const int sw = min(w, tab.off[s + 1] - tab.off[s]);
            // next entry's raw seam rows and gates start loading now
            float gab = 0.f;
            if (w > 0 && e + 1 < n_ent) {
                if (tid == 0) load_raw(e + 1);
                gab = load_gates(e + 1);
            }
            if (a.S_prefix) {
                float *dst = a.S_prefix + (((size_t)l * n_ent + e) * dm.H + h) * D * D + j;
#pragma unroll
                for (int r = 0; r < HR; ++r) dst[(size_t)RW(r) * D] = x[r];
            }
            // ---- seam of entry e (tokens staged in buffer e & 1)
            if (w > 0) {
                tc::bar_sync(BAR_MAIN, NMAIN);  // staged tokens visible
                const float *tok = toks;
                float *o_dst = a.o_out + (((size_t)l * n_ent + e) * w) * dm.H * D + (size_t)h * D + j;
                for (int t = 0; t < w; ++t) {
                    float o = 0.f;
                    if (t < sw) {
                        const float *row = tok + t * TOK_F;
                        const float al = row[3 * D], be = row[3 * D + 1];
                        float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
                        for (int r = 0; r < HR; r += 4) {
                            const float4 k4 = *reinterpret_cast<const float4 *>(row + D + RW(r));
                            u0 = fmaf(k4.x, x[r], u0);
                            u1 = fmaf(k4.y, x[r + 1], u1);
                            u2 = fmaf(k4.z, x[r + 2], u2);
                            u3 = fmaf(k4.w, x[r + 3], u3);
                        }
                        float u = (u0 + u1) + (u2 + u3);
                        u += __shfl_xor_sync(0xffffffffu, u, 1);
                        const float coef = be * (row[2 * D + j] - al * u);
                        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
                        for (int r = 0; r < HR; r += 4) {
                            const float4 k4 = *reinterpret_cast<const float4 *>(row + D + RW(r));
                            const float4 q4 = *reinterpret_cast<const float4 *>(row + RW(r));
                            x[r] = fmaf(k4.x, coef, al * x[r]);
                            x[r + 1] = fmaf(k4.y, coef, al * x[r + 1]);
                            x[r + 2] = fmaf(k4.z, coef, al * x[r + 2]);
                            x[r + 3] = fmaf(k4.w, coef, al * x[r + 3]);
                            o0 = fmaf(q4.x, x[r], o0);
                            o1 = fmaf(q4.y, x[r + 1], o1);
                            o2 = fmaf(q4.z, x[r + 2], o2);
                            o3 = fmaf(q4.w, x[r + 3], o3);
                        }
                        o = (o0 + o1) + (o2 + o3);
                    }
                    o += __shfl_xor_sync(0xffffffffu, o, 1);
                    if (hf == 0) o_dst[(size_t)t * dm.H * D] = o;
                }
            }
            // ---- B operand: S^T row j = column j of S, rounded to tf32
#pragma unroll
            for (int r = 0; r < HR; r += 4)
                *reinterpret_cast<float4 *>(sm + SM_ST + tc::sw128_f32(j, RW(r), D)) =
                    make_float4(tc::round_tf32(x[r]), tc::round_tf32(x[r + 1]), tc::round_tf32(x[r + 2]),
                                tc::round_tf32(x[r + 3]));
            tc::fence_async_smem();
            tc::bar_sync(BAR_MAIN, NMAIN);
            bool wm = true;
            if (tid == 0) {
                wm = wait_bar(bar(B_FULLT), e & 1, abort_flag);
                if (wm) {
                    tc::fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 8; ++ks)
                        tc::mma_ss(tb, tc::sdesc_kstep(s_base + SM_T, D, ks),
                                   tc::sdesc_kstep(s_base + SM_ST, D, ks), tc::idesc_tf32(128, 128), ks > 0);
                    tc::commit(bar(B_MMADONE));
                }
            }
            // ---- stage the next entry's seam tokens while the MMA runs
            if (w > 0 && e + 1 < n_ent && !stage(e + 1, gab)) { ok = false; break; }
            // ---- epilogue: S_new row i = (T_C S)[i][:] + S(C|0)[i][:], transposed into S^T
            bool wt = wm;
            if (tid == 0 && wt) {
                wt = wait_bar(bar(B_MMADONE), e & 1, abort_flag);
                if (wt && e + 1 < n_ent) load_T(e + 1);  // T buffer free once the MMA is done
                if (wt) wt = wait_bar(bar(B_FULLSC), e & 1, abort_flag);
            }
            if (!tc::bar_and(BAR_MAIN, NMAIN, wt)) { ok = false; break; }
            tc::fence_after();
            {
                float dv[32];
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    const int cc = cbase + c0;
                    tc::tmem_ld32(my + cc, dv);
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        const float4 s4 =
                            *reinterpret_cast<const float4 *>(sm + SM_SC + tc::sw128_f32(lane_i, cc + q, D));
                        *reinterpret_cast<float *>(sm + SM_ST + tc::sw128_f32(cc + q, lane_i, D)) = dv[q] + s4.x;
                        *reinterpret_cast<float *>(sm + SM_ST + tc::sw128_f32(cc + q + 1, lane_i, D)) = dv[q + 1] + s4.y;
                        *reinterpret_cast<float *>(sm + SM_ST + tc::sw128_f32(cc + q + 2, lane_i, D)) = dv[q + 2] + s4.z;
                        *reinterpret_cast<float *>(sm + SM_ST + tc::sw128_f32(cc + q + 3, lane_i, D)) = dv[q + 3] + s4.w;
                    }
                }
            }
            tc::fence_before();
            tc::bar_sync(BAR_MAIN, NMAIN);
            if (tid == 0 && e + 1 < n_ent) {  // S(C|0) buffer consumed
                load_SC(e + 1);
                armed = e + 2;
            }
            // ---- back to columns
#pragma unroll
            for (int r = 0; r < HR; r += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(sm + SM_ST + tc::sw128_f32(j, RW(r), D));
                x[r] = v4.x;
                x[r + 1] = v4.y;
                x[r + 2] = v4.z;
                x[r + 3] = v4.w;
            }
        }
        if (ok) {
#pragma unroll
            for (int r = 0; r < HR; ++r) a.S_final[st_base + (size_t)RW(r) * D + j] = x[r];
        } else if (tid == 0 && armed > 0) {
            // aborted: let the copies in flight land before the CTA exits
            const long long t0 = clock64();
            while ((!tc::mbar_test(bar(B_FULLT), (armed - 1) & 1) || !tc::mbar_test(bar(B_FULLSC), (armed - 1) & 1)) &&
                   clock64() - t0 < kWaitCycles) {
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tb, 128);
}

}  // namespace

bool compose_tc_supported(const Dims &dm)
{
    return dm.mode == HYPIC_GATED_DELTA && dm.dtype == HYPIC_BF16 && dm.D == 128 && dm.w <= WMAX &&
           (dm.conv_k == 0 || dm.conv_k == 4);
}

cudaError_t launch_compose_tc(const ComposeArgs &a, const SegTable &tab, cudaStream_t st)
{
    const int n_chain = a.dm.L * a.dm.H;
    CUtensorMap tmT, tmS;
    cudaError_t e;
    // T and S(C|0) as 2-D [rows = L * n_seg * H * 128][128] fp32, 32-column
    // boxes of 128 rows in the 128-byte swizzle.
    const cuuint64_t rows = (cuuint64_t)a.dm.L * (cuuint64_t)(tab.n_seg > 0 ? tab.n_seg : 1) * a.dm.H * D;
    const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 4};
    const cuuint32_t box[2] = {32u, (cuuint32_t)D};
    const void *tb = a.T ? a.T : a.S_final;  // unused when the request is empty
    const void *sb = a.S ? a.S : a.S_final;
    if ((e = encode_tiled(&tmT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, tb, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    if ((e = encode_tiled(&tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, sb, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
        return e;
    // raw token rows for the seams: [L][N][H][128] bf16, boxes of WMAX and HIST rows
    TokMaps tmX;
    memset(&tmX, 0, sizeof(tmX));
    if (a.dm.w > 0 && a.tok.N > 0) {
        const void *bases[3] = {a.tok.q, a.tok.k, a.tok.v};
        const cuuint64_t tdims[4] = {(cuuint64_t)D, (cuuint64_t)a.dm.H, (cuuint64_t)a.tok.N, (cuuint64_t)a.dm.L};
        const cuuint64_t tstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.dm.H * D * 2,
                                    (cuuint64_t)a.tok.N * a.dm.H * D * 2};
        const cuuint32_t box8[4] = {(cuuint32_t)D, 1u, (cuuint32_t)WMAX, 1u};
        const cuuint32_t box3[4] = {(cuuint32_t)D, 1u, (cuuint32_t)HIST, 1u};
        for (int x3 = 0; x3 < 3; ++x3) {
            if ((e = encode_tiled(&tmX.rows8[x3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bases[x3], tdims, tstr, box8,
                                  CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
                return e;
            if ((e = encode_tiled(&tmX.rows3[x3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bases[x3], tdims, tstr, box3,
                                  CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
                return e;
        }
    }
    if (a.dm.conv_k == 0) {
        if ((e = cudaFuncSetAttribute(compose_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN)))
            return e;
        compose_tc_kernel<0><<<n_chain, NT, SMEM_DYN, st>>>(a, tab, tmT, tmS, tmX);
    } else {
        if ((e = cudaFuncSetAttribute(compose_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN)))
            return e;
        compose_tc_kernel<4><<<n_chain, NT, SMEM_DYN, st>>>(a, tab, tmT, tmS, tmX);
    }
    return cudaGetLastError();
}

}  // namespace hypic
