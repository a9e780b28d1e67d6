// compose_tc.cu -- running-state composition with fused seams on the tcgen05
// tensor core, for gated delta with bf16 inputs at d_k = d_v = 128.
//
// HYPIC pages (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, sections "线性层" and "全注意力层";
// article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, linear-layer and seam-window paragraphs): at reuse the
// running state advances entry by entry as S <- T_C S + S(C|0), each segment's
// seam tokens first re-run under the running state, emitting their outputs.
//
// One CTA per (layer, head) chain.  The running state lives in tensor memory
// transposed, X = S^T (lane j holds column j of S), in fp32, with its tf32
// rounding Xhi beside it for use as an MMA operand.  Per request entry:
//
//   seam (w <= 8 tokens, one chunk of the WY form of the recurrence; with
//   g_t = sum_{r<=t} log alpha_r, Gamma_t = e^{g_t}):
//     [u_t | z_t]    = S^T [k_t | q_t]                 tensor core, tf32
//     U              = (I + L)^{-1} (V - diag(Gamma) K S)   per column, CUDA cores
//                      L_ts = beta_s e^{g_t - g_s} k_t.k_s  (s < t)
//     o_t            = Gamma_t z_t + sum_{s<=t} e^{g_t - g_s} beta_s (q_t.k_s) U_s
//     S             <- Gamma_w S + K^T diag(beta_s e^{g_w - g_s}) U
//                      (X pre-scaled by Gamma_w when the previous entry's
//                      state is formed, then one K = 8 MMA, 3xTF32)
//   body:  S <- T_C S + S(C|0)     (tensor core: A = Xhi from tensor memory,
//                                   B = T_C rows from shared memory)
//
// Warp roles: warps 0-7 own the state (two warps per tensor-memory lane
// quadrant, each half of the columns; lane j = column j of S), thread 0 also
// issuing the MMAs and the T_C / S(C|0) copies; warps 8-11 stage each
// entry's seam ahead of time (conv warm-up across the segment boundary, L2
// normalisation, the seam's 8 x 8 Gram and triangular inverse, all
// independent of the state) into double buffers.  T_C and S(C|0) of the next
// entry stream in by TMA as soon as their buffers free up.
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace hypic {
namespace {

constexpr int D = 128;
constexpr int WMAX = 8;       // seam window served by this kernel
constexpr int HIST = 3;       // conv history rows (taps - 1, taps <= 4)
constexpr int NS = 256;       // state threads (warps 0-7, two per tensor-memory lane quadrant)
constexpr int NG = 128;       // staging threads (warps 8-11)
constexpr int NT = NS + NG;
constexpr int BAR_STATE = 1, BAR_STAGE = 2;
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds

// tensor-memory columns
constexpr uint32_t TM_X = 0;      // S^T, fp32 (pre-scaled by Gamma_w of the next seam)
constexpr uint32_t TM_XHI = 128;  // tf32(S^T), unscaled
constexpr uint32_t TM_Y = 256;    // T_C S (transposed); during the seam: [u | z] and W
constexpr uint32_t TM_D2 = TM_Y;       // 4 x 16 columns: partial [u_t | z_t] over quarters of k
constexpr uint32_t TM_W = TM_Y + 64;   // 24 columns: Whi, Wlo, Whi
constexpr uint32_t TM_COLS = 512;

// shared memory
constexpr uint32_t SM_T = 0;         // T_C    [128][128] fp32, sw128 (B of the body MMA)
constexpr uint32_t SM_SC = 65536;    // S(C|0) [128][128] fp32, sw128
constexpr uint32_t SM_BUF = 131072;  // 2 x staged seam
constexpr uint32_t BF_KQH = 0;       //   [k_t ; q_t] tf32 hi [16][128], sw128 (B of the seam MMA)
constexpr uint32_t BF_KQF = 8192;    //   the same in fp32 (for the seam's Gram)
constexpr uint32_t BF_KP = 16384;    //   K^T [128][32] sw128: columns t, 8 + t = hi(k_t), 16 + t = lo(k_t)
constexpr uint32_t BF_V = 32768;     //   v_t [8][128] fp32
constexpr uint32_t BF_SMALL = 36864; //   M [8][8], AQ [8][8], Gamma [8], d [8], Gamma_w, beta [8], g [8]
constexpr uint32_t BUF_BYTES = 37888;
constexpr int SMALL_M = 0, SMALL_AQ = 64, SMALL_G = 128, SMALL_D = 136, SMALL_GL = 144, SMALL_SW = 145,
              SMALL_B = 152, SMALL_LG = 160;
constexpr uint32_t RAW_T = (HIST + WMAX) * D * 2;           // raw rows per tensor (bf16)
constexpr uint32_t SM_RAW = SM_BUF + 2 * BUF_BYTES;         // 2 x {q, k, v} raw rows (TMA)
constexpr uint32_t SM_RED = SM_RAW + 2 * 3 * RAW_T;         // staging scratch (below)
constexpr int RED_DOTS = 4 * WMAX * 2;                      //   after [4 warps][8 tokens][2] norms: dots [64]
constexpr int RED_SCR = RED_DOTS + 64;                      //   beta_s e^{g_t - g_s} [64], L [64]
constexpr uint32_t SM_BAR = SM_RED + (RED_SCR + 128) * 4;
constexpr uint32_t SM_MISC = SM_BAR + 16 * 8;
constexpr uint32_t SM_BYTES = SM_MISC + 64;
constexpr uint32_t SMEM_DYN = SM_BYTES + 1024;
static_assert(SMEM_DYN <= 232448, "shared memory budget");
static_assert(SM_BUF % 1024 == 0 && BUF_BYTES % 1024 == 0 && BF_KP % 1024 == 0 && BF_KQF % 1024 == 0,
              "operand tile alignment");
static_assert(SM_RAW % 128 == 0 && RAW_T % 128 == 0 && (HIST * D * 2) % 128 == 0, "TMA alignment");

enum {
    B_FULLT = 0,   // T_C of the entry landed                     TMA -> state
    B_FULLSC,      // S(C|0) of the entry landed                  TMA -> state
    B_FULLR0,      // [2] raw seam rows landed                    TMA -> staging
    B_STAGED0 = B_FULLR0 + 2,    // [2] seam staged               staging -> state
    B_BUFFREE0 = B_STAGED0 + 2,  // [2] staged buffer consumed    MMA -> staging
    B_SEAMDONE = B_BUFFREE0 + 2, // [u | z] in tensor memory      MMA -> state
    B_UPDDONE,     // seam update of X done                       MMA -> state
    B_BODYDONE,    // T_C S in tensor memory                      MMA -> state
    B_COUNT
};

__device__ __forceinline__ bool wait_bar(uint32_t mbar, uint32_t parity, volatile int *abort_flag, int *status)
{
    return tc::wait_bounded(mbar, parity, abort_flag, kWaitCycles, status);
}

struct TokMaps {
    CUtensorMap rows8[3];  // q, k, v: boxes of WMAX token rows
    CUtensorMap rows3[3];  // q, k, v: boxes of HIST token rows (conv history)
};

// What the staging needs of request entry e, read from the request table in
// one go (the table sits in the constant bank, where misses are slow, so the
// staging looks entries up ahead of their use).
struct EntryInfo {
    int32_t off;   // first token of the segment
    int sw;        // seam length
    int htma;      // conv history by TMA (the previous entry has >= HIST tokens)
    int32_t hrow;  // first conv-history row when htma
};

__device__ __forceinline__ EntryInfo entry_info(const SegTable &tab, int e, int w, int ck)
{
    EntryInfo r{0, 0, 0, 0};
    const int s = tab.perm[e];
    r.off = tab.off[s];
    r.sw = min(w, tab.off[s + 1] - r.off);
    if (ck > 0 && e > 0) {
        const int sp = tab.perm[e - 1];
        const int32_t pend = tab.off[sp + 1];
        r.htma = (pend - tab.off[sp]) >= HIST;
        r.hrow = pend - HIST;
    }
    return r;
}

// Dot product index p (0..63) of the staged seam: 28 k_t.k_s (s < t), then
// 36 q_t.k_s (s <= t).  Rows of the [k ; q] tile: k_t in row t, q_t in row 8 + t.
__device__ __forceinline__ void dot_rows(int p, int &ra, int &rb, int &t, int &s)
{
    if (p < 28) {
        t = 1;
        while (p >= t) { p -= t; ++t; }
        s = p;
        ra = t;
        rb = s;
    } else {
        p -= 28;
        t = 0;
        while (p > t) { p -= t + 1; ++t; }
        s = p;
        ra = WMAX + t;
        rb = s;
    }
}

template <int CK>
__global__ void __launch_bounds__(NT, 1)
compose_tc_kernel(const __grid_constant__ ComposeArgs a, const __grid_constant__ SegTable tab,
                  const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmS,
                  const __grid_constant__ TokMaps tmX)
{
    extern __shared__ uint8_t smem_raw[];
    // the 1024-aligned base, derived from the shared array itself so that every
    // access through it stays a shared-memory access
    const uint32_t raw_u32 = tc::smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t s_base = tc::smem_u32(sm);
    auto bar = [&](int i) { return s_base + SM_BAR + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM_MISC);
    uint32_t *tmem_base_sh = reinterpret_cast<uint32_t *>(sm + SM_MISC + 16);

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
    // K^T tiles: columns 24..31 stay zero
    for (int i = tid; i < 2 * D * 32; i += NT)
        reinterpret_cast<float *>(sm + SM_BUF + (i >> 12) * BUF_BYTES + BF_KP)[i & 4095] = 0.f;
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_base_sh), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = *tmem_base_sh;

    // first row of entry e's pair in the [L * n_seg * H * 128][128] views of T and S
    auto pair_row = [&](int e) { return (int)((((size_t)l * tab.n_seg + tab.perm[e]) * dm.H + h) * D); };
    auto load_T = [&](int row) {
        tc::mbar_arrive_expect_tx(bar(B_FULLT), D * D * 4);
#pragma unroll
        for (int at = 0; at < 4; ++at)
            tc::tma_load_2d(s_base + SM_T + at * 16384, &tmT, 32 * at, row, bar(B_FULLT));
    };
    // T_C and S(C|0) of a pair into L2 ahead of their copies to shared memory
    auto prefetch_pair = [&](int row) {
#pragma unroll
        for (int at = 0; at < 4; ++at) {
            tc::tma_prefetch_2d(&tmT, 32 * at, row);
            tc::tma_prefetch_2d(&tmS, 32 * at, row);
        }
    };
    auto load_SC = [&](int row) {
        tc::mbar_arrive_expect_tx(bar(B_FULLSC), D * D * 4);
#pragma unroll
        for (int at = 0; at < 4; ++at)
            tc::tma_load_2d(s_base + SM_SC + at * 16384, &tmS, 32 * at, row, bar(B_FULLSC));
    };
    // raw seam rows of entry e (and the conv history rows when they are the
    // previous entry's last tokens) into raw buffer e & 1
    auto load_raw = [&](int e, const EntryInfo &ei) {
        const uint32_t fb = bar(B_FULLR0 + (e & 1));
        if (ei.sw == 0) {
            tc::mbar_arrive(fb);
            return;
        }
        const bool htma = CK > 0 && ei.htma;
        tc::mbar_arrive_expect_tx(fb, 3 * WMAX * D * 2 + (htma ? 3 * HIST * D * 2 : 0));
        const uint32_t rb = s_base + SM_RAW + (e & 1) * 3 * RAW_T;
#pragma unroll
        for (int x3 = 0; x3 < 3; ++x3) {
            tc::tma_load_4d(rb + x3 * RAW_T + HIST * D * 2, &tmX.rows8[x3], 0, h, ei.off, l, fb);
            if (htma) tc::tma_load_4d(rb + x3 * RAW_T, &tmX.rows3[x3], 0, h, ei.hrow, l, fb);
        }
    };

    const size_t st_base = ((size_t)l * dm.H + h) * D * D;
    if (warp < NS / 32) {
        // ================================================= state warps
        // lane j = 32 (warp % 4) + lane of tensor memory = column j of S;
        // this thread's columns of X are 64 hf .. 64 hf + 63.  Thread 0 also
        // issues every MMA and the T_C / S(C|0) copies.
        const int j = 32 * (warp & 3) + lane, hf = warp >> 2;
        const uint32_t my = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        int t_armed = 0, sc_armed = 0;  // copies issued
        auto issue_seam = [&](int e) {
            const uint32_t buf = s_base + SM_BUF + (e & 1) * BUF_BYTES;
            tc::fence_after();
            // [u | z] = Xhi [k | q]^T in tf32, as four independent partial sums
            // over quarters of k (columns 16 p .. 16 p + 15) so the MMAs overlap
#pragma unroll 1
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_ts(tb + TM_D2 + 16 * (ks & 3), tb + TM_XHI + ks * 8,
                           tc::sdesc_kstep(buf + BF_KQH, 2 * WMAX, ks), tc::idesc_tf32(128, 2 * WMAX), ks >= 4);
            tc::commit(bar(B_SEAMDONE));
        };
        auto issue_body = [&](int e) -> bool {
            if (!wait_bar(bar(B_FULLT), e & 1, abort_flag, a.status)) return false;
            tc::fence_after();
            // Y = Xhi T_C^T, i.e. (T_C S)^T
#pragma unroll 1
            for (int ks = 0; ks < D / 8; ++ks)
                tc::mma_ts(tb + TM_Y, tb + TM_XHI + ks * 8, tc::sdesc_kstep(s_base + SM_T, D, ks),
                           tc::idesc_tf32(128, 128), ks > 0);
            tc::commit(bar(B_BODYDONE));
            return true;
        };
        // Gamma_w of entry e's seam (1 without seams); waits for the staging of
        // entry e, which runs ahead
        auto seam_scale = [&](int e, bool &okw) -> float {
            if (w == 0) return 1.f;
            bool wt = true;
            if (tid == 0) wt = wait_bar(bar(B_STAGED0 + (e & 1)), (e >> 1) & 1, abort_flag, a.status);
            okw = tc::bar_and(BAR_STATE, NS, wt);
            return reinterpret_cast<const float *>(sm + SM_BUF + (e & 1) * BUF_BYTES + BF_SMALL)[SMALL_GL];
        };
        // thread 0 keeps the pair rows of entries e + 1 and e + 2 in registers;
        // the request table lives in the constant bank, whose misses cost
        // thousands of cycles, so each lookup is issued an entry before its use
        int row1 = 0, row2 = 0, row3 = 0;
        if (tid == 0 && n_ent > 0) {
            load_T(pair_row(0));
            load_SC(pair_row(0));
            t_armed = sc_armed = 1;
            if (n_ent > 1) {
                row1 = pair_row(1);
                prefetch_pair(row1);
            }
            if (n_ent > 2) row2 = pair_row(2);
        }
        bool ok = true;
        // X = Gamma_w S_init^T (or 0), Xhi = tf32(S_init^T); S_prefix[0] = S_init
        {
            const float g0 = n_ent > 0 ? seam_scale(0, ok) : 1.f;
            for (int c0 = 64 * hf; ok && c0 < 64 * hf + 64; c0 += 32) {
                float xv[32], hv[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const float x = a.S_init ? a.S_init[st_base + (size_t)(c0 + q) * D + j] : 0.f;
                    xv[q] = g0 * x;
                    hv[q] = tc::round_tf32(x);
                    if (n_ent > 0 && a.S_prefix)
                        a.S_prefix[(((size_t)l * n_ent) * dm.H + h) * D * D + (size_t)(c0 + q) * D + j] = x;
                    if (n_ent == 0) a.S_final[st_base + (size_t)(c0 + q) * D + j] = x;
                }
                tc::tmem_st32_async(my + TM_X + c0, xv);
                tc::tmem_st32_async(my + TM_XHI + c0, hv);
            }
            tc::tmem_wait_st();
            tc::fence_before();
            tc::bar_sync(BAR_STATE, NS);
            if (tid == 0 && ok && n_ent > 0 && w > 0) issue_seam(0);
        }
        for (int e = 0; e < n_ent && ok; ++e) {
            const uint8_t *buf = sm + SM_BUF + (e & 1) * BUF_BYTES;
            if (tid == 0) {
                if (e + 2 < n_ent) prefetch_pair(row2);
                if (e + 3 < n_ent) row3 = pair_row(e + 3);
            }
            bool wt = true;
            if (w > 0) {
                // ---- seam outputs and the update operand W
                if (tid == 0) wt = wait_bar(bar(B_SEAMDONE), e & 1, abort_flag, a.status);
                if (!tc::bar_and(BAR_STATE, NS, wt)) { ok = false; break; }
                tc::fence_after();
                const float *smf = reinterpret_cast<const float *>(buf + BF_SMALL);
                const float *Vr = reinterpret_cast<const float *>(buf + BF_V);
                const int sw = reinterpret_cast<const int *>(smf)[SMALL_SW];
                float uz[2 * WMAX];
                {
                    float p0[32], p1[32];
                    tc::tmem_ld32x2(my + TM_D2, p0, p1);
#pragma unroll
                    for (int cc = 0; cc < 2 * WMAX; ++cc) uz[cc] = (p0[cc] + p0[16 + cc]) + (p1[cc] + p1[16 + cc]);
                }
                float U[WMAX];
#pragma unroll
                for (int t = 0; t < WMAX; ++t) {
                    float acc = 0.f;
#pragma unroll
                    for (int s = 0; s <= t; ++s)
                        acc = fmaf(smf[SMALL_M + t * WMAX + s], Vr[s * D + j] - smf[SMALL_G + s] * uz[s], acc);
                    U[t] = acc;
                }
                if (hf == 0) {
                    float wv[32];
#pragma unroll
                    for (int s = 0; s < WMAX; ++s) {
                        const float x = smf[SMALL_D + s] * U[s];
                        const float hi = tc::round_tf32(x);
                        wv[s] = hi;
                        wv[WMAX + s] = tc::round_tf32(x - hi);
                        wv[2 * WMAX + s] = hi;
                        wv[3 * WMAX + s] = 0.f;
                    }
                    tc::tmem_st32(my + TM_W, wv);
                    tc::fence_before();
                }
                tc::bar_sync(BAR_STATE, NS);
                if (tid == 0) {
                    tc::fence_after();
                    // X += W K: [Whi | Wlo | Whi] against K^T columns [hi | hi | lo]
                    const uint32_t bufa = s_base + SM_BUF + (e & 1) * BUF_BYTES;
#pragma unroll 1
                    for (int ks = 0; ks < 3; ++ks)
                        tc::mma_ts(tb + TM_X, tb + TM_W + ks * 8, tc::sdesc_kstep(bufa + BF_KP, D, ks),
                                   tc::idesc_tf32(128, 128), 1);
                    tc::commit(bar(B_UPDDONE));
                    tc::commit(bar(B_BUFFREE0 + (e & 1)));
                }
                if (hf == 1) {
                    // outputs while the update MMA runs
                    float *o_dst = a.o_out + (((size_t)l * n_ent + e) * w) * dm.H * D + (size_t)h * D + j;
#pragma unroll
                    for (int t = 0; t < WMAX; ++t) {
                        if (t < w) {
                            float o = smf[SMALL_G + t] * uz[WMAX + t];
#pragma unroll
                            for (int s = 0; s <= t; ++s) o = fmaf(smf[SMALL_AQ + t * WMAX + s], U[s], o);
                            o_dst[(size_t)t * dm.H * D] = (t < sw) ? o : 0.f;
                        }
                    }
                }
                // ---- Xhi of the state after the seam (operand of the body MMA)
                if (tid == 0) wt = wait_bar(bar(B_UPDDONE), e & 1, abort_flag, a.status);
                if (!tc::bar_and(BAR_STATE, NS, wt)) { ok = false; break; }
                tc::fence_after();
#pragma unroll
                for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 32) {
                    float xv[32];
                    tc::tmem_ld32(my + TM_X + c0, xv);
#pragma unroll
                    for (int q = 0; q < 32; ++q) xv[q] = tc::round_tf32(xv[q]);
                    tc::tmem_st32_async(my + TM_XHI + c0, xv);
                }
                tc::tmem_wait_st();
                tc::fence_before();
                tc::bar_sync(BAR_STATE, NS);
            }
            if (tid == 0) wt = issue_body(e);
            // ---- body: S = T_C S + S(C|0); X takes the next seam's Gamma_w
            const bool last = e + 1 == n_ent;
            const float gn = last ? 1.f : seam_scale(e + 1, ok);
            if (!ok) break;
            if (tid == 0 && wt) {
                wt = wait_bar(bar(B_BODYDONE), e & 1, abort_flag, a.status);
                if (wt) wt = wait_bar(bar(B_FULLSC), e & 1, abort_flag, a.status);
            }
            if (!tc::bar_and(BAR_STATE, NS, wt)) { ok = false; break; }
            tc::fence_after();
            if (tid == 0 && !last) {
                load_T(row1);  // T_C buffer free: the body MMA is done
                t_armed = e + 2;
            }
            float *out = last ? a.S_final + st_base
                              : (a.S_prefix ? a.S_prefix + (((size_t)l * n_ent + e + 1) * dm.H + h) * D * D : nullptr);
#pragma unroll
            for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 32) {
                float xv[32], hv[32];
                tc::tmem_ld32(my + TM_Y + c0, xv);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    xv[q] += *reinterpret_cast<const float *>(sm + SM_SC + tc::sw128_f32(c0 + q, j, D));
                    hv[q] = tc::round_tf32(xv[q]);
                }
                tc::tmem_st32_async(my + TM_XHI + c0, hv);
                if (out) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) out[(size_t)(c0 + q) * D + j] = xv[q];
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) xv[q] *= gn;
                tc::tmem_st32_async(my + TM_X + c0, xv);
            }
            tc::tmem_wait_st();
            tc::fence_before();
            tc::bar_sync(BAR_STATE, NS);
            if (tid == 0 && !last) {
                load_SC(row1);  // S(C|0) buffer consumed
                sc_armed = e + 2;
                if (w > 0) issue_seam(e + 1);
                row1 = row2;
                row2 = row3;
            }
        }
        if (!ok && tid == 0) {
            // aborted: let the copies in flight land before the CTA exits
            const long long t0 = clock64();
            while (((t_armed > 0 && !tc::mbar_test(bar(B_FULLT), (t_armed - 1) & 1)) ||
                    (sc_armed > 0 && !tc::mbar_test(bar(B_FULLSC), (sc_armed - 1) & 1))) &&
                   clock64() - t0 < kWaitCycles) {
            }
        }
    } else {
        // ================================================= staging warps
        const int c = tid - NS;  // channel
        const int gw = warp - NS / 32;
        constexpr int NL = CK > 0 ? CK : 1;
        float wq[NL], wk[NL], wvv[NL];
        if (CK > 0) {
            const float *w0 = a.tok.conv_w + (((size_t)l * 3 + 0) * dm.H + h) * D * CK + c * CK;
#pragma unroll
            for (int jj = 0; jj < NL; ++jj) {
                wq[jj] = __ldg(w0 + jj);
                wk[jj] = __ldg(w0 + (size_t)dm.H * D * CK + jj);
                wvv[jj] = __ldg(w0 + 2 * (size_t)dm.H * D * CK + jj);
            }
        }
        float *red = reinterpret_cast<float *>(sm + SM_RED);
        float *dots = red + RED_DOTS;
        float *scr = red + RED_SCR;
        // gates of entry e's seam tokens: threads 0-7 alpha_t (1 past the
        // segment), 8-15 beta_t (0 past the segment)
        auto gate = [&](const EntryInfo &ei) {
            float v = (c < WMAX) ? 1.f : 0.f;
            if (c < 2 * WMAX && (c & (WMAX - 1)) < ei.sw) {
                const size_t gi = gate_index(dm, a.tok.N, l, ei.off + (c & (WMAX - 1)), h);
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(c < WMAX ? a.tok.alpha : a.tok.beta);
                v = __bfloat162float(src[gi]);
            }
            return v;
        };
        // entries e (cur), e + 1 (nx1) and e + 2 (nx2) of the request table
        EntryInfo cur{0, 0, 0, 0}, nx1{0, 0, 0, 0}, nx2{0, 0, 0, 0};
        if (w > 0 && n_ent > 0) cur = entry_info(tab, 0, w, CK);
        if (w > 0 && n_ent > 1) nx1 = entry_info(tab, 1, w, CK);
        int raw_armed = 0;
        if (w > 0 && c == 0) {
            if (n_ent > 0) load_raw(0, cur);
            if (n_ent > 1) load_raw(1, nx1);
            raw_armed = min(2, n_ent);
        }
        float gab_next = (w > 0 && n_ent > 0) ? gate(cur) : 0.f;
        bool ok = true;
        for (int e = 0; w > 0 && e < n_ent && ok; ++e) {
            const int b = e & 1;
            uint8_t *buf = sm + SM_BUF + b * BUF_BYTES;
            const uint8_t *raw = sm + SM_RAW + b * 3 * RAW_T;
            const int sw = cur.sw;
            if (e + 2 < n_ent) nx2 = entry_info(tab, e + 2, w, CK);  // used after the conv
            const float gab = gab_next;
            gab_next = (e + 1 < n_ent) ? gate(nx1) : 0.f;  // in flight while this entry is staged
            bool wt = true;
            if (c == 0) {
                if (e >= 2) wt = wait_bar(bar(B_BUFFREE0 + b), ((e - 2) >> 1) & 1, abort_flag, a.status);
                if (wt) wt = wait_bar(bar(B_FULLR0 + b), (e >> 1) & 1, abort_flag, a.status);
            }
            if (!tc::bar_and(BAR_STAGE, NG, wt)) { ok = false; break; }
            // ---- conv (along the request stream) and L2 normalisation of q, k
            const bool htma = CK > 0 && cur.htma;
            auto raw_at = [&](int tensor, int row) {
                const uint16_t u = *reinterpret_cast<const uint16_t *>(raw + tensor * RAW_T + (row * D + c) * 2);
                return __uint_as_float(static_cast<uint32_t>(u) << 16);
            };
            float qv[WMAX], kv[WMAX], vv[WMAX];
#pragma unroll
            for (int t = 0; t < WMAX; ++t) {
                qv[t] = kv[t] = vv[t] = 0.f;
                if (t >= sw) continue;
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
                        const int32_t tbk = stream_back(tab, e, t, lag);
                        rq = rk = rv = 0.f;
                        if (tbk >= 0) {
                            const size_t ix = tok_index(dm, a.tok.N, l, tbk, h, c);
                            rq = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.tok.q)[ix]);
                            rk = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.tok.k)[ix]);
                            rv = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.tok.v)[ix]);
                        }
                    }
                    if (CK == 0) {
                        qv[t] = rq;
                        kv[t] = rk;
                        vv[t] = rv;
                    } else {
                        qv[t] = fmaf(wq[lag], rq, qv[t]);
                        kv[t] = fmaf(wk[lag], rk, kv[t]);
                        vv[t] = fmaf(wvv[lag], rv, vv[t]);
                    }
                }
            }
            if (CK > 0 && dm.act) {
#pragma unroll
                for (int t = 0; t < WMAX; ++t) {
                    qv[t] = silu(qv[t]);
                    kv[t] = silu(kv[t]);
                    vv[t] = silu(vv[t]);
                }
            }
            if (CK > 0) {
                float sq[WMAX], sk[WMAX];
#pragma unroll
                for (int t = 0; t < WMAX; ++t) {
                    sq[t] = qv[t] * qv[t];
                    sk[t] = kv[t] * kv[t];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int t = 0; t < WMAX; ++t) {
                        sq[t] += __shfl_xor_sync(0xffffffffu, sq[t], o);
                        sk[t] += __shfl_xor_sync(0xffffffffu, sk[t], o);
                    }
                if (lane == 0) {
#pragma unroll
                    for (int t = 0; t < WMAX; ++t) {
                        red[(gw * WMAX + t) * 2] = sq[t];
                        red[(gw * WMAX + t) * 2 + 1] = sk[t];
                    }
                }
                tc::bar_sync(BAR_STAGE, NG);
#pragma unroll
                for (int t = 0; t < WMAX; ++t) {
                    float aa = 0.f, bb = 0.f;
#pragma unroll
                    for (int ww = 0; ww < 4; ++ww) {
                        aa += red[(ww * WMAX + t) * 2];
                        bb += red[(ww * WMAX + t) * 2 + 1];
                    }
                    qv[t] *= rsqrtf(aa + kL2Eps);  // hardware reciprocal square root
                    kv[t] *= rsqrtf(bb + kL2Eps);
                }
            }
            // raw buffer b consumed: the rows of entry e + 2 may load into it
            tc::bar_sync(BAR_STAGE, NG);
            if (c == 0 && e + 2 < n_ent) {
                load_raw(e + 2, nx2);
                raw_armed = e + 3;
            }
            // ---- operand tiles: [k ; q] in tf32 and in fp32, K^T split hi / lo, V
#pragma unroll
            for (int t = 0; t < WMAX; ++t) {
                const float kh = tc::round_tf32(kv[t]), kl = tc::round_tf32(kv[t] - kh);
                *reinterpret_cast<float *>(buf + BF_KQH + tc::sw128_f32(t, c, 2 * WMAX)) = kh;
                *reinterpret_cast<float *>(buf + BF_KQH + tc::sw128_f32(WMAX + t, c, 2 * WMAX)) = tc::round_tf32(qv[t]);
                *reinterpret_cast<float *>(buf + BF_KQF + tc::sw128_f32(t, c, 2 * WMAX)) = kv[t];
                *reinterpret_cast<float *>(buf + BF_KQF + tc::sw128_f32(WMAX + t, c, 2 * WMAX)) = qv[t];
                *reinterpret_cast<float *>(buf + BF_KP + tc::sw128_f32(c, t, D)) = kh;
                *reinterpret_cast<float *>(buf + BF_KP + tc::sw128_f32(c, WMAX + t, D)) = kh;
                *reinterpret_cast<float *>(buf + BF_KP + tc::sw128_f32(c, 2 * WMAX + t, D)) = kl;
                reinterpret_cast<float *>(buf + BF_V)[t * D + c] = vv[t];
            }
            // ---- gates: g_t, Gamma_t, d_s = beta_s e^{g_w - g_s}
            float *smf = reinterpret_cast<float *>(buf + BF_SMALL);
            if (gw == 0) {
                // lanes 0-7 hold alpha_t, lanes 8-15 beta_t
                const float la = (lane < WMAX) ? fmaxf(logf(gab), -88.f) : 0.f;
                float g = la;
#pragma unroll
                for (int o = 1; o < WMAX; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, g, o);
                    if (lane >= o && lane < WMAX) g += y;
                }
                const float gw7 = __shfl_sync(0xffffffffu, g, WMAX - 1);
                const float be = __shfl_sync(0xffffffffu, gab, (lane & (WMAX - 1)) + WMAX);
                if (lane < WMAX) {
                    smf[SMALL_LG + lane] = g;
                    smf[SMALL_B + lane] = be;
                    smf[SMALL_G + lane] = expf(g);
                    smf[SMALL_D + lane] = be * expf(gw7 - g);
                    if (lane == 0) {
                        smf[SMALL_GL] = expf(gw7);
                        reinterpret_cast<int *>(smf)[SMALL_SW] = sw;
                    }
                }
            }
            tc::fence_async_smem();
            tc::bar_sync(BAR_STAGE, NG);
            // ---- the 64 dot products k_t.k_s (s < t), q_t.k_s (s <= t) (two threads each),
            // and the decays e^{g_t - g_s} (s <= t)
            {
                const int p = c >> 1, half = c & 1;
                int ra, rb, tt, ss;
                dot_rows(p, ra, rb, tt, ss);
                float acc = 0.f;
#pragma unroll 4
                for (int cc = 64 * half; cc < 64 * half + 64; cc += 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(buf + BF_KQF + tc::sw128_f32(ra, cc, 2 * WMAX));
                    const float4 bv = *reinterpret_cast<const float4 *>(buf + BF_KQF + tc::sw128_f32(rb, cc, 2 * WMAX));
                    acc = fmaf(av.x, bv.x, acc);
                    acc = fmaf(av.y, bv.y, acc);
                    acc = fmaf(av.z, bv.z, acc);
                    acc = fmaf(av.w, bv.w, acc);
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                if (half == 0) dots[p] = acc;
                if (c >= 64) {
                    const int t = (c - 64) >> 3, s2 = (c - 64) & 7;
                    scr[c - 64] = (s2 <= t) ? smf[SMALL_B + s2] * expf(smf[SMALL_LG + t] - smf[SMALL_LG + s2]) : 0.f;
                }
            }
            tc::bar_sync(BAR_STAGE, NG);
            // ---- AQ_ts = beta_s e^{g_t - g_s} q_t.k_s, L_ts = beta_s e^{g_t - g_s} k_t.k_s
            if (c < 64) {
                const int t = c >> 3, s2 = c & 7;
                const float be = scr[c];
                smf[SMALL_AQ + c] = (s2 <= t) ? be * dots[28 + t * (t + 1) / 2 + s2] : 0.f;
                scr[64 + c] = (s2 < t) ? be * dots[t * (t - 1) / 2 + s2] : 0.f;
            }
            tc::bar_sync(BAR_STAGE, NG);
            // ---- M = (I + L)^{-1}, one column per thread
            if (c < WMAX) {
                const float *Lm = scr + 64;
                float x[WMAX];
#pragma unroll
                for (int t = 0; t < WMAX; ++t) {
                    float acc = (t == c) ? 1.f : 0.f;
#pragma unroll
                    for (int r = 0; r < t; ++r) acc = fmaf(-Lm[t * WMAX + r], x[r], acc);
                    x[t] = (t < c) ? 0.f : acc;
                }
#pragma unroll
                for (int t = 0; t < WMAX; ++t) smf[SMALL_M + t * WMAX + c] = x[t];
            }
            tc::bar_sync(BAR_STAGE, NG);
            if (c == 0) tc::mbar_arrive(bar(B_STAGED0 + b));
            cur = nx1;
            nx1 = nx2;
        }
        if (!ok && c == 0 && raw_armed > 0) {
            const long long t0 = clock64();
            for (int k = (raw_armed > 2 ? raw_armed - 2 : 0); k < raw_armed; ++k)
                while (!tc::mbar_test(bar(B_FULLR0 + (k & 1)), (k >> 1) & 1) && clock64() - t0 < kWaitCycles) {
                }
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tb, TM_COLS);
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
