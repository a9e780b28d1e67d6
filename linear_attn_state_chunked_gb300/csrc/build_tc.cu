// build_tc.cu -- segment build of the gated-delta pair on the tcgen05 tensor
// cores, chunked in the WY form, for d_k = d_v = 128 and bf16 inputs.
//
// Math (derived from the recurrence S_t = alpha_t (I - beta_t k_t k_t^T)
// S_{t-1} + beta_t k_t v_t^T and the pair (T_C, S(C|0)) of section "线性层"
// of the article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token
// 延迟降低 3.25 倍，实现位置无关缓存”).  Within a chunk of C = 64 tokens let g_t = sum_{s<=t} log alpha_s,
// Gamma_t = exp(g_t).  Writing u_t = v_t - alpha_t S_{t-1}^T k_t, one finds
//   S_C = Gamma_C S_0 + K^T D U,   U = (I + L)^{-1} (V - diag(Gamma) K S_0),
//   L_tj = beta_j exp(g_t - g_j) k_t.k_j  (j < t),  D = diag(beta_j exp(g_C - g_j)).
// The same map advances T (with V replaced by 0), so X = [T | S] (d_k x 2d)
// is carried as one matrix.  Kept transposed in tensor memory (Xt = X^T,
// two 128-lane halves x 128 columns), one chunk is
//   Pt = Xt K^T                       (tf32 MMA, A = Xt from tensor memory)
//   Rt = [0 | V]^T - Pt diag(Gamma)   (CUDA cores, written back over Pt)
//   Xt = Gamma_C Xt + Rt U~           (tf32 MMA, A = Rt from tensor memory)
//   U~^T = K^T D (I + L)^{-1}         (Gram K K^T and U~ on the tensor core,
//                                      the 64 x 64 unit lower inverse by
//                                      doubling from 8 x 8 blocks: forward
//                                      substitution on CUDA cores, block
//                                      products on warp-level MMAs)
// Operands written by threads are rounded to tf32 (the tensor core
// truncates).
//
// Warp roles (one CTA per SM, persistent over work items):
//   warp 13     TMA producer: raw bf16 K/V rows (+ conv history) and gates of
//               each chunk into a 3-stage ring;
//   warp 12     one thread issues every tcgen05.mma: chunk n's Gram, Pt, U~
//               and Xt updates, each as soon as its inputs are ready;
//   warps 4-11  preparation of chunk n+1 while chunk n runs (two warps per
//               tensor-memory lane quadrant): gates, conv + normalisation,
//               tf32 K, L, the inverse, U~;
//   warps 0-3   epilogue of chunk n: Rt and the Gamma_C rescale of Xt, both
//               halves, and the emission of each finished pair.
// Work items (segment body, layer, head) arrive longest body first; CTA b
// takes items b, b + grid, ... -- the greedy LPT order of that article's "段并行"
// section as a single-GPU stand-in for its scatter workers.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace hypic {
namespace {

constexpr int D = 128;   // head width
constexpr int C = 64;    // chunk length
constexpr int RS = 2;    // raw-input ring stages
constexpr int HMAX = 3;  // conv history rows kept per chunk (conv_k <= 4)
constexpr int ROWS = C + HMAX;
constexpr int NP = 256;  // preparation threads (warps 4-11, two per tensor-memory lane quadrant)
constexpr int NT = 448;  // 14 warps
constexpr int WARP_MMA = 12, WARP_TMA = 13;
constexpr int BAR_EPI = 1, BAR_PREP = 2;
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds

// tensor-memory columns
constexpr uint32_t TM_XT = 0;    // Xt, T half: 128 lanes x 128
constexpr uint32_t TM_XS = 128;  // Xt, S half
constexpr uint32_t TM_PT = 256;  // Pt then Rt, T half: 128 x 64
constexpr uint32_t TM_PS = 320;  // Pt then Rt, S half
constexpr uint32_t TM_G = 384;   // Gram (M = 64 layout), then K^T (A of U~): 64 columns
constexpr uint32_t TM_U = 448;   // U~^T: 128 x 64
constexpr uint32_t TM_COLS = 512;

// raw stage: K rows, V rows (bf16 [ROWS][128]), alpha[64], beta[64] (fp32)
constexpr uint32_t ST_K = 0;
constexpr uint32_t ST_V = ROWS * D * 2;
constexpr uint32_t ST_G = 2 * ROWS * D * 2;  // the chunk's Gates, written by the producer warp
constexpr uint32_t ST_BYTES = ST_G + 5 * C * 4;

// shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t SM_RAW = 0;
constexpr uint32_t SM_K32 = (RS * ST_BYTES + 1023) / 1024 * 1024;  // K [64][128] tf32, sw128
constexpr uint32_t SM_UT = SM_K32 + 32768;     // U~^T [128][64] tf32, sw128 (B of the Xt update)
constexpr uint32_t SM_MT = SM_UT + 32768;      // (D M)^T [64][64] tf32, sw128 (B of U~)
constexpr int LP = C + 4;                      // row pitch of L and M: 16-byte rows for ldmatrix
constexpr uint32_t SM_L = SM_MT + 16384;       // L [64][68], tf32 values
constexpr uint32_t SM_M = SM_L + C * LP * 4;   // M = (I + L)^-1 [64][68], tf32 values
constexpr int QP = 36;                         // row pitch of the per-warp Q^T scratch
constexpr uint32_t SM_Q = SM_M + C * LP * 4;   // per-warp Q^T [8][36] for the inverse
constexpr uint32_t SM_WK = SM_Q + 8 * 8 * QP * 4;  // K conv weights of the current item [4 lags][128]
constexpr uint32_t SM_BAR = SM_WK + D * 4 * 4;
constexpr uint32_t SM_MISC = SM_BAR + 32 * 8;
constexpr uint32_t SM_BYTES = SM_MISC + 64;
constexpr uint32_t SMEM_DYN = SM_BYTES + 1024;
static_assert(SM_K32 % 1024 == 0 && SM_UT % 1024 == 0 && SM_MT % 1024 == 0, "tile alignment");
static_assert(SM_L % 16 == 0 && SM_M % 16 == 0 && SM_Q % 16 == 0, "ldmatrix row alignment");
static_assert(ST_BYTES % 128 == 0 && ST_V % 128 == 0, "TMA destination alignment");
static_assert(SMEM_DYN <= 232448, "shared memory budget");

struct Gates {
    float g[C];   // inclusive log-gate sums
    float eg[C];  // exp(g_t)
    float dc[C];  // beta_j exp(g_C - g_j)
    float b[C];   // beta
    float fb[C];  // beta_j exp(g_m - g_j), g_m = (g_0 + g_C) / 2
};

// mbarriers
enum {
    B_FULL = 0,          // [RS] raw stage loaded (TMA bytes + producer arrive)
    B_EMPTY = RS,        // [RS] raw stage released (prep + epilogue)
    B_KREADY = 2 * RS,   // K32 written                      prep -> mma
    B_GRAM,              // Gram done                        mma -> prep
    B_KTREADY,           // K^T in TMEM and (D M)^T written   prep -> mma
    B_UDONE,             // U~ done                          mma -> prep
    B_UTREADY,           // U~^T copied to smem               prep -> mma
    B_PTDONE,            // Pt (T half) done                 mma -> epilogue
    B_PSDONE,            // Pt (S half) done                 mma -> epilogue, prep (K32 free)
    B_RTREADY,           // Rt (T half) written, Xt_T scaled  epilogue -> mma
    B_RSREADY,           // Rt (S half) written, Xt_S scaled  epilogue -> mma
    B_DSDONE,            // both Xt updates done              mma -> epilogue, prep (U~^T free)
    B_XREADY,            // Xt initialised for a new item     epilogue -> mma
    B_COUNT
};

struct Item {
    int s, l, h;
    int32_t seg0, b0, n;  // segment start, body start, body length
    int nch;              // chunks
};

__device__ __forceinline__ Item decode_item(int item, const Dims &dm, const SegTable &tab)
{
    Item it;
    const int LH = dm.L * dm.H;
    it.s = tab.perm[item / LH];
    const int lh = item % LH;
    it.l = lh / dm.H;
    it.h = lh % dm.H;
    it.seg0 = tab.off[it.s];
    const int32_t seg1 = tab.off[it.s + 1];
    it.b0 = it.seg0 + min(dm.w, seg1 - it.seg0);
    it.n = seg1 - it.b0;
    it.nch = (it.n + C - 1) / C;
    return it;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ void unpack8(const uint4 &u, float *x)
{
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}
__device__ __forceinline__ float bf16_at(const uint8_t *tile, int row, int col)
{
    const uint16_t u = *reinterpret_cast<const uint16_t *>(tile + (row * D + col) * 2);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// Bounded wait by one thread; any failure (or another role's) aborts the CTA.
__device__ __forceinline__ bool wait_bar(uint32_t mbar, uint32_t parity, volatile int *abort_flag)
{
    return tc::wait_bounded(mbar, parity, abort_flag, kWaitCycles);
}

// Warp-level tf32 MMA, 16 x 8 x 8, accumulate into c.
__device__ __forceinline__ void mma16x8x8(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Warp-level tf32 MMA operands straight from shared memory (ldmatrix of 8 x 4
// fp32 tiles: lane 4g + t receives element (g, t) of each tile).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}

// Row-major fp32 matrix with pitch LP floats: A fragment of the 16 x 8 tile at (r0, k0).
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], uint32_t base, int r0, int k0, int lane)
{
    const int row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8, col = k0 + (lane >> 4) * 4;
    ldsm_x4(a, base + (row * LP + col) * 4);
}

// B fragment (k0 .. k0+8) x (n0 .. n0+8) of a matrix stored transposed in the
// 64 x 64 sw128 tile at base (row n holds column n of the matrix).
__device__ __forceinline__ void frag_b_sw(uint32_t (&b)[2], uint32_t base, int k0, int n0, int lane)
{
    ldsm_x2(b, base + tc::sw128_f32(n0 + (lane & 7), k0 + ((lane >> 3) & 1) * 4, C));
}

// B fragment of the per-warp Q^T scratch (pitch QP): rows k0 .. k0+8 of Q.
__device__ __forceinline__ void frag_b_q(uint32_t (&b)[2], uint32_t qt, int k0, int lane)
{
    ldsm_x2(b, qt + ((lane & 7) * QP + k0 + ((lane >> 3) & 1) * 4) * 4);
}

// Store a 16 x 8 accumulator fragment (rows r0.., columns c0..) as tf32 values,
// negated, into M (row-major) and M^T (sw128 tile).
__device__ __forceinline__ void store_m(float *Ms, uint8_t *Mt, int r0, int c0, const float (&c)[4], int lane)
{
    const int g = lane >> 2, t4 = lane & 3;
    const float v0 = tc::round_tf32(-c[0]), v1 = tc::round_tf32(-c[1]);
    const float v2 = tc::round_tf32(-c[2]), v3 = tc::round_tf32(-c[3]);
    *reinterpret_cast<float2 *>(Ms + (r0 + g) * LP + c0 + 2 * t4) = make_float2(v0, v1);
    *reinterpret_cast<float2 *>(Ms + (r0 + g + 8) * LP + c0 + 2 * t4) = make_float2(v2, v3);
    *reinterpret_cast<float *>(Mt + tc::sw128_f32(c0 + 2 * t4, r0 + g, C)) = v0;
    *reinterpret_cast<float *>(Mt + tc::sw128_f32(c0 + 2 * t4 + 1, r0 + g, C)) = v1;
    *reinterpret_cast<float *>(Mt + tc::sw128_f32(c0 + 2 * t4, r0 + g + 8, C)) = v2;
    *reinterpret_cast<float *>(Mt + tc::sw128_f32(c0 + 2 * t4 + 1, r0 + g + 8, C)) = v3;
}

// Store a 16 x 8 accumulator fragment as tf32 values into rows r0.. of the Q^T scratch.
__device__ __forceinline__ void store_q(float *Qt, int r0, const float (&c)[4], int lane)
{
    const int g = lane >> 2, t4 = lane & 3;
    Qt[(2 * t4) * QP + r0 + g] = tc::round_tf32(c[0]);
    Qt[(2 * t4 + 1) * QP + r0 + g] = tc::round_tf32(c[1]);
    Qt[(2 * t4) * QP + r0 + g + 8] = tc::round_tf32(c[2]);
    Qt[(2 * t4 + 1) * QP + r0 + g + 8] = tc::round_tf32(c[3]);
}

// M = (I + L)^{-1} for the unit lower triangular 64 x 64 matrix I + L, by
// doubling: with I + L = [[A, 0], [B, E]] in equal halves,
//   M = [[A^{-1}, 0], [-E^{-1} B A^{-1}, E^{-1}]],
// applied from 8 x 8 diagonal blocks (forward substitution) up to 16, 32
// and 64.  The 8 -> 16 step runs on CUDA cores inside each of four warps;
// the 16 -> 32 and 32 -> 64 products on the warp-level tensor-core MMA
// (tf32 operands, fp32 accumulation).  L holds tf32 values; M is written as
// tf32 values twice, row-major (Ms, A operands) and transposed into the
// sw128 tile Mt (B operands, and later (D M)^T in place).  Only the lower
// blocks are written: the strictly upper 8 x 8 blocks stay zero from the
// start of the kernel.  pt = 0 .. NP-1.
__device__ __noinline__ void unit_lower_inverse(const float *Ls, float *Ms, uint8_t *Mt, float *Qs, int pt)
{
    const int wq = pt >> 5, ln = pt & 31;
    float *Qt = Qs + wq * 8 * QP;  // this warp's Q^T
    const uint32_t sL = tc::smem_u32(Ls), sM = tc::smem_u32(Ms), sMt = tc::smem_u32(Mt), sQ = tc::smem_u32(Qt);
    if (wq < 4) {
        // 16 x 16 diagonal block wq: its two 8 x 8 diagonal blocks (one column per lane) ...
        const int B = 16 * wq;
        if (ln < 16) {
            const int base = B + 8 * (ln >> 3), cc = ln & 7;
            float x[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < r; ++j) acc = fmaf(-Ls[(base + r) * LP + base + j], x[j], acc);
                x[r] = (r < cc) ? 0.f : tc::round_tf32(acc);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) Ms[(base + r) * LP + base + cc] = x[r];
            *reinterpret_cast<float4 *>(Mt + tc::sw128_f32(base + cc, base, C)) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4 *>(Mt + tc::sw128_f32(base + cc, base + 4, C)) = make_float4(x[4], x[5], x[6], x[7]);
        }
        __syncwarp();
        // ... then its lower-left 8 x 8: -M_bb (L_ba M_aa), two entries per lane
        float q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = (ln >> 3) + 4 * h, j = ln & 7;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc = fmaf(Ls[(B + 8 + i) * LP + B + k], Ms[(B + k) * LP + B + j], acc);
            q[h] = acc;
        }
        Qt[ln] = q[0];
        Qt[ln + 32] = q[1];
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = (ln >> 3) + 4 * h, j = ln & 7;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc = fmaf(Ms[(B + 8 + i) * LP + B + 8 + k], Qt[k * 8 + j], acc);
            const float v = tc::round_tf32(-acc);
            Ms[(B + 8 + i) * LP + B + j] = v;
            *reinterpret_cast<float *>(Mt + tc::sw128_f32(B + j, B + 8 + i, C)) = v;
        }
    }
    tc::bar_sync(BAR_PREP, NP);
    if (wq < 4) {
        // 16 -> 32: M_10 and M_32 (16 x 16), one 8-column half per warp
        const int bj = 2 * (wq >> 1), bi = bj + 1, c0 = 16 * bj + 8 * (wq & 1);
        float q[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], b[2];
        // M_jj[k][c0..] vanishes for the first k-step when c0 is the upper half
        if ((wq & 1) == 0) {
            frag_a(a, sL, 16 * bi, 16 * bj, ln);
            frag_b_sw(b, sMt, 16 * bj, c0, ln);
            mma16x8x8(q, a, b);
        }
        frag_a(a, sL, 16 * bi, 16 * bj + 8, ln);
        frag_b_sw(b, sMt, 16 * bj + 8, c0, ln);
        mma16x8x8(q, a, b);
        store_q(Qt, 0, q, ln);
        __syncwarp();
        float r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            frag_a(a, sM, 16 * bi, 16 * bi + 8 * ks, ln);
            frag_b_q(b, sQ, 8 * ks, ln);
            mma16x8x8(r, a, b);
        }
        store_m(Ms, Mt, 16 * bi, c0, r, ln);
    }
    tc::bar_sync(BAR_PREP, NP);
    {
        // 32 -> 64: rows 32..63 x columns 0..31; warp wq takes row block
        // 32 + 16 rb and the 8-column strip cs.  Q = L[32.., 0..32) M[0..32, strip]
        // (M[k][strip] = 0 for k < 8 cs), then -M[rows, 32..64) Q.
        const int rb = wq >> 2, cs = wq & 3, c0 = 8 * cs;
        float q0[4] = {0.f, 0.f, 0.f, 0.f}, q1[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], b[2];
        for (int ks = cs; ks < 4; ++ks) {
            frag_b_sw(b, sMt, 8 * ks, c0, ln);
            frag_a(a, sL, 32, 8 * ks, ln);
            mma16x8x8(q0, a, b);
            if (rb) {
                frag_a(a, sL, 48, 8 * ks, ln);
                mma16x8x8(q1, a, b);
            }
        }
        store_q(Qt, 0, q0, ln);
        if (rb) store_q(Qt, 16, q1, ln);
        __syncwarp();
        float r[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ks = 0; ks < 2 * (rb + 1); ++ks) {
            frag_a(a, sM, 32 + 16 * rb, 32 + 8 * ks, ln);
            frag_b_q(b, sQ, 8 * ks, ln);
            mma16x8x8(r, a, b);
        }
        store_m(Ms, Mt, 32 + 16 * rb, c0, r, ln);
    }
    tc::bar_sync(BAR_PREP, NP);
}

// Cursor over this CTA's chunks (non-empty items only), used by the MMA issuer.
struct Cursor {
    int item;  // global item index (blockIdx.x + k * gridDim.x)
    int c;     // chunk within the item
    int nch;
    int n;     // CTA-wide chunk number
    int xi;    // index of the item among this CTA's non-empty items
    Item it;   // the item, decoded once
};

__device__ __forceinline__ void cursor_seek(Cursor &cu, int n_items, const Dims &dm, const SegTable &tab)
{
    while (cu.item < n_items) {
        cu.it = decode_item(cu.item, dm, tab);
        if (cu.it.nch > 0) {
            cu.nch = cu.it.nch;
            return;
        }
        cu.item += gridDim.x;
    }
}

__device__ __forceinline__ void cursor_next(Cursor &cu, int n_items, const Dims &dm, const SegTable &tab)
{
    ++cu.n;
    if (++cu.c == cu.nch) {
        cu.c = 0;
        ++cu.xi;
        cu.item += gridDim.x;
        cursor_seek(cu, n_items, dm, tab);
    }
}

// The three K32-operand MMA groups of a chunk (issued by one thread).
__device__ __forceinline__ void issue_gram(uint32_t tb, uint32_t sK32)
{
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks)
        tc::mma_ss(tb + TM_G, tc::sdesc_kstep(sK32, C, ks), tc::sdesc_kstep(sK32, C, ks), tc::idesc_tf32(64, 64),
                   ks > 0);
}
__device__ __forceinline__ void issue_pt(uint32_t tb, uint32_t sK32)
{
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks)
        tc::mma_ts(tb + TM_PT, tb + TM_XT + ks * 8, tc::sdesc_kstep(sK32, C, ks), tc::idesc_tf32(128, 64), ks > 0);
}
__device__ __forceinline__ void issue_ps(uint32_t tb, uint32_t sK32)
{
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks)
        tc::mma_ts(tb + TM_PS, tb + TM_XS + ks * 8, tc::sdesc_kstep(sK32, C, ks), tc::idesc_tf32(128, 64), ks > 0);
}

template <int CK, bool ACT>
__global__ void __launch_bounds__(NT, 1)
build_tc_kernel(const __grid_constant__ BuildArgs a, const __grid_constant__ SegTable tab,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV)
{
    constexpr int HIST = CK > 0 ? CK - 1 : 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = tc::smem_u32(sm);
    const uint32_t sK32 = s_base + SM_K32, sUT = s_base + SM_UT, sMT = s_base + SM_MT;
    auto bar = [&](int i) { return s_base + SM_BAR + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM_MISC);
    uint32_t *tmem_base_sh = reinterpret_cast<uint32_t *>(sm + SM_MISC + 16);
    float *Ls = reinterpret_cast<float *>(sm + SM_L);
    float *Ms = reinterpret_cast<float *>(sm + SM_M);
    float *Qs = reinterpret_cast<float *>(sm + SM_Q);
    uint8_t *Mt = sm + SM_MT;  // M^T during the inverse, then (D M)^T in place

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Dims dm = a.dm;
    const int32_t N = a.tok.N;
    const int n_items = tab.n_seg * dm.L * dm.H;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i >= B_EMPTY && i < B_EMPTY + RS) cnt = 2;
            tc::mbar_init(bar(i), cnt);
        }
        tc::fence_mbar_init();
    }
    for (int i = tid; i < C * LP; i += NT) Ms[i] = 0.f;  // the upper blocks of M stay zero
    for (int i = tid; i < C * C; i += NT) reinterpret_cast<float *>(Mt)[i] = 0.f;
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_base_sh), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = *tmem_base_sh;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t my = tb + lane_off;  // this thread's lane (quadrant of its warp), column 0

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ producer
        const __nv_bfloat16 *ap = static_cast<const __nv_bfloat16 *>(a.tok.alpha);
        const __nv_bfloat16 *bp = static_cast<const __nv_bfloat16 *>(a.tok.beta);
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            for (int c = 0; c < it.nch; ++c) {
                const int s = n % RS, use = n / RS;
                if (use > 0) {
                    bool w = true;
                    if (lane == 0) w = wait_bar(bar(B_EMPTY + s), (use - 1) & 1, abort_flag);
                    if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                }
                uint8_t *stg = sm + SM_RAW + s * ST_BYTES;
                const int32_t t0 = c * C;
                const int nc = min(C, (int)(it.n - t0));
                {
                    // gates of tokens 2 lane, 2 lane + 1 (padding: alpha = 1, beta = 0)
                    float al[2] = {1.f, 1.f}, be[2] = {0.f, 0.f};
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int tt = 2 * lane + u;
                        if (tt < nc) {
                            const size_t gi = gate_index(dm, N, it.l, it.b0 + t0 + tt, it.h);
                            al[u] = __bfloat162float(ap[gi]);
                            be[u] = __bfloat162float(bp[gi]);
                        }
                    }
                    Gates &G = *reinterpret_cast<Gates *>(stg + ST_G);
                    const float x0 = fmaxf(logf(al[0]), -88.f);  // alpha = 0 -> exp(-88)
                    const float x1 = fmaxf(logf(al[1]), -88.f);
                    float sum = x0 + x1;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, sum, o);
                        if (lane >= o) sum += y;
                    }
                    const float total = __shfl_sync(0xffffffffu, sum, 31);
                    const float g1 = sum, g0 = sum - x1;
                    G.g[2 * lane] = g0;
                    G.g[2 * lane + 1] = g1;
                    G.eg[2 * lane] = expf(g0);
                    G.eg[2 * lane + 1] = expf(g1);
                    G.b[2 * lane] = be[0];
                    G.b[2 * lane + 1] = be[1];
                    G.dc[2 * lane] = be[0] * expf(total - g0);
                    G.dc[2 * lane + 1] = be[1] * expf(total - g1);
                    const float gm = 0.5f * (__shfl_sync(0xffffffffu, x0, 0) + total);
                    G.fb[2 * lane] = be[0] * __expf(fmaxf(gm - g0, -87.f));
                    G.fb[2 * lane + 1] = be[1] * __expf(fmaxf(gm - g1, -87.f));
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t fb = bar(B_FULL + s);
                    tc::mbar_arrive_expect_tx(fb, 2u * (C + HIST) * D * 2);
                    const int row0 = it.b0 + t0 - HIST;
                    tc::tma_load_4d(s_base + SM_RAW + s * ST_BYTES + ST_K, &tmK, 0, it.h, row0, it.l, fb);
                    tc::tma_load_4d(s_base + SM_RAW + s * ST_BYTES + ST_V, &tmV, 0, it.h, row0, it.l, fb);
                }
                ++n;
            }
        }
        if (!ok && lane == 0) {
            // aborted: let the copies this warp started land before the CTA exits
            for (int k = (n > RS ? n - RS : 0); k < n; ++k) {
                const long long t0 = clock64();
                while (!tc::mbar_test(bar(B_FULL + k % RS), (k / RS) & 1) && clock64() - t0 < kWaitCycles) {
                }
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        // Issue order: Gram(0), Pt(0); then per chunk n: U~(n), Gram(n+1),
        // Xt_T update (n), Xt_S update (n), Pt(n+1) -- each as soon as its
        // inputs are ready (hardware-suspended bounded waits).  Gram(n+1)
        // runs ahead of chunk n's Xt updates so that the preparation warps
        // find it done; tcgen05.mma from one thread execute in issue order, so
        // a later MMA never overwrites tensor memory that an earlier one reads.
        if (lane == 0) {
            Cursor mc{static_cast<int>(blockIdx.x), 0, 0, 0, 0, {}};
            cursor_seek(mc, n_items, dm, tab);
            bool go = mc.item < n_items;
            if (go) {
                go = wait_bar(bar(B_KREADY), 0, abort_flag) && wait_bar(bar(B_XREADY), 0, abort_flag);
                tc::fence_after();
                if (go) {
                    issue_gram(tb, sK32);
                    tc::commit(bar(B_GRAM));
                    issue_pt(tb, sK32);
                    tc::commit(bar(B_PTDONE));
                    issue_ps(tb, sK32);
                    tc::commit(bar(B_PSDONE));
                }
            }
            while (go && mc.item < n_items) {
                const uint32_t par = mc.n & 1;
                if (!wait_bar(bar(B_KTREADY), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ts(tb + TM_U, tb + TM_G + ks * 8, tc::sdesc_kstep(sMT, C, ks),
                               tc::idesc_tf32(128, 64), ks > 0);
                tc::commit(bar(B_UDONE));
                Cursor nx = mc;
                cursor_next(nx, n_items, dm, tab);
                const bool more = nx.item < n_items;
                if (more) {
                    if (!wait_bar(bar(B_KREADY), par ^ 1u, abort_flag)) break;
                    tc::fence_after();
                    issue_gram(tb, sK32);
                    tc::commit(bar(B_GRAM));
                }
                if (!wait_bar(bar(B_UTREADY), par, abort_flag)) break;
                if (!wait_bar(bar(B_RTREADY), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ts(tb + TM_XT, tb + TM_PT + ks * 8, tc::sdesc_kstep(sUT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
                if (!wait_bar(bar(B_RSREADY), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ts(tb + TM_XS, tb + TM_PS + ks * 8, tc::sdesc_kstep(sUT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
                tc::commit(bar(B_DSDONE));
                if (more) {
                    if (nx.c == 0 && !wait_bar(bar(B_XREADY), nx.xi & 1, abort_flag)) break;
                    tc::fence_after();
                    issue_pt(tb, sK32);
                    tc::commit(bar(B_PTDONE));
                    issue_ps(tb, sK32);
                    tc::commit(bar(B_PSDONE));
                }
                mc = nx;
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ preparation
        // Step k: finish chunk k-1 up to its U~ operands (L, inverse, K^T,
        // (D M)^T), convert chunk k (gates, conv + normalisation, tf32 K)
        // while U~(k-1) runs, then copy U~(k-1)^T to shared memory.
        const int pt = tid - 128;      // 0 .. NP-1
        const int li = pt & 127;       // tensor-memory lane of this thread
        const int hh = pt >> 7;        // which half of a 64-column operand this warp handles
        const int c0 = (pt & 15) * 8;  // the 8 channels this thread converts ...
        const int r0 = 4 * (pt >> 4);  // ... in chunk rows r0 .. r0+3
        int wk_item = -1;  // item whose conv weights are in shared memory
        Cursor cv{static_cast<int>(blockIdx.x), 0, 0, 0, 0, {}};
        cursor_seek(cv, n_items, dm, tab);
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const bool conv_k = cv.item < n_items;  // chunk k exists
            if (k > 0) {
                // ---- chunk m = k-1: L from the Gram rows (M = 64 layout: row 16q + i in lane 32q + i)
                const int m = k - 1;
                const Gates &G = *reinterpret_cast<const Gates *>(sm + SM_RAW + (m % RS) * ST_BYTES + ST_G);
                bool w = true;
                if (pt == 0) w = wait_bar(bar(B_GRAM), m & 1, abort_flag);
                if (!tc::bar_and(BAR_PREP, NP, w)) { ok = false; break; }
                tc::fence_after();
                {
                    // Gram row 16q + i sits in lane 32q + i (i < 16) of quadrant q; this
                    // warp takes columns 32hh .. 32hh+31 of its 16 rows, lanes 16-31
                    // the upper 16 of those (shuffled from their partner lane).
                    float gr[32];
                    tc::tmem_ld32(my + TM_G + hh * 32, gr);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float o = __shfl_up_sync(0xffffffffu, gr[16 + j], 16);
                        if (lane >= 16) gr[j] = o;
                    }
                    const int t = 16 * (warp & 3) + (lane & 15);
                    const int j0 = hh * 32 + ((lane >= 16) ? 16 : 0);
                    const float gt_t = G.g[t];
                    if (G.g[0] - G.g[C - 1] < 80.f) {
                        // exp(g_t - g_j) = exp(g_t - g_m) exp(g_m - g_j), g_m the chunk midpoint:
                        // both factors stay within e^{+-40}, one exp per row
                        const float gm = 0.5f * (G.g[0] + G.g[C - 1]);
                        const float et = __expf(gt_t - gm);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            gr[j] = (j0 + j < t) ? tc::round_tf32(G.fb[j0 + j] * et * gr[j]) : 0.f;
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            gr[j] = (j0 + j < t) ? tc::round_tf32(G.b[j0 + j] * __expf(gt_t - G.g[j0 + j]) * gr[j]) : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4 *>(Ls + t * LP + j0 + j) = make_float4(gr[j], gr[j + 1], gr[j + 2], gr[j + 3]);
                }
                tc::bar_sync(BAR_PREP, NP);
                unit_lower_inverse(Ls, Ms, Mt, Qs, pt);
                // K^T into tensor memory (A of U~): lane i holds K[j][i], this warp j = 32hh .. +31
                {
                    float kt[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        kt[j] = *reinterpret_cast<const float *>(sm + SM_K32 + tc::sw128_f32(hh * 32 + j, li, C));
                    tc::tmem_st32(my + TM_G + hh * 32, kt);
                }
                // B of U~: element (t, j) = dc_j M[j][t], scaled in place in the M^T tile
#pragma unroll
                for (int e = pt; e < C * C / 4; e += NP) {
                    const int t = e & (C - 1), j = (e >> 6) * 4;
                    float4 *p = reinterpret_cast<float4 *>(Mt + tc::sw128_f32(t, j, C));
                    const float4 mv = *p;
                    *p = make_float4(tc::round_tf32(G.dc[j] * mv.x), tc::round_tf32(G.dc[j + 1] * mv.y),
                                     tc::round_tf32(G.dc[j + 2] * mv.z), tc::round_tf32(G.dc[j + 3] * mv.w));
                }
                tc::fence_async_smem();
                tc::fence_before();
                tc::bar_sync(BAR_PREP, NP);
                if (pt == 0) {
                    tc::mbar_arrive(bar(B_KTREADY));
                    tc::mbar_arrive(bar(B_EMPTY + m % RS));  // K rows and gates consumed
                }
            }
            if (conv_k) {
                // ---- chunk k: gates and K -> tf32 (conv + L2 normalisation first when present)
                const Item &it = cv.it;
                if (CK > 0 && cv.item != wk_item) {
                    // visible to all preparation threads after the barrier below
                    const float *wk = a.tok.conv_w + (((size_t)it.l * 3 + 1) * dm.H + it.h) * D * CK;
                    if (pt < D) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(wk + pt * CK);
                        float *ws = reinterpret_cast<float *>(sm + SM_WK);
                        ws[pt] = w4.x;
                        ws[D + pt] = w4.y;
                        ws[2 * D + pt] = w4.z;
                        ws[3 * D + pt] = w4.w;
                    }
                    wk_item = cv.item;
                }
                const int s = k % RS;
                const uint8_t *stg = sm + SM_RAW + s * ST_BYTES;
                const int nc = min(C, (int)(it.n - cv.c * C));
                bool w = true;
                if (pt == 0) w = wait_bar(bar(B_FULL + s), (k / RS) & 1, abort_flag);
                if (pt == 32 && k > 0) w = wait_bar(bar(B_PSDONE), (k - 1) & 1, abort_flag);  // K32 free
                if (!tc::bar_and(BAR_PREP, NP, w)) { ok = false; break; }
                {
                    // rows r0 .. r0+3 use staged rows r0 .. r0+3+HIST (row t + HIST - j is lag j)
                    uint4 raw[4 + HIST];
#pragma unroll
                    for (int i = 0; i < 4 + HIST; ++i)
                        raw[i] = *reinterpret_cast<const uint4 *>(stg + ST_K + ((r0 + i) * D + c0) * 2);
                    float kx[4][8];
                    if (CK == 0) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) unpack8(raw[r], kx[r]);
                    } else {
#pragma unroll
                        for (int r = 0; r < 4; ++r)
#pragma unroll
                            for (int i = 0; i < 8; ++i) kx[r][i] = 0.f;
#pragma unroll
                        for (int j = 0; j < (CK > 0 ? CK : 1); ++j) {
                            // lag-j weights of channels c0 .. c0+7
                            const float4 wa = *reinterpret_cast<const float4 *>(sm + SM_WK + (j * D + c0) * 4);
                            const float4 wb = *reinterpret_cast<const float4 *>(sm + SM_WK + (j * D + c0 + 4) * 4);
                            const float wj[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                float rk[8];
                                unpack8(raw[r + HIST - j], rk);
#pragma unroll
                                for (int i = 0; i < 8; ++i) kx[r][i] = fmaf(wj[i], rk[i], kx[r][i]);
                            }
                        }
                        if (ACT) {
#pragma unroll
                            for (int r = 0; r < 4; ++r)
#pragma unroll
                                for (int i = 0; i < 8; ++i) kx[r][i] = silu(kx[r][i]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        if (r0 + r >= nc) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) kx[r][i] = 0.f;
                        }
                    }
                    if (CK > 0) {
                        float ss[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            ss[r] = 0.f;
#pragma unroll
                            for (int i = 0; i < 8; ++i) ss[r] = fmaf(kx[r][i], kx[r][i], ss[r]);
                        }
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                            for (int r = 0; r < 4; ++r) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], o);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float inv = rsqrtf(ss[r] + kL2Eps);  // hardware reciprocal square root
#pragma unroll
                            for (int i = 0; i < 8; ++i) kx[r][i] *= inv;
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        *reinterpret_cast<float4 *>(sm + SM_K32 + tc::sw128_f32(r0 + r, c0, C)) =
                            make_float4(tc::round_tf32(kx[r][0]), tc::round_tf32(kx[r][1]),
                                        tc::round_tf32(kx[r][2]), tc::round_tf32(kx[r][3]));
                        *reinterpret_cast<float4 *>(sm + SM_K32 + tc::sw128_f32(r0 + r, c0 + 4, C)) =
                            make_float4(tc::round_tf32(kx[r][4]), tc::round_tf32(kx[r][5]),
                                        tc::round_tf32(kx[r][6]), tc::round_tf32(kx[r][7]));
                    }
                }
                tc::fence_async_smem();
                tc::bar_sync(BAR_PREP, NP);
                if (pt == 0) tc::mbar_arrive(bar(B_KREADY));
                cursor_next(cv, n_items, dm, tab);
            }
            if (k > 0) {
                // ---- chunk m = k-1: U~^T rows into shared memory once the previous Xt update is done
                const int m = k - 1;
                bool w = true;
                if (pt == 0) w = wait_bar(bar(B_UDONE), m & 1, abort_flag);
                if (pt == 32 && m > 0) w = wait_bar(bar(B_DSDONE), (m - 1) & 1, abort_flag);
                if (!tc::bar_and(BAR_PREP, NP, w)) { ok = false; break; }
                tc::fence_after();
                {
                    float u[32];
                    tc::tmem_ld32(my + TM_U + hh * 32, u);
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(sm + SM_UT + tc::sw128_f32(li, hh * 32 + i, D)) =
                            make_float4(tc::round_tf32(u[i]), tc::round_tf32(u[i + 1]), tc::round_tf32(u[i + 2]),
                                        tc::round_tf32(u[i + 3]));
                }
                tc::fence_async_smem();
                tc::fence_before();
                tc::bar_sync(BAR_PREP, NP);
                if (pt == 0) tc::mbar_arrive(bar(B_UTREADY));
            }
            if (!conv_k) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-3)
        const int m = tid;  // row of Xt / Pt in each half = tensor-memory lane
        float wvr[CK > 0 ? CK : 1];
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            const size_t pair = ((size_t)it.l * tab.n_seg + it.s) * dm.H + it.h;
            float *To = a.T_out + pair * D * D + m;
            float *So = a.S_out + pair * D * D + m;
            if (it.nch == 0) {
                for (int i = 0; i < D; ++i) {
                    To[(size_t)i * D] = (i == m) ? 1.f : 0.f;
                    So[(size_t)i * D] = 0.f;
                }
                continue;
            }
            if (CK > 0) {
                const float *wv = a.tok.conv_w + (((size_t)it.l * 3 + 2) * dm.H + it.h) * D * CK;
#pragma unroll
                for (int j = 0; j < (CK > 0 ? CK : 1); ++j) wvr[j] = __ldg(wv + m * CK + j);
            }
            // Xt = [I | 0]^T
            {
                float v[32];
#pragma unroll
                for (int c = 0; c < D; c += 32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (c + i == m) ? 1.f : 0.f;
                    tc::tmem_st32(my + TM_XT + c, v);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll
                for (int c = 0; c < D; c += 32) tc::tmem_st32(my + TM_XS + c, v);
            }
            tc::fence_before();
            tc::bar_sync(BAR_EPI, 128);
            if (m == 0) tc::mbar_arrive(bar(B_XREADY));
            for (int c = 0; c < it.nch; ++c, ++n) {
                const int s = n % RS;
                const uint8_t *stg = sm + SM_RAW + s * ST_BYTES;
                const Gates &G = *reinterpret_cast<const Gates *>(stg + ST_G);
                const int nc = min(C, (int)(it.n - c * C));
                // ---- T half
                bool w = true;
                if (m == 0) w = wait_bar(bar(B_PTDONE), n & 1, abort_flag);
                if (!tc::bar_and(BAR_EPI, 128, w)) { ok = false; break; }
                tc::fence_after();
                const float gC = G.eg[C - 1];
                {
                    float p[32];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        tc::tmem_ld32(my + TM_PT + h2 * 32, p);
#pragma unroll
                        for (int i = 0; i < 32; ++i) p[i] = tc::round_tf32(-G.eg[h2 * 32 + i] * p[i]);
                        tc::tmem_st32(my + TM_PT + h2 * 32, p);
                    }
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        tc::tmem_ld32(my + TM_XT + cc, p);
#pragma unroll
                        for (int i = 0; i < 32; ++i) p[i] *= gC;
                        tc::tmem_st32(my + TM_XT + cc, p);
                    }
                }
                tc::fence_before();
                tc::bar_sync(BAR_EPI, 128);
                if (m == 0) tc::mbar_arrive(bar(B_RTREADY));
                // ---- S half
                if (m == 0) {
                    w = wait_bar(bar(B_PSDONE), n & 1, abort_flag);
                    if (w) w = wait_bar(bar(B_FULL + s), (n / RS) & 1, abort_flag);
                }
                if (!tc::bar_and(BAR_EPI, 128, w)) { ok = false; break; }
                tc::fence_after();
                {
                    float p[32];
                    // raw V history window for the conv: win[j] = row t + HIST - j
                    float win[HMAX + 1];
#pragma unroll
                    for (int j = 1; j <= HMAX; ++j) win[j] = (j <= HIST) ? bf16_at(stg + ST_V, HIST - j, m) : 0.f;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        tc::tmem_ld32(my + TM_PS + h2 * 32, p);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int t = h2 * 32 + i;
                            win[0] = bf16_at(stg + ST_V, t + HIST, m);
                            float vv = 0.f;
                            if (CK == 0) {
                                vv = win[0];
                            } else {
#pragma unroll
                                for (int j = 0; j < (CK > 0 ? CK : 1); ++j) vv = fmaf(wvr[j], win[j], vv);
                                if (ACT) vv = silu(vv);
                            }
                            if (t >= nc) vv = 0.f;
                            p[i] = tc::round_tf32(fmaf(-G.eg[t], p[i], vv));
#pragma unroll
                            for (int j = HMAX; j > 0; --j) win[j] = win[j - 1];
                        }
                        tc::tmem_st32(my + TM_PS + h2 * 32, p);
                    }
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        tc::tmem_ld32(my + TM_XS + cc, p);
#pragma unroll
                        for (int i = 0; i < 32; ++i) p[i] *= gC;
                        tc::tmem_st32(my + TM_XS + cc, p);
                    }
                }
                tc::fence_before();
                tc::bar_sync(BAR_EPI, 128);
                if (m == 0) {
                    tc::mbar_arrive(bar(B_RSREADY));
                    tc::mbar_arrive(bar(B_EMPTY + s));  // V rows consumed
                }
            }
            if (!ok) break;
            // ---- emit the finished pair: T[i][m] = Xt_T[m][i], S[i][m] = Xt_S[m][i]
            bool w = true;
            if (m == 0) w = wait_bar(bar(B_DSDONE), (n - 1) & 1, abort_flag);
            if (!tc::bar_and(BAR_EPI, 128, w)) { ok = false; break; }
            tc::fence_after();
            {
                float x[32];
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    tc::tmem_ld32(my + TM_XT + cc, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) To[(size_t)(cc + i) * D] = x[i];
                    tc::tmem_ld32(my + TM_XS + cc, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) So[(size_t)(cc + i) * D] = x[i];
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0 && *abort_flag) atomicOr(a.status, 1);
    if (warp == 0) tc::tmem_dealloc(tb, TM_COLS);
}

int g_num_sms = 0;

cudaError_t make_token_map(CUtensorMap *map, const void *base, const Dims &dm, int32_t N, int rows)
{
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)dm.H, (cuuint64_t)N, (cuuint64_t)dm.L};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)dm.H * D * 2, (cuuint64_t)N * dm.H * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)D, 1u, (cuuint32_t)rows, 1u};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

bool build_tc_supported(const Dims &dm)
{
    return dm.mode == HYPIC_GATED_DELTA && dm.dtype == HYPIC_BF16 && dm.D == 128 &&
           (dm.conv_k == 0 || dm.conv_k == 4);
}

cudaError_t launch_build_tc(const BuildArgs &a, const SegTable &tab, cudaStream_t st)
{
    const int n_items = tab.n_seg * a.dm.L * a.dm.H;
    if (n_items == 0) return cudaSuccess;
    cudaError_t e;
    if (g_num_sms == 0) {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    }
    const int rows = C + (a.dm.conv_k > 0 ? a.dm.conv_k - 1 : 0);
    CUtensorMap tmK, tmV;
    if ((e = make_token_map(&tmK, a.tok.k, a.dm, a.tok.N, rows)) != cudaSuccess) return e;
    if ((e = make_token_map(&tmV, a.tok.v, a.dm, a.tok.N, rows)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(int), st)) != cudaSuccess) return e;
    const int grid = n_items < g_num_sms ? n_items : g_num_sms;
    // the activation after the conv is a template flag: no cost when off
    auto kern = a.dm.conv_k == 0 ? build_tc_kernel<0, false>
                                 : (a.dm.act ? build_tc_kernel<4, true> : build_tc_kernel<4, false>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN))) return e;
    kern<<<grid, NT, SMEM_DYN, st>>>(a, tab, tmK, tmV);
    return cudaGetLastError();
}

}  // namespace hypic
