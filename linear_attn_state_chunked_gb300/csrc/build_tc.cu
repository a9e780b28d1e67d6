// build_tc.cu -- segment build of the gated-delta pair on the tcgen05 tensor
// cores, chunked in the WY form, for d_k = d_v = 128 and bf16 inputs.
//
// Math (derived from the recurrence S_t = alpha_t (I - beta_t k_t k_t^T)
// S_{t-1} + beta_t k_t v_t^T and the pair (T_C, S(C|0)) of section "线性层"
// of the article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token
// 延迟降低 3.25 倍，实现位置无关缓存”).  Within a chunk of C = 64 tokens let
// g_t = sum_{s<=t} log alpha_s, Gamma_t = exp(g_t), Gamma_C = Gamma_{C-1},
//   L_tj = beta_j exp(g_t - g_j) k_t.k_j  (j < t),  D = diag(beta_j exp(g_C - g_j)).
// Writing u_t = v_t - alpha_t S_{t-1}^T k_t one finds that X = [T | S]
// (d_k x 2d, T from I and S from 0) advances per chunk as
//   X <- Gamma_C X + U~^T R,   R = [0 | V] - diag(Gamma) K X,
//   U~ = (I + L)^{-T} D K      (C x d_k).
// The decays drop out of the triangular system: entry by entry
// L^T D = D L''^T with L''_tj = beta_t k_t.k_j (j < t), so
// (I + L)^T D = D (I + L'')^T and
//   U~ = D W^T K ,   W = (I + L'')^{-1}  (unit lower triangular, no exponentials).
// W is built by doubling: the eight 8 x 8 diagonal blocks by forward
// substitution, then the block rule
//   [[A, 0], [B, C]]^{-1} = [[A^-1, 0], [-C^-1 B A^-1, C^-1]]
// at 16, 32 and 64 tokens with warp-level fp16 MMAs (W and L'' are O(1): fp16 keeps
// the tf32 mantissa).  In 16-token blocks
//   U~_i = D_i sum_{j >= i} W_ji^T K_j ,
// ten independent block products per 32-channel slice of U~.
//
// Kernel form: X is kept transposed in tensor memory (Xt = X^T, two 128-lane
// halves: Xt_T = T^T and Xt_S = S^T).  Per chunk
//   Pt   = Xt K^T                         tcgen05 tf32, A = Xt from tensor memory
//   Rt_S = V^T - Pt_S diag(Gamma),   Xt_S <- Gamma_C Xt_S      (CUDA cores)
//   Rt_T = -Pt_T diag(Gamma / Gamma_C)    (Xt_T was multiplied by Gamma_C when
//                                          the previous chunk finished)
//   Xt  += Rt U~                          tcgen05 tf32, A = Rt from tensor memory
// The tensor core reads an fp32 A operand truncated to tf32.  For the T half
// that truncation would bias the product chunk after chunk, so the part it
// drops, Xt_T - trunc(Xt_T), is kept beside Xt_T in bf16 and multiplied by K
// in bf16 into the same accumulator: Pt_T is then exact to ~2^-19.
// Operands written by threads are rounded to nearest tf32.
//
// Warp roles (one CTA per SM, persistent over work items (segment body,
// layer, head); every role walks the same items and chunks in order):
//   warp 17      TMA producer: lane 0 streams raw bf16 K rows (+ conv history)
//                into a 3-stage ring, lane 1 raw V rows into a 2-stage ring;
//   warp 16      one thread issues every tcgen05.mma of chunk n: Pt_S, Pt_T
//                (+ its bf16 correction), the Gram of chunk n+1, the Xt_T and
//                Xt_S updates, each behind a bounded mbarrier wait;
//   warps 8-11   conversion: causal conv + L2 normalisation of K, rounded to
//                tf32 and stored in fp16 (double-buffered; fp16 holds those
//                values exactly: operand of the fp16 Gram and of the solve),
//                copied to bf16 (in place in the raw ring stage, operand of
//                the correction) and, once the previous Pt_T is done, to tf32
//                (single buffer, operand of Pt);
//   warps 12-15  solve: L'' from the Gram, W = (I + L'')^{-1}, and U~ = D W^T K
//                into the 128-byte-swizzled B operand of the Xt update;
//   warps 0-7    epilogue, each pass split over two warps per lane quadrant:
//                Rt_S (conv of V in registers, done before Pt_S is ready) and
//                the Gamma_C rescale of Xt_S; Rt_T; after the update Xt_T
//                scaled by the next chunk's Gamma_C and its bf16 low part;
//                emits T and S;
//   warp 18      gates: the chunk's cumulative log-gates, decays and beta
//                factors from alpha and beta (loaded a chunk ahead).
// Work items arrive longest body first; CTA b takes items b, b + grid, ... --
// the greedy LPT order of that article's "段并行" section as a single-GPU
// stand-in for its scatter workers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace hypic {
namespace {

constexpr int D = 128;   // head width
constexpr int C = 64;    // chunk length
constexpr int NB = 16;   // block of the back substitution
constexpr int RK = 2;    // raw-K ring stages
constexpr int RV = 2;    // raw-V ring stages
constexpr int RG = 4;    // gate ring stages
constexpr int HMAX = 3;  // conv history rows kept per chunk (conv_k <= 4)
constexpr int NT = 608;  // 19 warps
constexpr int WARP_MMA = 16, WARP_TMA = 17, WARP_GATE = 18;
constexpr int BAR_EPI = 1, BAR_CONV = 3, BAR_SOLVE = 4;
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds
// Largest log-decay span g_0 - g_{C-1} of a chunk for which Xt_T is
// pre-multiplied by Gamma_C (the factors Gamma_t / Gamma_C stay below e^80).
constexpr float kSpan = 80.f;

// tensor-memory columns
constexpr uint32_t TM_XT = 0;     // Xt_T: 128 lanes x 128
constexpr uint32_t TM_XS = 128;   // Xt_S
constexpr uint32_t TM_PT = 256;   // Pt_T, then Rt_T: 128 x 64
constexpr uint32_t TM_PS = 320;   // Pt_S, then Rt_S
constexpr uint32_t TM_G = 384;    // Gram (M = 64 layout): 64 columns
constexpr uint32_t TM_XLO = 448;  // Xt_T - trunc(Xt_T) in bf16 pairs: 64 columns
constexpr uint32_t TM_COLS = 512;

// shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t KR_STAGE = 17408;  // raw K rows [C + 3][128] bf16
constexpr uint32_t VR_STAGE = 17152;  // raw V rows [C + 3][128] bf16
constexpr uint32_t G_STAGE = 1296;    // Gates
constexpr int ZP = C + 8;             // row pitch (halves) of Z and the solve tiles: 16-byte, conflict-free ldmatrix rows
constexpr int TP2 = 24;               // row pitch (halves) of the 16 x 16 solve tiles
constexpr uint32_t SM_KR = 0;
constexpr uint32_t SM_VR = SM_KR + RK * KR_STAGE;
constexpr uint32_t SM_GATE = SM_VR + RV * VR_STAGE;
constexpr uint32_t SM_K32 = (SM_GATE + RG * G_STAGE + 1023) / 1024 * 1024;  // K [64][128] tf32, sw128 (B of Pt)
constexpr uint32_t SM_KH = SM_K32 + 32768;      // 2 x K [64][128] fp16, token-major sw128 (Gram, U~)
constexpr uint32_t SM_KB = SM_KH + 2 * 16384;   // 2 x K [64][128] bf16, token-major sw128 (Pt_T correction)
constexpr uint32_t SM_UT = SM_KB + 2 * 16384;   // U~^T [128][64] tf32, sw128 (B of the Xt update)
constexpr uint32_t SM_L = SM_UT + 32768;        // Z [64][ZP] fp16: L'' below the diagonal, W^T on and above
constexpr uint32_t SM_TMP = SM_L + C * ZP * 2;  // solve scratch: 4 x G^T [8][8] fp32, then 4 x [16][TP2] fp16
constexpr uint32_t SM_WK = SM_TMP + 4 * 64 * 4 + 4 * 16 * TP2 * 2;  // K conv weights of the current item [4 lags][128]
constexpr uint32_t SM_BAR = SM_WK + D * 4 * 4;
constexpr uint32_t SM_MISC = SM_BAR + 40 * 8;
constexpr uint32_t SM_BYTES = SM_MISC + 64;
constexpr uint32_t SMEM_DYN = SM_BYTES + 1024;
static_assert(KR_STAGE % 1024 == 0 && SM_K32 % 1024 == 0 && SM_KH % 1024 == 0 && SM_KB % 1024 == 0 &&
                  SM_UT % 1024 == 0, "tile alignment");
static_assert((C + HMAX) * D * 2 <= (int)KR_STAGE && (C + HMAX) * D * 2 <= (int)VR_STAGE, "ring stage size");
static_assert(SM_VR % 128 == 0 && VR_STAGE % 128 == 0, "TMA destination alignment");
static_assert(SM_L % 16 == 0 && SM_TMP % 16 == 0 && (ZP * 2) % 16 == 0 && (TP2 * 2) % 16 == 0,
              "ldmatrix row alignment");
static_assert(SMEM_DYN <= 232448, "shared memory budget");

struct Gates {
    float eg[C];  // exp(g_t), g_t the inclusive log-gate sum
    float dc[C];  // beta_j exp(g_C - g_j)
    float b[C];   // beta
    float nrc[C]; // -exp(g_t - g_C) (used when the chunk is pre-scaled)
    float neg[C]; // -exp(g_t)
    int safe;     // g_0 - g_C <= kSpan
};
static_assert(sizeof(Gates) <= G_STAGE, "gate stage size");

// mbarriers
enum {
    B_KRF = 0,            // [RK] raw K stage loaded                    TMA -> conversion
    B_KRE = B_KRF + RK,   // [RK] stage free (raw rows converted)       conversion -> TMA
    B_VRF = B_KRE + RK,   // [RV] raw V stage loaded                    TMA -> S epilogue
    B_VRE = B_VRF + RV,   // [RV] stage free                            S epilogue -> TMA
    B_GF = B_VRE + RV,    // [RG] gates written                         conversion -> solve, epilogues
    B_GE = B_GF + RG,     // [RG] gates consumed (2 arrivals)           solve, epilogue -> gates
    B_KRDY = B_GE + RG,   // [2] K tf32 + bf16 written                  conversion -> MMA
    B_KHE = B_KRDY + 2,   // [2] K fp16 and bf16 free (2 arrivals)      MMA, solve -> conversion
    B_K32E = B_KHE + 2,   // K tf32 free (Pt_T done)                    MMA -> conversion
    B_K32R,               // K tf32 written                             conversion -> MMA
    B_GRAMF,              // Gram done                                  MMA -> solve
    B_GRAME,              // Gram read into L                           solve -> MMA
    B_UTF,                // U~^T written                               solve -> MMA
    B_UTE,                // U~^T consumed (Xt_S update done)           MMA -> solve
    B_PTF,                // Pt_T done                                  MMA -> T epilogue
    B_RTF,                // Rt_T written                               T epilogue -> MMA
    B_PSF,                // Pt_S done                                  MMA -> S epilogue
    B_RSF,                // Rt_S written, Xt_S rescaled                S epilogue -> MMA
    B_XTD,                // Xt_T update done                           MMA -> T epilogue
    B_XTR,                // Xt_T (+ low part) ready for Pt_T           T epilogue -> MMA
    B_XSD,                // Xt_S update done                           MMA -> S epilogue
    B_XSI,                // Xt_S zeroed for a new item                 S epilogue -> MMA
    B_FIN,                // every MMA of the CTA completed             MMA -> MMA
    B_COUNT
};
static_assert(B_COUNT <= 40, "barrier space");

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
__device__ __forceinline__ float bf16_at(const uint8_t *tile, int row, int col)
{
    const uint16_t u = *reinterpret_cast<const uint16_t *>(tile + (row * D + col) * 2);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}
// Two floats as bf16 (round to nearest even), the first in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// Two floats as fp16 (round to nearest even), the first in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi)
{
    const __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// Bounded wait by one thread; any failure (or another role's) aborts the CTA.
__device__ __forceinline__ bool wait_bar(uint32_t mbar, uint32_t parity, volatile int *abort_flag)
{
    return tc::wait_bounded(mbar, parity, abort_flag, kWaitCycles);
}

// ldmatrix of four / two 8 x 8 16-bit tiles (optionally transposed).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}

// Warp-level fp16 MMA, 16 x 8 x 16, fp32 accumulate into c.
__device__ __forceinline__ void mma16x8x16_f16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// m16n8k16 operand fragments from row-major fp16 tiles in shared memory (base:
// address of the tile's first element, pitch in halves):
//   frag_a16  A (16 x 16) stored row-major;
//   frag_b16t B (16 x 8) stored transposed (row n holds column n of B);
//   frag_b16  B (16 x 8) stored row-major (row k), read by transposing ldmatrix.
__device__ __forceinline__ void frag_a16(uint32_t (&a)[4], uint32_t base, int pitch, int lane)
{
    ldsm_x4(a, base + (((lane & 7) + ((lane >> 3) & 1) * 8) * pitch + (lane >> 4) * 8) * 2);
}
__device__ __forceinline__ void frag_b16t(uint32_t (&b)[2], uint32_t base, int pitch, int lane)
{
    ldsm_x2(b, base + ((lane & 7) * pitch + ((lane >> 3) & 1) * 8) * 2);
}
__device__ __forceinline__ void frag_b16(uint32_t (&b)[2], uint32_t base, int pitch, int lane)
{
    ldsm_x2_t(b, base + ((lane & 7) + ((lane >> 3) & 1) * 8) * pitch * 2);
}

// Cursor over this CTA's chunks (non-empty items only), used by the MMA issuer.
struct Cursor {
    int item;  // global item index (blockIdx.x + k * gridDim.x)
    int c;     // chunk within the item
    int nch;
    int n;     // CTA-wide chunk number
    int xi;    // index of the item among this CTA's non-empty items
    Item it;
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

// Gram K K^T (M = N = 64 tokens) from the fp16 K tile: 16 channels per MMA.
// fp16 holds the tf32-rounded K exactly (same 10-bit mantissa; |k| <= 1).
__device__ __forceinline__ void issue_gram(uint32_t tb, uint32_t sKH)
{
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
        tc::mma_ss_f16(tb + TM_G, tc::sdesc_kstep(sKH, C, ks), tc::sdesc_kstep(sKH, C, ks), tc::idesc_f16(64, 64),
                       ks > 0);
}

// Xt_T <- s Xt_T and its truncated-away low part in bf16, columns c0 .. c0+63
// of this thread's lane.
__device__ __forceinline__ void scale_split_xt(uint32_t my, int c0, float s)
{
    const float2 s2 = make_float2(s, s), m1 = make_float2(-1.f, -1.f);
#pragma unroll 1
    for (int cc = c0; cc < c0 + 64; cc += 32) {
        float x[32];
        uint32_t lo[16];
        tc::tmem_ld32(my + TM_XT + cc, x);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 v = __fmul2_rn(s2, make_float2(x[2 * i], x[2 * i + 1]));
            const float2 h = make_float2(__uint_as_float(__float_as_uint(v.x) & 0xffffe000u),
                                         __uint_as_float(__float_as_uint(v.y) & 0xffffe000u));
            const float2 l = __ffma2_rn(h, m1, v);  // v - h, exact
            lo[i] = pack_bf16(l.x, l.y);
            x[2 * i] = v.x;
            x[2 * i + 1] = v.y;
        }
        tc::tmem_st32_async(my + TM_XT + cc, x);
        tc::tmem_st16_async(my + TM_XLO + cc / 2, lo);
        tc::tmem_wait_st();
    }
}

// 64 consecutive columns of this thread's lane scaled by s.
__device__ __forceinline__ void scale_cols(uint32_t taddr, float s)
{
    const float2 s2 = make_float2(s, s);
#pragma unroll 1
    for (int cc = 0; cc < 64; cc += 32) {
        float x[32];
        tc::tmem_ld32(taddr + cc, x);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 v = __fmul2_rn(s2, make_float2(x[2 * i], x[2 * i + 1]));
            x[2 * i] = v.x;
            x[2 * i + 1] = v.y;
        }
        tc::tmem_st32(taddr + cc, x);
    }
}

template <int CK, bool ACT>
__global__ void __launch_bounds__(NT, 1)
build_tc_kernel(const __grid_constant__ BuildArgs a, const __grid_constant__ SegTable tab,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV)
{
    constexpr int HIST = CK > 0 ? CK - 1 : 0;
    extern __shared__ uint8_t smem_raw[];
    // the 1024-aligned base, derived from the shared array itself so that every
    // access through it stays a shared-memory access
    const uint32_t raw_u32 = tc::smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
    const uint32_t s_base = tc::smem_u32(sm);
    auto bar = [&](int i) { return s_base + SM_BAR + 8u * i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + SM_MISC);
    uint32_t *tmem_base_sh = reinterpret_cast<uint32_t *>(sm + SM_MISC + 16);
    auto gates = [&](int n) -> const Gates & {
        return *reinterpret_cast<const Gates *>(sm + SM_GATE + (n % RG) * G_STAGE);
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Dims dm = a.dm;
    const int32_t N = a.tok.N;
    const int n_items = tab.n_seg * dm.L * dm.H;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i >= B_GE && i < B_GE + RG) cnt = 2;
            if (i >= B_KHE && i < B_KHE + 2) cnt = 2;
            tc::mbar_init(bar(i), cnt);
        }
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_base_sh), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = *tmem_base_sh;
    const uint32_t my = tb + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // this warp's lane quadrant

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ producer
        // lane 0: raw K ring, lane 1: raw V ring (independent loops)
        if (lane < 2) {
            const bool kside = lane == 0;
            const int R = kside ? RK : RV;
            const int bfull = kside ? B_KRF : B_VRF, bempty = kside ? B_KRE : B_VRE;
            const uint32_t dst0 = s_base + (kside ? SM_KR : SM_VR);
            const uint32_t stage = kside ? KR_STAGE : VR_STAGE;
            const CUtensorMap *map = kside ? &tmK : &tmV;
            int n = 0;
            bool ok = true;
            for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
                const Item it = decode_item(itx, dm, tab);
                for (int c = 0; c < it.nch; ++c, ++n) {
                    const int s = n % R, use = n / R;
                    if (use > 0 && !wait_bar(bar(bempty + s), (use - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(bar(bfull + s), (C + HIST) * D * 2);
                    tc::tma_load_4d(dst0 + s * stage, map, 0, it.h, it.b0 + c * C - HIST, it.l, bar(bfull + s));
                }
            }
            if (!ok) {
                // aborted: let the copies this lane started land before the CTA exits
                for (int k = (n > R ? n - R : 0); k < n; ++k) {
                    const long long t0 = clock64();
                    while (!tc::mbar_test(bar(bfull + k % R), (k / R) & 1) && clock64() - t0 < kWaitCycles) {
                    }
                }
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        // Per chunk n: Pt_S(n), Pt_T(n) and its bf16 correction, Gram(n+1),
        // Xt_T update(n), Xt_S update(n).  tcgen05.mma from one thread execute
        // in issue order, so a later MMA never overwrites tensor memory that
        // an earlier one still reads.
        if (lane == 0) {
            Cursor mc{static_cast<int>(blockIdx.x), 0, 0, 0, 0, {}};
            cursor_seek(mc, n_items, dm, tab);
            bool ok = true;
            if (mc.item < n_items) {
                ok = wait_bar(bar(B_KRDY), 0, abort_flag);
                tc::fence_after();
                if (ok) {
                    issue_gram(tb, s_base + SM_KH);
                    tc::commit(bar(B_GRAMF));
                }
            }
            while (ok && mc.item < n_items) {
                const int n = mc.n;
                const uint32_t par = n & 1;
                const uint32_t sK = s_base + SM_K32;
                const uint32_t sK16 = s_base + SM_KB + (n & 1) * 16384;
                if (mc.c == 0 && !wait_bar(bar(B_XSI), mc.xi & 1, abort_flag)) break;
                if (!wait_bar(bar(B_K32R), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_ts(tb + TM_PS, tb + TM_XS + ks * 8, tc::sdesc_kstep(sK, C, ks), tc::idesc_tf32(128, 64),
                               ks > 0);
                tc::commit(bar(B_PSF));
                if (!wait_bar(bar(B_XTR), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_ts(tb + TM_PT, tb + TM_XT + ks * 8, tc::sdesc_kstep(sK, C, ks), tc::idesc_tf32(128, 64),
                               ks > 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ts_bf16(tb + TM_PT, tb + TM_XLO + ks * 8, tc::sdesc_kstep(sK16, C, ks),
                                    tc::idesc_bf16(128, 64), 1);
                tc::commit(bar(B_PTF));
                tc::commit(bar(B_K32E));
                tc::commit(bar(B_KHE + (n & 1)));  // its Gram and Pt_T have read K in fp16 and bf16
                Cursor nx = mc;
                cursor_next(nx, n_items, dm, tab);
                if (nx.item < n_items) {
                    const int n1 = n + 1;
                    if (!wait_bar(bar(B_KRDY + (n1 & 1)), (n1 >> 1) & 1, abort_flag)) break;
                    if (!wait_bar(bar(B_GRAME), par, abort_flag)) break;
                    tc::fence_after();
                    issue_gram(tb, s_base + SM_KH + (n1 & 1) * 16384);
                    tc::commit(bar(B_GRAMF));
                }
                if (!wait_bar(bar(B_UTF), par, abort_flag)) break;
                if (!wait_bar(bar(B_RTF), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ts(tb + TM_XT, tb + TM_PT + ks * 8, tc::sdesc_kstep(s_base + SM_UT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
                tc::commit(bar(B_XTD));
                if (!wait_bar(bar(B_RSF), par, abort_flag)) break;
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ts(tb + TM_XS, tb + TM_PS + ks * 8, tc::sdesc_kstep(s_base + SM_UT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
                tc::commit(bar(B_XSD));
                tc::commit(bar(B_UTE));
                mc = nx;
            }
            // every MMA issued must complete before tensor memory is released
            tc::commit(bar(B_FIN));
            const long long t0 = clock64();
            while (!tc::mbar_test(bar(B_FIN), 0) && clock64() - t0 < kWaitCycles) {
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ conversion
        const int ct = tid - 256;       // 0 .. 127
        const int c0 = lane * 4;        // the 4 channels this thread converts ...
        const int r0 = 16 * (warp - 8); // ... in chunk rows r0 .. r0+15 (one warp per 16 rows)
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            if (it.nch == 0) continue;
            if (CK > 0) {
                // K conv weights of this item (the previous chunk's readers
                // passed the group barrier that ends it); read after the
                // barrier below
                const float *wk = a.tok.conv_w + (((size_t)it.l * 3 + 1) * dm.H + it.h) * D * CK;
                const float4 w4 = *reinterpret_cast<const float4 *>(wk + ct * CK);
                float *ws = reinterpret_cast<float *>(sm + SM_WK);
                ws[ct] = w4.x;
                ws[D + ct] = w4.y;
                ws[2 * D + ct] = w4.z;
                ws[3 * D + ct] = w4.w;
            }
            for (int c = 0; c < it.nch && ok; ++c, ++n) {
                const int nc = min(C, (int)(it.n - c * C));
                bool w = true;
                if (ct == 0) w = wait_bar(bar(B_KRF + n % RK), (n / RK) & 1, abort_flag);
                if (ct == 32 && n >= 2) w = wait_bar(bar(B_KHE + (n & 1)), ((n >> 1) - 1) & 1, abort_flag);
                if (!tc::bar_and(BAR_CONV, 128, w)) { ok = false; break; }
                uint8_t *stg = sm + SM_KR + (n % RK) * KR_STAGE;
                uint8_t *kh = sm + SM_KH + (n & 1) * 16384;
                uint8_t *kb = sm + SM_KB + (n & 1) * 16384;
                // byte offset of channels c0 .. c0+3 of row `row` in a 16-bit token-major sw128 tile
                auto o16 = [&](int row) {
                    return (c0 >> 6) * 8192 + row * 128 + ((((c0 & 63) >> 3) ^ (row & 7)) << 4) + (c0 & 7) * 2;
                };
                // K conv weights of this thread's four channels (lag j, channel pairs)
                float2 w2[CK > 0 ? CK : 1][2];
#pragma unroll
                for (int j = 0; j < (CK > 0 ? CK : 1); ++j) {
                    const float4 wa = *reinterpret_cast<const float4 *>(sm + SM_WK + (j * D + c0) * 4);
                    w2[j][0] = make_float2(wa.x, wa.y);
                    w2[j][1] = make_float2(wa.z, wa.w);
                }
#pragma unroll 1
                for (int hf = 0; hf < 4; ++hf) {
                    const int rb = r0 + 4 * hf;
                    // rows rb .. rb+3 from staged rows rb .. rb+3+HIST (staged row t + HIST - j is
                    // lag j of row t); channel pairs (c0, c0 + 1), (c0 + 2, c0 + 3) packed
                    float2 kx[4][2];
                    if (CK == 0) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint2 u = *reinterpret_cast<const uint2 *>(stg + ((rb + r) * D + c0) * 2);
                            kx[r][0] = make_float2(bf16_lo(u.x), bf16_hi(u.x));
                            kx[r][1] = make_float2(bf16_lo(u.y), bf16_hi(u.y));
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 4; ++r) kx[r][0] = kx[r][1] = make_float2(0.f, 0.f);
                        // each staged row is unpacked once and feeds every output row that uses it
#pragma unroll
                        for (int i = 0; i < 4 + HIST; ++i) {
                            const uint2 u = *reinterpret_cast<const uint2 *>(stg + ((rb + i) * D + c0) * 2);
                            const float2 x0 = make_float2(bf16_lo(u.x), bf16_hi(u.x));
                            const float2 x1 = make_float2(bf16_lo(u.y), bf16_hi(u.y));
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const int j = r + HIST - i;
                                if (j >= 0 && j < CK) {
                                    kx[r][0] = __ffma2_rn(w2[j][0], x0, kx[r][0]);
                                    kx[r][1] = __ffma2_rn(w2[j][1], x1, kx[r][1]);
                                }
                            }
                        }
                        if (ACT) {
#pragma unroll
                            for (int r = 0; r < 4; ++r)
#pragma unroll
                                for (int pp = 0; pp < 2; ++pp)
                                    kx[r][pp] = make_float2(silu(kx[r][pp].x), silu(kx[r][pp].y));
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        if (rb + r >= nc) kx[r][0] = kx[r][1] = make_float2(0.f, 0.f);
                    }
                    if (CK > 0) {
                        // L2 norm over the row's 128 channels: the warp's 32 lanes
                        float ss[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float2 s2 = __ffma2_rn(kx[r][1], kx[r][1], __fmul2_rn(kx[r][0], kx[r][0]));
                            ss[r] = s2.x + s2.y;
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                            for (int r = 0; r < 4; ++r) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], o);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float inv = rsqrtf(ss[r] + kL2Eps);  // hardware reciprocal square root
                            const float2 i2 = make_float2(inv, inv);
                            kx[r][0] = __fmul2_rn(kx[r][0], i2);
                            kx[r][1] = __fmul2_rn(kx[r][1], i2);
                        }
                    }
                    // K rounded to tf32, stored in fp16 (which holds it exactly) and in bf16
                    // (operand of the Pt_T correction: a second rounding ~2^-11 of a term that
                    // is ~2^-11 of Pt_T); a row's 32 8-byte pieces, one per lane
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float x0 = tc::round_tf32(kx[r][0].x), x1 = tc::round_tf32(kx[r][0].y);
                        const float x2 = tc::round_tf32(kx[r][1].x), x3 = tc::round_tf32(kx[r][1].y);
                        *reinterpret_cast<uint2 *>(kh + o16(rb + r)) = make_uint2(pack_f16(x0, x1), pack_f16(x2, x3));
                        *reinterpret_cast<uint2 *>(kb + o16(rb + r)) = make_uint2(pack_bf16(x0, x1), pack_bf16(x2, x3));
                    }
                }
                tc::fence_async_smem();
                tc::bar_sync(BAR_CONV, 128);  // every raw row read, K in fp16 and bf16 written
                if (ct == 0) {
                    tc::mbar_arrive(bar(B_KRDY + (n & 1)));
                    tc::mbar_arrive(bar(B_KRE + n % RK));
                }
                // K in tf32 (B of Pt_S and Pt_T, single buffer) once the previous chunk's Pt_T
                // has read it: a row's 32 16-byte chunks, one per lane
                w = true;
                if (ct == 0 && n > 0) w = wait_bar(bar(B_K32E), (n - 1) & 1, abort_flag);
                if (!tc::bar_and(BAR_CONV, 128, w)) { ok = false; break; }
                {
                    uint8_t *k32 = sm + SM_K32;
#pragma unroll 4
                    for (int r = 0; r < 16; ++r) {
                        const int row = r0 + r;
                        const uint2 h = *reinterpret_cast<const uint2 *>(kh + o16(row));
                        const float2 a0 = __half22float2(*reinterpret_cast<const __half2 *>(&h.x));
                        const float2 a1 = __half22float2(*reinterpret_cast<const __half2 *>(&h.y));
                        *reinterpret_cast<float4 *>(k32 + tc::sw128_f32(row, c0, C)) = make_float4(a0.x, a0.y, a1.x, a1.y);
                    }
                }
                tc::fence_async_smem();
                tc::bar_sync(BAR_CONV, 128);
                if (ct == 0) tc::mbar_arrive(bar(B_K32R));
            }
        }
    } else if (warp == WARP_GATE) {
        // ------------------------------------------------------------ gates
        // The chunk's gates from alpha and beta (lane: tokens 2 lane, 2 lane + 1).
        // The bf16 bits of the next chunk's alpha and beta are loaded while
        // this chunk's are turned into gates (padding: alpha = 1, beta = 0).
        const uint16_t *ap = static_cast<const uint16_t *>(a.tok.alpha);
        const uint16_t *bp = static_cast<const uint16_t *>(a.tok.beta);
        auto load_raw = [&](const Item &itg, int cg, uint32_t (&ra)[2], uint32_t (&rb)[2]) {
            const int ncg = min(C, (int)(itg.n - cg * C));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int tt = 2 * lane + u;
                ra[u] = 0x3F80u;
                rb[u] = 0u;
                if (tt < ncg) {
                    const size_t gi = gate_index(dm, N, itg.l, itg.b0 + cg * C + tt, itg.h);
                    ra[u] = ap[gi];
                    rb[u] = bp[gi];
                }
            }
        };
        uint32_t ca[2] = {0x3F80u, 0x3F80u}, cb[2] = {0u, 0u};
        bool first = true;
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            if (it.nch == 0) continue;
            if (first) {
                load_raw(it, 0, ca, cb);
                first = false;
            }
            for (int c = 0; c < it.nch; ++c, ++n) {
                // the next chunk of this CTA: the next one of this item, else the
                // first of the next non-empty item
                uint32_t na[2] = {0x3F80u, 0x3F80u}, nb[2] = {0u, 0u};
                if (c + 1 < it.nch) {
                    load_raw(it, c + 1, na, nb);
                } else {
                    for (int nx = itx + gridDim.x; nx < n_items; nx += gridDim.x) {
                        const Item itn = decode_item(nx, dm, tab);
                        if (itn.nch > 0) {
                            load_raw(itn, 0, na, nb);
                            break;
                        }
                    }
                }
                if (n >= RG && !wait_bar(bar(B_GE + n % RG), ((n / RG) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                Gates &G = *reinterpret_cast<Gates *>(sm + SM_GATE + (n % RG) * G_STAGE);
                const float al0 = __uint_as_float(ca[0] << 16), al1 = __uint_as_float(ca[1] << 16);
                const float be[2] = {__uint_as_float(cb[0] << 16), __uint_as_float(cb[1] << 16)};
                const float x0 = fmaxf(logf(al0), -88.f);  // alpha = 0 -> exp(-88)
                const float x1 = fmaxf(logf(al1), -88.f);
                float sum = x0 + x1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sum, o);
                    if (lane >= o) sum += y;
                }
                const float total = __shfl_sync(0xffffffffu, sum, 31);
                const float first_g = __shfl_sync(0xffffffffu, x0, 0);
                const float g1 = sum, g0 = sum - x1;
                G.eg[2 * lane] = expf(g0);
                G.eg[2 * lane + 1] = expf(g1);
                G.b[2 * lane] = be[0];
                G.b[2 * lane + 1] = be[1];
                G.dc[2 * lane] = be[0] * expf(total - g0);
                G.dc[2 * lane + 1] = be[1] * expf(total - g1);
                *reinterpret_cast<float2 *>(&G.nrc[2 * lane]) =
                    make_float2(-expf(fminf(g0 - total, 88.f)), -expf(fminf(g1 - total, 88.f)));
                *reinterpret_cast<float2 *>(&G.neg[2 * lane]) = make_float2(-expf(g0), -expf(g1));
                if (lane == 0) G.safe = (first_g - total <= kSpan) ? 1 : 0;
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(B_GF + n % RG));
                ca[0] = na[0];
                ca[1] = na[1];
                cb[0] = nb[0];
                cb[1] = nb[1];
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ solve
        const int sp = tid - 384;  // 0 .. 127
        const int q = warp & 3;    // lane quadrant; 16-token block; channels 32q .. 32q+31
        const int g = lane >> 2, t4 = lane & 3;
        // Z: L'' strictly below the diagonal, W^T on and above it, fp16 (the tf32-rounded
        // values' mantissa, and |entries| stay far inside fp16's range)
        __half *Zh = reinterpret_cast<__half *>(sm + SM_L);
        float *gtb = reinterpret_cast<float *>(sm + SM_TMP);                  // 4 x G^T [8][8]
        const uint32_t sZ = s_base + SM_L, sX = s_base + SM_TMP + 4 * 64 * 4; // 4 x [16][TP2] fp16
        auto zh = [&](int r, int c) -> __half & { return Zh[r * ZP + c]; };
        auto zad = [&](int r, int c) { return sZ + static_cast<uint32_t>((r * ZP + c) * 2); };
        auto xad = [&](int w, int r, int c) { return sX + static_cast<uint32_t>(((w * 16 + r) * TP2 + c) * 2); };
        // fp16 pair (row r, columns c, c + 1) of a tile
        auto put2 = [&](uint32_t addr, float lo, float hi) {
            *reinterpret_cast<uint32_t *>(sm + (addr - s_base)) = pack_f16(lo, hi);
        };
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            for (int c = 0; c < it.nch; ++c, ++n) {
                bool w = true;
                if (sp == 0) w = wait_bar(bar(B_GRAMF), n & 1, abort_flag);
                if (sp == 32) w = wait_bar(bar(B_GF + n % RG), (n / RG) & 1, abort_flag);
                if (!tc::bar_and(BAR_SOLVE, 128, w)) { ok = false; break; }
                tc::fence_after();
                const Gates &G = gates(n);
                {
                    // L''_tj = beta_t k_t.k_j from the Gram rows: row 16q + i sits in lane
                    // 32q + i (i < 16); lanes 0-15 take its columns 0-31, lanes 16-31
                    // columns 32-63.  Entries on and above the diagonal are overwritten
                    // by W^T before anything reads them.
                    float gr[32];
                    tc::tmem_ld16x2_32(my + TM_G, gr);
                    const int t = 16 * q + (lane & 15);
                    const int j0 = (lane >= 16) ? 32 : 0;
                    const float bt = G.b[t];
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        *reinterpret_cast<uint4 *>(&zh(t, j0 + j)) =
                            make_uint4(pack_f16(bt * gr[j], bt * gr[j + 1]), pack_f16(bt * gr[j + 2], bt * gr[j + 3]),
                                       pack_f16(bt * gr[j + 4], bt * gr[j + 5]), pack_f16(bt * gr[j + 6], bt * gr[j + 7]));
                }
                tc::fence_before();
                tc::bar_sync(BAR_SOLVE, 128);
                if (sp == 0) tc::mbar_arrive(bar(B_GRAME));
                if (lane < 16) {
                    // column j of the 8 x 8 diagonal block E_b = (I + L''_bb)^{-1}, b = 2q + lane / 8,
                    // by forward substitution in fp32; column r of L''_bb is loaded one step ahead
                    const int hb = lane >> 3, base = 16 * q + 8 * hb, j = lane & 7;
                    float x[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) x[r] = (r == j) ? 1.f : 0.f;
                    float col[7];
#pragma unroll
                    for (int k = 0; k < 7; ++k) col[k] = __half2float(zh(base + k + 1, base));
#pragma unroll
                    for (int r = 0; r < 7; ++r) {
                        float nxt[6];
#pragma unroll
                        for (int k = 0; k < 6 - r; ++k) nxt[k] = __half2float(zh(base + r + 2 + k, base + r + 1));
                        asm volatile("" ::: "memory");  // issue them before this step's products
#pragma unroll
                        for (int k = 0; k < 7 - r; ++k) x[r + 1 + k] = fmaf(-col[k], x[r], x[r + 1 + k]);
#pragma unroll
                        for (int k = 0; k < 6 - r; ++k) col[k] = nxt[k];
                    }
                    __syncwarp(0x0000ffffu);  // every read of L''_bb is done
                    // row j of E_b^T into Z (its strictly lower part, zero, replaces the
                    // consumed L''_bb)
                    *reinterpret_cast<uint4 *>(&zh(base + j, base)) =
                        make_uint4(pack_f16(x[0], x[1]), pack_f16(x[2], x[3]), pack_f16(x[4], x[5]), pack_f16(x[6], x[7]));
                }
                __syncwarp();
                {
                    // M_q = (I + L''_qq)^{-1}: its lower-left 8 x 8 F = -E_{2q+1} L''_{2q+1,2q} E_{2q}
                    // (lane: row r, columns c0, c0 + 1), in fp32
                    const int r = lane >> 2, c0 = 2 * (lane & 3), b0 = 16 * q;
                    float la[8];
                    {
                        const uint4 h = *reinterpret_cast<const uint4 *>(&zh(b0 + 8 + r, b0));
                        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hw[k]));
                            la[2 * k] = f.x;
                            la[2 * k + 1] = f.y;
                        }
                    }
                    float *gt = gtb + q * 64;  // G^T [8][8], G = L''_{2q+1,2q} E_{2q}
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        // column c0 + u of E_{2q}: row c0 + u of E_{2q}^T
                        const uint4 h = *reinterpret_cast<const uint4 *>(&zh(b0 + c0 + u, b0));
                        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
                        float gv = 0.f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hw[k]));
                            gv = fmaf(la[2 * k], f.x, gv);
                            gv = fmaf(la[2 * k + 1], f.y, gv);
                        }
                        gt[(c0 + u) * 8 + r] = gv;
                    }
                    __syncwarp();
                    float er[8];  // row r of E_{2q+1}
#pragma unroll
                    for (int k = 0; k < 8; ++k) er[k] = __half2float(zh(b0 + 8 + k, b0 + 8 + r));
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float4 ga = *reinterpret_cast<const float4 *>(gt + (c0 + u) * 8);
                        const float4 gb = *reinterpret_cast<const float4 *>(gt + (c0 + u) * 8 + 4);
                        float f = er[0] * ga.x;
                        f = fmaf(er[1], ga.y, f);
                        f = fmaf(er[2], ga.z, f);
                        f = fmaf(er[3], ga.w, f);
                        f = fmaf(er[4], gb.x, f);
                        f = fmaf(er[5], gb.y, f);
                        f = fmaf(er[6], gb.z, f);
                        f = fmaf(er[7], gb.w, f);
                        zh(b0 + c0 + u, b0 + 8 + r) = __float2half_rn(-f);  // W^T[b0 + c][b0 + 8 + r]
                        zh(b0 + 8 + r, b0 + c0 + u) = __float2half_rn(0.f);  // upper-right 8 x 8 of M_q
                    }
                }
                tc::bar_sync(BAR_SOLVE, 128);
                {
                    // 32-token blocks, transposed: W_ji^T = -(M_i^T L''_ji^T) M_j^T for
                    // (j, i) = (1, 0), (3, 2); warp: pair w / 2, output columns 8 (w % 2) ..
                    const int jb = (q >> 1) ? 3 : 1, ib = jb - 1, nt = q & 1;
                    uint32_t af[4], bf[2];
                    frag_a16(af, zad(16 * ib, 16 * ib), ZP, lane);  // M_i^T
#pragma unroll
                    for (int qt = 0; qt < 2; ++qt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        frag_b16t(bf, zad(16 * jb + 8 * qt, 16 * ib), ZP, lane);  // L''_ji rows = (L''_ji^T) columns
                        mma16x8x16_f16(acc, af, bf);
                        put2(xad(q, g, 8 * qt + 2 * t4), acc[0], acc[1]);
                        put2(xad(q, g + 8, 8 * qt + 2 * t4), acc[2], acc[3]);
                    }
                    __syncwarp();
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    frag_a16(af, xad(q, 0, 0), TP2, lane);
                    frag_b16(bf, zad(16 * jb, 16 * jb + 8 * nt), ZP, lane);  // M_j^T, row-major
                    mma16x8x16_f16(acc, af, bf);
                    put2(zad(16 * ib + g, 16 * jb + 8 * nt + 2 * t4), -acc[0], -acc[1]);
                    put2(zad(16 * ib + g + 8, 16 * jb + 8 * nt + 2 * t4), -acc[2], -acc[3]);
                }
                tc::bar_sync(BAR_SOLVE, 128);
                {
                    // 64 tokens: Y^T = W_a^T L''_ba^T (warp: block (w / 2, w % 2) of Y, transposed)
                    const int yr = q >> 1, yc = q & 1;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int kb = yc; kb < 2; ++kb) {
                            uint32_t af[4], bf[2];
                            frag_a16(af, zad(16 * yc, 16 * kb), ZP, lane);
                            frag_b16t(bf, zad(16 * (2 + yr) + 8 * nt, 16 * kb), ZP, lane);
                            mma16x8x16_f16(acc, af, bf);
                        }
                        put2(xad(q, g, 8 * nt + 2 * t4), acc[0], acc[1]);
                        put2(xad(q, g + 8, 8 * nt + 2 * t4), acc[2], acc[3]);
                    }
                }
                tc::bar_sync(BAR_SOLVE, 128);
                {
                    // W_ba^T = -Y^T W_b^T (warp: block (2 + w / 2, w % 2) of W, transposed)
                    const int wr = 2 + (q >> 1), wc = q & 1;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int kb = 2; kb <= wr; ++kb) {
                            uint32_t af[4], bf[2];
                            frag_a16(af, xad((kb - 2) * 2 + wc, 0, 0), TP2, lane);
                            frag_b16(bf, zad(16 * kb, 16 * wr + 8 * nt), ZP, lane);  // W_{wr,kb}^T, row-major
                            mma16x8x16_f16(acc, af, bf);
                        }
                        put2(zad(16 * wc + g, 16 * wr + 8 * nt + 2 * t4), -acc[0], -acc[1]);
                        put2(zad(16 * wc + g + 8, 16 * wr + 8 * nt + 2 * t4), -acc[2], -acc[3]);
                    }
                }
                w = true;
                if (sp == 0 && n > 0) w = wait_bar(bar(B_UTE), (n - 1) & 1, abort_flag);  // U~^T free
                if (!tc::bar_and(BAR_SOLVE, 128, w)) { ok = false; break; }
                {
                    // U~_i = D_i sum_{j >= i} W_ji^T K_j for channels 32q .. 32q+31 with fp16 warp
                    // MMAs (m16n8k16): A = the (i, j) block of W^T from Z; B = K_j from the fp16
                    // K tile by transposing ldmatrix.
                    const uint32_t skh = s_base + SM_KH + (n & 1) * 16384;
                    // ldmatrix rows: token 16 j + (lane & 7) + 8 ((lane >> 3) & 1), channel group
                    // 8 (2 p + lane / 16) of this warp's 32 (n-tile pair p)
                    const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;
                    uint32_t bro[2];
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const int ch = 32 * q + 8 * (2 * pp + (lane >> 4));
                        bro[pp] = (ch >> 6) * 8192 + lr * 128 + ((((ch & 63) >> 3) ^ (lr & 7)) << 4);
                    }
                    // C stores: element e = (channel + (e & 1), token + 8 (e >> 1))
                    uint32_t so[2][4];
#pragma unroll
                    for (int i1 = 0; i1 < 2; ++i1)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            so[i1][e] = (e & 1) * 128 +
                                        ((((4 * i1 + (g >> 2) + 2 * (e >> 1)) ^ (2 * t4 + (e & 1))) << 4) + (g & 3) * 4);
                    const uint32_t sbase = SM_UT + (32 * q + 2 * t4) * 128;
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        float acc[4][4];
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll 1
                        for (int j = i; j < 4; ++j) {
                            // every operand of the term first, then its four MMAs
                            uint32_t af[4], bf[4][2];
                            frag_a16(af, zad(NB * i, NB * j), ZP, lane);
#pragma unroll
                            for (int pp = 0; pp < 2; ++pp) {
                                uint32_t r4[4];
                                ldsm_x4_t(r4, skh + bro[pp] + NB * j * 128);
                                bf[2 * pp][0] = r4[0];
                                bf[2 * pp][1] = r4[1];
                                bf[2 * pp + 1][0] = r4[2];
                                bf[2 * pp + 1][1] = r4[3];
                            }
#pragma unroll
                            for (int nt = 0; nt < 4; ++nt) mma16x8x16_f16(acc[nt], af, bf[nt]);
                        }
                        uint8_t *ub = sm + sbase + (i >> 1) * 16384;
                        const float dd[2] = {G.dc[NB * i + g], G.dc[NB * i + g + 8]};
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                *reinterpret_cast<float *>(ub + nt * 1024 + ((i & 1) ? so[1][e] : so[0][e])) =
                                    tc::round_tf32(acc[nt][e] * dd[e >> 1]);
                    }
                }
                tc::fence_async_smem();
                tc::bar_sync(BAR_SOLVE, 128);
                if (sp == 0) {
                    tc::mbar_arrive(bar(B_UTF));
                    tc::mbar_arrive(bar(B_KHE + (n & 1)));
                    tc::mbar_arrive(bar(B_GE + n % RG));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-7)
        // Warp w works on tensor-memory lane quadrant w % 4 -- lane m is row m of Xt_T,
        // Pt_T, Xt_S and Pt_S: column m of T and of S, value channel m -- and on half
        // h = w / 4 of every pass: tokens 32h .. 32h+31 of Rt_S and Rt_T, columns
        // 64h .. 64h+63 of Xt_T and Xt_S.
        const int m = (warp & 3) * 32 + lane;
        const int et = tid;              // 0 .. 255
        const int pc = 32 * (warp >> 2); // Pt columns (tokens) of this thread
        const int xc = 64 * (warp >> 2); // Xt columns of this thread
        float wvr[CK > 0 ? CK : 1];
        int n = 0;
        bool ok = true;
        for (int itx = blockIdx.x; itx < n_items && ok; itx += gridDim.x) {
            const Item it = decode_item(itx, dm, tab);
            const size_t pair = ((size_t)it.l * tab.n_seg + it.s) * dm.H + it.h;
            float *To = a.T_out + pair * D * D + m;
            float *So = a.S_out + pair * D * D + m;
            if (it.nch == 0) {
                for (int i = xc; i < xc + 64; ++i) {
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
            // Xt_T = s I with s = Gamma_C of the first chunk (pre-scaled) or 1, its low part; Xt_S = 0
            bool w = true;
            if (et == 0) w = wait_bar(bar(B_GF + n % RG), (n / RG) & 1, abort_flag);
            if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
            {
                const Gates &G0 = gates(n);
                const float s = G0.safe ? G0.eg[C - 1] : 1.f;
                const float slo = s - __uint_as_float(__float_as_uint(s) & 0xffffe000u);
#pragma unroll 1
                for (int cc = xc; cc < xc + 64; cc += 32) {
                    float v[32];
                    uint32_t lo[16];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (cc + i == m) ? s : 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        lo[i] = pack_bf16((cc + 2 * i == m) ? slo : 0.f, (cc + 2 * i + 1 == m) ? slo : 0.f);
                    tc::tmem_st32_async(my + TM_XT + cc, v);
                    tc::tmem_st16_async(my + TM_XLO + cc / 2, lo);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    tc::tmem_st32_async(my + TM_XS + cc, v);
                    tc::tmem_wait_st();
                }
            }
            tc::fence_before();
            tc::bar_sync(BAR_EPI, 256);
            if (et == 0) {
                tc::mbar_arrive(bar(B_XTR));
                tc::mbar_arrive(bar(B_XSI));
            }
            for (int c = 0; c < it.nch; ++c, ++n) {
                const int nc = min(C, (int)(it.n - c * C));
                const uint8_t *stg = sm + SM_VR + (n % RV) * VR_STAGE;
                w = true;
                if (et == 32) w = wait_bar(bar(B_VRF + n % RV), (n / RV) & 1, abort_flag);
                if (et == 64) w = wait_bar(bar(B_GF + n % RG), (n / RG) & 1, abort_flag);
                if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
                const Gates &G = gates(n);
                {
                    // conv of raw V, channel m, tokens pc .. pc+31 (0 past the chunk's end);
                    // it does not wait for Pt_S
                    float vv[32];
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        // staged rows tq .. tq + 15 + HIST: lag j of token t is staged row t + HIST - j
                        const int tq = pc + 16 * qq;
                        float v[16 + HIST];
#pragma unroll
                        for (int i = 0; i < 16 + HIST; ++i) v[i] = bf16_at(stg, tq + i, m);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            float2 x;
                            if (CK == 0) {
                                x = make_float2(v[i], v[i + 1]);
                            } else {
                                x = make_float2(0.f, 0.f);
#pragma unroll
                                for (int j = 0; j < (CK > 0 ? CK : 1); ++j)
                                    x = __ffma2_rn(make_float2(wvr[j], wvr[j]),
                                                   make_float2(v[i + HIST - j], v[i + 1 + HIST - j]), x);
                                if (ACT) x = make_float2(silu(x.x), silu(x.y));
                            }
                            vv[16 * qq + i] = (tq + i < nc) ? x.x : 0.f;
                            vv[16 * qq + i + 1] = (tq + i + 1 < nc) ? x.y : 0.f;
                        }
                    }
                    w = true;
                    if (et == 0) w = wait_bar(bar(B_PSF), n & 1, abort_flag);
                    if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
                    tc::fence_after();
                    // Rt_S = V^T - Pt_S diag(Gamma), then Xt_S <- Gamma_C Xt_S (Pt_S has read it)
                    uint32_t p[32];
                    tc::tmem_ld32_issue(my + TM_PS + pc, p);
                    tc::tmem_wait_ld32(p);
                    const float2 *ng = reinterpret_cast<const float2 *>(G.neg + pc);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 r = __ffma2_rn(ng[i], make_float2(__uint_as_float(p[2 * i]), __uint_as_float(p[2 * i + 1])),
                                                    make_float2(vv[2 * i], vv[2 * i + 1]));
                        p[2 * i] = __float_as_uint(tc::round_tf32(r.x));
                        p[2 * i + 1] = __float_as_uint(tc::round_tf32(r.y));
                    }
                    tc::tmem_st32_async(my + TM_PS + pc, reinterpret_cast<const float *>(p));
                    scale_cols(my + TM_XS + xc, G.eg[C - 1]);
                }
                tc::fence_before();
                tc::bar_sync(BAR_EPI, 256);
                if (et == 0) {
                    tc::mbar_arrive(bar(B_RSF));
                    tc::mbar_arrive(bar(B_VRE + n % RV));
                }
                w = true;
                if (et == 0) w = wait_bar(bar(B_PTF), n & 1, abort_flag);
                if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
                tc::fence_after();
                const bool safe = G.safe != 0;
                {
                    // pre-scaled: Rt_T = -Pt_T Gamma_t / Gamma_C; else -Pt_T Gamma_t
                    float p[32];
                    const float2 *f = reinterpret_cast<const float2 *>((safe ? G.nrc : G.neg) + pc);
                    tc::tmem_ld32(my + TM_PT + pc, p);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 r = __fmul2_rn(f[i], make_float2(p[2 * i], p[2 * i + 1]));
                        p[2 * i] = tc::round_tf32(r.x);
                        p[2 * i + 1] = tc::round_tf32(r.y);
                    }
                    tc::tmem_st32(my + TM_PT + pc, p);
                    // not pre-scaled: Xt_T <- Gamma_C Xt_T here, after Pt_T has read it
                    if (!safe) scale_cols(my + TM_XT + xc, G.eg[C - 1]);
                }
                tc::fence_before();
                tc::bar_sync(BAR_EPI, 256);
                if (et == 0) {
                    tc::mbar_arrive(bar(B_RTF));
                    tc::mbar_arrive(bar(B_GE + n % RG));
                }
                const bool last = c + 1 == it.nch;
                w = true;
                if (et == 0) {
                    w = wait_bar(bar(B_XTD), n & 1, abort_flag);
                    if (w && !last) w = wait_bar(bar(B_GF + (n + 1) % RG), ((n + 1) / RG) & 1, abort_flag);
                }
                if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
                tc::fence_after();
                if (last) {
                    // emit T[i][m] = Xt_T[m][i], then S[i][m] = Xt_S[m][i] once the last update is done
                    float x[32];
#pragma unroll 1
                    for (int cc = xc; cc < xc + 64; cc += 32) {
                        tc::tmem_ld32(my + TM_XT + cc, x);
#pragma unroll
                        for (int i = 0; i < 32; ++i) To[(size_t)(cc + i) * D] = x[i];
                    }
                    w = true;
                    if (et == 0) w = wait_bar(bar(B_XSD), n & 1, abort_flag);
                    if (!tc::bar_and(BAR_EPI, 256, w)) { ok = false; break; }
                    tc::fence_after();
#pragma unroll 1
                    for (int cc = xc; cc < xc + 64; cc += 32) {
                        tc::tmem_ld32(my + TM_XS + cc, x);
#pragma unroll
                        for (int i = 0; i < 32; ++i) So[(size_t)(cc + i) * D] = x[i];
                    }
                } else {
                    const Gates &G1 = gates(n + 1);
                    scale_split_xt(my, xc, G1.safe ? G1.eg[C - 1] : 1.f);
                    tc::fence_before();
                    tc::bar_sync(BAR_EPI, 256);
                    if (et == 0) tc::mbar_arrive(bar(B_XTR));
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
    // the SM count of the device this launch runs on (cheap; no caching across devices)
    int dev = 0, n_sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int rows = C + (a.dm.conv_k > 0 ? a.dm.conv_k - 1 : 0);
    CUtensorMap tmK, tmV;
    if ((e = make_token_map(&tmK, a.tok.k, a.dm, a.tok.N, rows)) != cudaSuccess) return e;
    if ((e = make_token_map(&tmV, a.tok.v, a.dm, a.tok.N, rows)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(int), st)) != cudaSuccess) return e;
    const int grid = n_items < n_sms ? n_items : n_sms;
    // the activation after the conv is a template flag: no cost when off
    auto kern = a.dm.conv_k == 0 ? build_tc_kernel<0, false>
                                 : (a.dm.act ? build_tc_kernel<4, true> : build_tc_kernel<4, false>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN))) return e;
    kern<<<grid, NT, SMEM_DYN, st>>>(a, tab, tmK, tmV);
    return cudaGetLastError();
}

}  // namespace hypic
