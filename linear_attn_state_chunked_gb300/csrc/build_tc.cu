// build_tc.cu -- segment build of the gated-delta pair on the tcgen05 tensor
// cores, chunked in the WY form, for d_k = d_v = 128 and bf16 inputs.
//
// Math (derived from the recurrence S_t = alpha_t (I - beta_t k_t k_t^T)
// S_{t-1} + beta_t k_t v_t^T and the pair of the HYPIC pages' "线性层"
// section).  Within a chunk of C = 64 tokens let g_t = sum_{s<=t} log alpha_s,
// Gamma_t = exp(g_t).  Writing u_t = v_t - alpha_t S_{t-1}^T k_t, one finds
//   S_C = Gamma_C S_0 + K^T D U,   U = (I + L)^{-1} (V - diag(Gamma) K S_0),
//   L_tj = beta_j exp(g_t - g_j) k_t.k_j  (j < t),  D = diag(beta_j exp(g_C - g_j)).
// The same map advances T (with V replaced by 0), so X = [T | S] (d_k x 2d)
// is carried as one matrix.  Kept transposed in tensor memory (Xt = X^T,
// 256 rows x 128), one chunk is
//   Pt = Xt K^T                       (tf32 MMA, A = Xt from tensor memory)
//   Rt = [0 | V]^T - Pt diag(Gamma)   (CUDA cores)
//   Xt = Gamma_C Xt + Rt U~,  U~^T = K^T D (I + L)^{-1}   (tf32 MMAs)
// with the Gram matrix K K^T on the tensor core and the 64 x 64 unit lower
// triangular inverse by blocked substitution on CUDA cores.  Every operand
// written to shared memory is rounded to tf32 (the tensor core truncates).
//
// Work items (segment body, layer, head) are taken longest body first from a
// device counter by persistent CTAs, one per SM: the greedy LPT schedule of
// the pages' "段并行" section as a single-GPU stand-in.
#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace hypic {
namespace {

constexpr int D = 128;   // head width
constexpr int C = 64;    // chunk length
constexpr int NT = 128;  // threads = tensor-memory lanes
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds

// tensor-memory columns
constexpr uint32_t TM_XT = 0;    // Xt, T half: 128 lanes x 128
constexpr uint32_t TM_XS = 128;  // Xt, S half
constexpr uint32_t TM_PT = 256;  // Pt, T half: 128 x 64
constexpr uint32_t TM_PS = 320;  // Pt, S half
constexpr uint32_t TM_G = 384;   // Gram K K^T (M = 64 layout): 64 x 64
constexpr uint32_t TM_U = 448;   // U~^T: 128 x 64
constexpr uint32_t TM_COLS = 512;

// shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t SM_K32 = 0;               // K   [64][128]  tf32, sw128
constexpr uint32_t SM_UT = 32768;            // U~^T [128][64] tf32, sw128 (B of the X update)
constexpr uint32_t SM_RT = 65536;            // Rt  [2][128][64] tf32, sw128
constexpr uint32_t SM_KT = SM_RT;            // K^T [128][64] (aliases Rt T half)
constexpr uint32_t SM_MT = SM_RT + 32768;    // (D M)^T [64][64] (aliases Rt S half)
constexpr uint32_t SM_V = 131072;            // V   [64][128] fp32
constexpr int LP = C + 1;                    // padded row of L and M
constexpr uint32_t SM_L = 163840;            // L   [64][65] fp32
constexpr uint32_t SM_M = SM_L + C * LP * 4; // M = (I + L)^-1 [64][65]
constexpr uint32_t SM_Q = SM_M + C * LP * 4; // block products [3][16][17]
constexpr uint32_t SM_GATE = SM_Q + 3 * 16 * 17 * 4 + 64;  // 5 x 64 floats
constexpr uint32_t SM_BYTES = SM_GATE + 5 * 64 * 4;
constexpr uint32_t SMEM_DYN = SM_BYTES + 1024;  // slack for 1024-byte alignment

struct Gates {
    float g[C];    // inclusive log-gate sums
    float b[C];    // beta
    float eg[C];   // exp(g_t)
    float dc[C];   // beta_j exp(g_C - g_j)
    float lg[C];   // log alpha
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &u, float *x)
{
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

// Blocked inverse of the unit lower triangular (I + L), 64 = 4 x 16 blocks:
// diagonal blocks by substitution, then M_ij = -M_ii sum_{k=j}^{i-1} L_ik M_kj
// level by level.
__device__ void unit_lower_inverse(const float *Ls, float *Ms, float *Qs, int tid)
{
    if (tid < 64) {
        const int b = tid >> 4, cc = tid & 15, base = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < r; ++j) acc = fmaf(-Ls[(base + r) * LP + base + j], x[j], acc);
            x[r] = (r < cc) ? 0.f : acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Ms[(base + r) * LP + base + cc] = x[r];
    }
    // strictly upper blocks are zero
    for (int e = tid; e < 6 * 256; e += NT) {
        const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const int bi = (blk < 3) ? 0 : (blk < 5 ? 1 : 2);
        const int bj = (blk < 3) ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Ms[(16 * bi + r) * LP + 16 * bj + cc] = 0.f;
    }
    __syncthreads();
    for (int delta = 1; delta <= 3; ++delta) {
        const int nblk = 4 - delta;
        for (int e = tid; e < nblk * 256; e += NT) {
            const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const int bj = blk, bi = blk + delta;
            float acc = 0.f;
            for (int bk = bj; bk < bi; ++bk) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    acc = fmaf(Ls[(16 * bi + r) * LP + 16 * bk + q], Ms[(16 * bk + q) * LP + 16 * bj + cc], acc);
            }
            Qs[(blk * 16 + r) * 17 + cc] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += NT) {
            const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const int bj = blk, bi = blk + delta;
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q)
                acc = fmaf(Ms[(16 * bi + r) * LP + 16 * bi + q], Qs[(blk * 16 + q) * 17 + cc], acc);
            Ms[(16 * bi + r) * LP + 16 * bj + cc] = -acc;
        }
        __syncthreads();
    }
}

template <int CK>
__global__ void __launch_bounds__(NT, 1)
build_tc_kernel(const __grid_constant__ BuildArgs a, const __grid_constant__ SegTable tab)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int item_sh;

    float *Vs = reinterpret_cast<float *>(sm + SM_V);
    float *Ls = reinterpret_cast<float *>(sm + SM_L);
    float *Ms = reinterpret_cast<float *>(sm + SM_M);
    float *Qs = reinterpret_cast<float *>(sm + SM_Q);
    Gates &gt = *reinterpret_cast<Gates *>(sm + SM_GATE);
    const uint32_t s_base = tc::smem_u32(sm);
    const uint32_t sK32 = s_base + SM_K32, sUT = s_base + SM_UT, sRT = s_base + SM_RT;
    const uint32_t sKT = s_base + SM_KT, sMT = s_base + SM_MT;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Dims dm = a.dm;
    const int32_t N = a.tok.N;
    const int LH = dm.L * dm.H;
    const int n_items = tab.n_seg * LH;
    const uint32_t mb = tc::smem_u32(&mbar);

    if (tid == 0) {
        tc::mbar_init(mb, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tc::smem_u32(&tmem_base_sh), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t my = tb + lane_off;  // this thread's lane, column 0
    uint32_t phase = 0;
    bool failed = false;

    const __nv_bfloat16 *kp = static_cast<const __nv_bfloat16 *>(a.tok.k);
    const __nv_bfloat16 *vp = static_cast<const __nv_bfloat16 *>(a.tok.v);
    const __nv_bfloat16 *ap = static_cast<const __nv_bfloat16 *>(a.tok.alpha);
    const __nv_bfloat16 *bp = static_cast<const __nv_bfloat16 *>(a.tok.beta);

    // issue from one thread, then wait for completion on every thread
    auto mma_done = [&]() -> bool {
        const bool ok = tc::mbar_wait(mb, phase, kWaitCycles);
        phase ^= 1u;
        tc::fence_after();
        return __syncthreads_and(ok);
    };

    while (true) {
        if (tid == 0) item_sh = static_cast<int>(atomicAdd(a.work_counter, 1u));
        __syncthreads();
        const int item = item_sh;
        if (item >= n_items) break;
        const int s = tab.perm[item / LH];
        const int lh = item % LH;
        const int l = lh / dm.H, h = lh % dm.H;
        const int32_t seg0 = tab.off[s], seg1 = tab.off[s + 1];
        const int32_t b0 = seg0 + min(dm.w, seg1 - seg0);
        const int32_t n = seg1 - b0;

        // X = [I | 0]
        {
            float v[32];
#pragma unroll
            for (int c = 0; c < D; c += 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = (c + i == tid) ? 1.f : 0.f;
                tc::tmem_st32(my + TM_XT + c, v);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll
            for (int c = 0; c < D; c += 32) tc::tmem_st32(my + TM_XS + c, v);
        }

        for (int32_t t0 = 0; t0 < n && !failed; t0 += C) {
            const int nc = min(C, (int)(n - t0));
            // ---- gates: inclusive scan of log alpha over the chunk
            if (tid < C) {
                const bool valid = tid < nc;
                float al = 1.f, be = 0.f;
                if (valid) {
                    const size_t gi = gate_index(dm, N, l, b0 + t0 + tid, h);
                    al = __bfloat162float(ap[gi]);
                    be = __bfloat162float(bp[gi]);
                }
                float x = fmaxf(logf(al), -88.f);  // alpha = 0 -> exp(-88), below fp32 normals
                gt.lg[tid] = x;
                gt.b[tid] = be;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                gt.g[tid] = x;
            }
            __syncthreads();
            if (tid >= 32 && tid < C) gt.g[tid] += gt.g[31];
            __syncthreads();
            if (tid < C) {
                const float gC = gt.g[C - 1];
                gt.eg[tid] = expf(gt.g[tid]);
                gt.dc[tid] = gt.b[tid] * expf(gC - gt.g[tid]);
            }
            // ---- tokens: K (tf32, both orientations) and V, 8 channels per thread step
            const float *wk = nullptr, *wv = nullptr;
            if (CK > 0) {
                wk = a.tok.conv_w + (((size_t)l * 3 + 1) * dm.H + h) * D * CK;
                wv = a.tok.conv_w + (((size_t)l * 3 + 2) * dm.H + h) * D * CK;
            }
#pragma unroll 1
            for (int it = 0; it < (C * D / 8) / NT; ++it) {
                const int t = it * (NT / 16) + (tid >> 4);
                const int c0 = (tid & 15) * 8;
                float kx[8], vx[8];
                if (t < nc) {
                    const int32_t tok = b0 + t0 + t;
                    if (CK == 0) {
                        unpack8(*reinterpret_cast<const uint4 *>(kp + tok_index(dm, N, l, tok, h, c0)), kx);
                        unpack8(*reinterpret_cast<const uint4 *>(vp + tok_index(dm, N, l, tok, h, c0)), vx);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) kx[i] = vx[i] = 0.f;
#pragma unroll
                        for (int j = 0; j < CK; ++j) {
                            const int32_t tj = tok - j;
                            if (tj >= seg0) {
                                float rk[8], rv[8];
                                unpack8(*reinterpret_cast<const uint4 *>(kp + tok_index(dm, N, l, tj, h, c0)), rk);
                                unpack8(*reinterpret_cast<const uint4 *>(vp + tok_index(dm, N, l, tj, h, c0)), rv);
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    kx[i] = fmaf(__ldg(wk + (c0 + i) * CK + j), rk[i], kx[i]);
                                    vx[i] = fmaf(__ldg(wv + (c0 + i) * CK + j), rv[i], vx[i]);
                                }
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) kx[i] = vx[i] = 0.f;
                }
                if (CK > 0) {
                    // per-token L2 normalisation of k over the 16 lanes holding the row
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) ss = fmaf(kx[i], kx[i], ss);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                    const float inv = 1.f / sqrtf(ss + kL2Eps);
#pragma unroll
                    for (int i = 0; i < 8; ++i) kx[i] *= inv;
                }
                float kr[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) kr[i] = tc::round_tf32(kx[i]);
                *reinterpret_cast<float4 *>(sm + SM_K32 + tc::sw128_f32(t, c0, C)) =
                    make_float4(kr[0], kr[1], kr[2], kr[3]);
                *reinterpret_cast<float4 *>(sm + SM_K32 + tc::sw128_f32(t, c0 + 4, C)) =
                    make_float4(kr[4], kr[5], kr[6], kr[7]);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    *reinterpret_cast<float *>(sm + SM_KT + tc::sw128_f32(c0 + i, t, D)) = kr[i];
                *reinterpret_cast<float4 *>(Vs + t * D + c0) = make_float4(vx[0], vx[1], vx[2], vx[3]);
                *reinterpret_cast<float4 *>(Vs + t * D + c0 + 4) = make_float4(vx[4], vx[5], vx[6], vx[7]);
            }
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            // ---- Gram K K^T (M = 64)
            if (tid == 0) {
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_ss(tb + TM_G, tc::sdesc_kstep(sK32, C, ks), tc::sdesc_kstep(sK32, C, ks),
                               tc::idesc_tf32(64, 64), ks > 0);
                tc::commit(mb);
            }
            if (!mma_done()) { failed = true; break; }
            // ---- L from the Gram rows (M = 64 layout: row 16w + i in lane 32w + i)
            {
                float gr[64];
                tc::tmem_ld32(my + TM_G, gr);
                tc::tmem_ld32(my + TM_G + 32, gr + 32);
                if (lane < 16) {
                    const int t = 16 * warp + lane;
                    const float gt_t = gt.g[t];
#pragma unroll
                    for (int j = 0; j < C; ++j)
                        Ls[t * LP + j] = (j < t) ? gt.b[j] * expf(gt_t - gt.g[j]) * gr[j] : 0.f;
                }
            }
            __syncthreads();
            unit_lower_inverse(Ls, Ms, Qs, tid);
            // ---- B operand of U~^T: element (t, j) = dc_j M[j][t]
            for (int e = tid; e < C * C; e += NT) {
                const int t = e >> 6, j = e & 63;
                *reinterpret_cast<float *>(sm + SM_MT + tc::sw128_f32(t, j, C)) =
                    tc::round_tf32(gt.dc[j] * Ms[j * LP + t]);
            }
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            // ---- U~^T = K^T (D M)   (M = 128, N = 64, K = 64)
            if (tid == 0) {
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ss(tb + TM_U, tc::sdesc_kstep(sKT, D, ks), tc::sdesc_kstep(sMT, C, ks),
                               tc::idesc_tf32(128, 64), ks > 0);
                tc::commit(mb);
            }
            if (!mma_done()) { failed = true; break; }
            {
                float u[32];
#pragma unroll
                for (int c = 0; c < C; c += 32) {
                    tc::tmem_ld32(my + TM_U + c, u);
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(sm + SM_UT + tc::sw128_f32(tid, c + i, D)) =
                            make_float4(tc::round_tf32(u[i]), tc::round_tf32(u[i + 1]),
                                        tc::round_tf32(u[i + 2]), tc::round_tf32(u[i + 3]));
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            // ---- Pt = Xt K^T for both halves (A from tensor memory)
            if (tid == 0) {
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_ts(tb + TM_PT, tb + TM_XT + ks * 8, tc::sdesc_kstep(sK32, C, ks),
                               tc::idesc_tf32(128, 64), ks > 0);
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    tc::mma_ts(tb + TM_PS, tb + TM_XS + ks * 8, tc::sdesc_kstep(sK32, C, ks),
                               tc::idesc_tf32(128, 64), ks > 0);
                tc::commit(mb);
            }
            if (!mma_done()) { failed = true; break; }
            // ---- Rt = [0 | V]^T - Pt diag(Gamma); Xt *= Gamma_C
            {
                float p[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t src = my + (half ? TM_PS : TM_PT);
                    const uint32_t dst = SM_RT + half * 32768;
#pragma unroll
                    for (int c = 0; c < C; c += 32) {
                        tc::tmem_ld32(src + c, p);
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float r4[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int t = c + i + q;
                                const float vb = half ? Vs[t * D + tid] : 0.f;
                                r4[q] = tc::round_tf32(fmaf(-gt.eg[t], p[i + q], vb));
                            }
                            *reinterpret_cast<float4 *>(sm + dst + tc::sw128_f32(tid, c + i, D)) =
                                make_float4(r4[0], r4[1], r4[2], r4[3]);
                        }
                    }
                }
                const float gC = gt.eg[C - 1];
#pragma unroll
                for (int c = 0; c < 2 * D; c += 32) {
                    tc::tmem_ld32(my + TM_XT + c, p);
#pragma unroll
                    for (int i = 0; i < 32; ++i) p[i] *= gC;
                    tc::tmem_st32(my + TM_XT + c, p);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            __syncthreads();
            // ---- Xt += Rt U~   (M = 128, N = 128, K = 64) per half
            if (tid == 0) {
                tc::fence_after();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ss(tb + TM_XT, tc::sdesc_kstep(sRT, D, ks), tc::sdesc_kstep(sUT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    tc::mma_ss(tb + TM_XS, tc::sdesc_kstep(sRT + 32768, D, ks), tc::sdesc_kstep(sUT, D, ks),
                               tc::idesc_tf32(128, 128), 1);
                tc::commit(mb);
            }
            if (!mma_done()) { failed = true; break; }
        }
        if (failed) break;
        // ---- emit: T[i][m] = Xt_T[m][i], S[i][m] = Xt_S[m][i]; thread m owns column m
        {
            const size_t pair = ((size_t)l * tab.n_seg + s) * dm.H + h;
            float *To = a.T_out + pair * D * D + tid;
            float *So = a.S_out + pair * D * D + tid;
            float x[32];
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                tc::tmem_ld32(my + TM_XT + c, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) To[(size_t)(c + i) * D] = x[i];
                tc::tmem_ld32(my + TM_XS + c, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) So[(size_t)(c + i) * D] = x[i];
            }
        }
        tc::fence_before();
        __syncthreads();
    }
    if (failed && tid == 0) atomicOr(a.status, 1);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tb, TM_COLS);
}

int g_num_sms = 0;

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
    if (g_num_sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaMemsetAsync(a.work_counter, 0, 256, st);
    if (e != cudaSuccess) return e;
    const int grid = n_items < g_num_sms ? n_items : g_num_sms;
    if (a.dm.conv_k == 0) {
        e = cudaFuncSetAttribute(build_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
        if (e != cudaSuccess) return e;
        build_tc_kernel<0><<<grid, NT, SMEM_DYN, st>>>(a, tab);
    } else {
        e = cudaFuncSetAttribute(build_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
        if (e != cudaSuccess) return e;
        build_tc_kernel<4><<<grid, NT, SMEM_DYN, st>>>(a, tab);
    }
    return cudaGetLastError();
}

}  // namespace hypic
