/*
 * hypic.h -- C ABI of the linear-attention hot path of position-independent
 * caching (PIC) for hybrid-attention models, as described in the HYPIC pages
 * (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”, sections "线性层", "全注意力层" and "段并行";
 * article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”, paragraphs on linear layers, seam windows and segment-level
 * parallelism).
 *
 * The method.  A linear-attention layer keeps a state S (d_k x d_v, fp32 here)
 * per head that every token advances:
 *     S_t = A_t S_{t-1} + W_t ,          o_t = S_t^T q_t ,
 * in the gated-delta convention
 *     A_t = alpha_t (I - beta_t k_t k_t^T),   W_t = beta_t k_t v_t^T,
 * or one of the two named specialisations
 *     scalar decay (RetNet):        A_t = gamma_h I,      W_t = k_t v_t^T,
 *     diagonal gate (Mamba2/GLA):   A_t = diag(alpha_t),  W_t = k_t v_t^T,
 * or the delta rule with a per-channel decay (the pages name the KDA family
 * without its formula; read here as decay first, then erase and write):
 *     KDA:   A_t = (I - beta_t k_t k_t^T) diag(alpha_t),  W_t = beta_t k_t v_t^T.
 * Plain DeltaNet is gated delta with alpha = 1.
 * For a segment C the pair (T_C, S(C|0)) -- the ordered product of the
 * segment's transitions and its final state from zero -- depends only on the
 * segment's own tokens, so it is cached once ("线性层": cache the pair at the
 * segment's first prefill) and reused in any prefix through the composition
 * law S(C1 C2) = T(C2) S(C1) + S(C2).  The first w tokens of a segment (its
 * seam window, w = 8 by default, "全注意力层") are not cached: at reuse they
 * are re-run under the composed prefix state, advancing it and emitting their
 * per-token outputs.
 *
 * Three calls form the hot path; a fourth serves a segment's first prefill:
 *   hypic_segment_build   -- the cached pair of every segment body, all
 *                            segments x layers x heads in one launch (the
 *                            single-GPU stand-in for "段并行"'s scatter stage,
 *                            longest segment first as in its LPT schedule);
 *   hypic_compose         -- the running state over a request's segment order,
 *                            with each entry's seam re-run in the same pass;
 *   hypic_seam_advance    -- the seams alone, all entries in parallel, from
 *                            given prefix states;
 * and
 *   hypic_segment_forward -- the segment bodies' per-token outputs from a zero
 *                            state (the segment's first prefill), with or
 *                            without the pair.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All device pointers are caller-owned device memory; the library never
 *   allocates or frees device memory.  It keeps two kinds of device state,
 *   both static variables compiled into it (held by every GPU that loads the
 *   library until exit): one status word per device, into which compose and
 *   seam-advance kernels report a bounded wait that gave up
 *   (hypic_async_status), and the scratch block of
 *   hypic_segment_build_noalloc (hypic_noalloc_status).
 *   Host pointers (segment offsets, request order, descriptors) are read
 *   before the call returns and may be freed afterwards.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *   stream) and runs asynchronously; outputs are valid once the stream has
 *   reached the call.  Calls on the same stream are ordered.
 * - Every argument is validated on the host before anything is enqueued.  On
 *   any error nothing is launched, no output is touched, and the call returns
 *   a nonzero hypic_status; hypic_last_error() then describes it (per thread).
 *   A failed launch returns HYPIC_ERR_CUDA.
 * - Layouts are row-major and packed, layer-major, token-major:
 *     q, k, v   [L][N][H][d]   (in_dtype; raw pre-convolution tokens when
 *                               conv_k > 0)
 *     alpha     gated delta [L][N][H]; diagonal gate and KDA [L][N][H][d_k];
 *               scalar decay [L][H] (one gamma per head), all in in_dtype
 *     beta      [L][N][H] in in_dtype (gated delta and KDA; NULL otherwise)
 *     conv_w    fp32 [L][3][H][d][conv_k]: channels of q, k, v; tap j
 *               multiplies the token j positions earlier
 *     T         gated delta and KDA fp32 [L][n_seg][H][d_k][d_k];
 *               diagonal gate fp32 [L][n_seg][H][d_k] (the diagonal);
 *               scalar decay fp32 [L][n_seg][H] (the scalar)
 *     S, states fp32 [..][d_k][d_v], row = key channel
 *   Token, alpha and beta pointers must be 16-byte aligned, as must every
 *   fp32 output.  d_k == d_v is required.
 * - Segments are contiguous token ranges of the packed token axis given by
 *   host offsets seg_off[0..n_seg] (non-decreasing, seg_off[n_seg] <= N).  A
 *   request is a host array order[0..n_order) of segment indices; the same
 *   segment may appear more than once.  n_seg and n_order are at most
 *   HYPIC_MAX_SEGMENTS.
 */
#ifndef HYPIC_H
#define HYPIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HYPIC_ABI_VERSION 4
#define HYPIC_MAX_SEGMENTS 2048

typedef struct CUstream_st *hypic_stream; /* same type as cudaStream_t */

typedef enum hypic_status {
    HYPIC_OK = 0,
    HYPIC_ERR_INVALID_ARG = 1,  /* NULL or misaligned pointer, bad enum */
    HYPIC_ERR_SHAPE = 2,        /* sizes, offsets or order out of range */
    HYPIC_ERR_DTYPE = 3,        /* unknown dtype */
    HYPIC_ERR_UNSUPPORTED = 4,  /* valid request this build does not serve */
    HYPIC_ERR_WORKSPACE = 5,    /* workspace missing, misaligned or too small */
    HYPIC_ERR_CUDA = 6,         /* the CUDA runtime reported an error */
    HYPIC_ERR_TIMEOUT = 7       /* a bounded device-side wait gave up */
} hypic_status;

typedef enum hypic_mode {
    HYPIC_GATED_DELTA = 0,   /* A_t = alpha_t (I - beta_t k k^T), W = beta k v^T */
    HYPIC_SCALAR_DECAY = 1,  /* A_t = gamma_h I,                  W = k v^T      */
    HYPIC_DIAG_GATE = 2,     /* A_t = diag(alpha_t),              W = k v^T      */
    HYPIC_KDA = 3            /* A_t = (I - beta_t k k^T) diag(alpha_t), W = beta k v^T */
} hypic_mode;

/* Activation between the causal conv and the L2 normalisation (conv_k > 0). */
typedef enum hypic_act {
    HYPIC_ACT_NONE = 0,  /* conv output used as is */
    HYPIC_ACT_SILU = 1   /* x * sigmoid(x) on q, k and v after the conv */
} hypic_act;

typedef enum hypic_dtype {
    HYPIC_F32 = 0,
    HYPIC_BF16 = 1
} hypic_dtype;

/* Shape and variant of one stack of linear-attention layers. */
typedef struct hypic_desc {
    int32_t n_layers;  /* L >= 1 */
    int32_t n_heads;   /* H >= 1 */
    int32_t d_k;       /* key width: 16, 32, 64 or 128 */
    int32_t d_v;       /* value width: must equal d_k */
    int32_t seam_w;    /* seam window w in [0, 64]; 0 = no seams */
    int32_t conv_k;    /* causal depthwise conv taps: 0 (none) or 2..4 */
    int32_t mode;      /* hypic_mode */
    int32_t in_dtype;  /* hypic_dtype of q, k, v, alpha, beta */
    int32_t conv_act;  /* hypic_act after the conv; must be HYPIC_ACT_NONE when conv_k == 0 */
} hypic_desc;

/* The packed per-token inputs of a request's tokens (all device pointers). */
typedef struct hypic_tokens {
    const void *q;       /* [L][N][H][d_k]; needed for seam outputs only */
    const void *k;       /* [L][N][H][d_k] */
    const void *v;       /* [L][N][H][d_v] */
    const void *alpha;   /* see layouts above */
    const void *beta;    /* [L][N][H] (gated delta only) */
    const float *conv_w; /* fp32 [L][3][H][d][conv_k] when conv_k > 0 */
    int64_t n_tokens;    /* N, < 2^31 */
} hypic_tokens;

/* ABI version of the loaded library (HYPIC_ABI_VERSION). */
int hypic_version(void);

/* Description of the last error on the calling thread ("" if none). */
const char *hypic_last_error(void);

/*
 * Bytes of device workspace hypic_segment_build needs (always > 0, a
 * multiple of 256).  The workspace carries the build's device status word;
 * it need not be initialised and may be reused by consecutive calls on one
 * stream.
 */
size_t hypic_workspace_size(const hypic_desc *desc);

/*
 * Device status of a workspace after the builds that used it: waits for
 * `stream`, then returns HYPIC_OK, or HYPIC_ERR_TIMEOUT if a bounded
 * device-side wait of the build gave up (its outputs are then incomplete; the
 * kernel returned instead of hanging).  The next build on the workspace
 * clears the word.
 */
int hypic_workspace_status(const void *workspace, hypic_stream stream);

/*
 * Device status of the calls that take no workspace (hypic_compose,
 * hypic_seam_advance) on the current device: waits for `stream`, then
 * returns HYPIC_OK, or HYPIC_ERR_TIMEOUT if one of their kernels' bounded
 * device-side waits gave up since the last query (that call's outputs are
 * incomplete; the kernel returned instead of hanging), and clears the word.
 * The word is shared by every such call on the device, whatever the stream:
 * a give-up is reported to whichever caller queries first.
 */
int hypic_async_status(hypic_stream stream);

/*
 * Segment forward: the per-token outputs of every segment body computed from
 * a zero state -- the segment's own first prefill, the main forward that the
 * pair is cached alongside (HYPIC pages: article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首 Token 延迟降低 3.25 倍，实现位置无关缓存”,
 * sections "线性层" and "段并行"; article “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention Models”,
 * linear-layer and segment-parallelism paragraphs) -- and, optionally, the
 * pair itself:
 *     o_out[l][t][h][:] = S_t^T q_t  for every body token t of every segment
 *         (S_t the zero-initial state after t; the rows of seam tokens are
 *         left untouched -- their outputs come from hypic_compose);
 *     T_out, S_out exactly as hypic_segment_build, each optional (NULL skips
 *         it: with both NULL this is the plain forward).
 * q is required.  Runs on the exact-fp32 token-serial build for every mode,
 * width and dtype (no tensor cores).  o_out: fp32 [L][N][H][d_v], 16-byte
 * aligned; no workspace.
 */
int hypic_segment_forward(const hypic_desc *desc, const hypic_tokens *tok,
                          const int64_t *seg_off, int32_t n_seg,
                          float *o_out, float *T_out, float *S_out,
                          hypic_stream stream);

/*
 * Self-test of the bounded device-side wait that every pipelined kernel
 * uses (so that a missing arrival ends a CTA instead of hanging the GPU):
 * clears the workspace status word and launches one CTA on `stream` in which
 * one thread waits on an mbarrier that nothing completes, giving up after
 * max_cycles SM cycles and raising the CTA's abort flag, while a thread of
 * another warp, waiting on the same barrier with a 64x longer limit, must
 * leave as soon as it sees the flag.  hypic_workspace_status then returns
 * HYPIC_ERR_TIMEOUT with status 3 (1: the flag was raised; 2: the second
 * waiter left without the phase completing).  The device stays usable.
 * max_cycles in [1, 2^34]; workspace as for hypic_segment_build, or NULL to
 * report through (after clearing) the device status word that
 * hypic_async_status reads.
 */
int hypic_selftest_bounded_wait(void *workspace, int64_t max_cycles, hypic_stream stream);

/*
 * Segment build: for every segment s, layer l and head h, the cached pair of
 * the segment's body -- the segment's tokens after its first min(w, len)
 * seam tokens -- computed from a zero state:
 *     T[l][s][h] = A_{n} ... A_{1}     (ordered product over the body)
 *     S[l][s][h] = S(body | 0)
 * (HYPIC pages: "线性层" -- the pair depends only on the segment's own tokens
 * and is cached at its first prefill; "全注意力层" -- seam tokens are not
 * cached.)  An empty body yields (I, 0).  With conv_k > 0 the body's q/k/v
 * are the causal convolution of the raw tokens (history inside the segment;
 * requires seam_w >= conv_k - 1 so that bodies stay prefix-independent)
 * followed by per-head L2 normalisation of k.
 *
 * All segments x layers x heads run in one launch, longest body first.
 * T_out/S_out: layouts above.  workspace: device, 256-byte aligned, at least
 * hypic_workspace_size(desc) bytes, not used concurrently by another call.
 */
int hypic_segment_build(const hypic_desc *desc, const hypic_tokens *tok,
                        const int64_t *seg_off, int32_t n_seg,
                        float *T_out, float *S_out,
                        void *workspace, size_t workspace_bytes,
                        hypic_stream stream);

/*
 * Segment build without a caller-provided workspace (the HYPIC pages have no
 * counterpart; this is a library convenience).  For callers that cannot
 * allocate device memory -- e.g. a plugin inside a host inference engine that
 * owns all device memory and hands its kernels only input and output buffers,
 * or a latency-critical path where cudaMalloc's possible device
 * synchronisation is not allowed.  Computes exactly what hypic_segment_build
 * computes, with the same arguments minus the workspace.
 *
 * The scratch is a 256-byte block compiled into the library (a static device
 * array that every GPU loading the library keeps until process exit); a
 * request needing more scratch than that is rejected with
 * HYPIC_ERR_WORKSPACE.  The first call on a device looks up the block's
 * device address (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture.  All calls share the block and it
 * keeps the last call's contents (the build clears what must start at zero):
 * calls whose work overlaps on the GPU race on it, status word included.
 * Nothing is allocated.
 */
int hypic_segment_build_noalloc(const hypic_desc *desc, const hypic_tokens *tok,
                                const int64_t *seg_off, int32_t n_seg,
                                float *T_out, float *S_out, hypic_stream stream);

/*
 * Device status of the last hypic_segment_build_noalloc on the current
 * device, as hypic_workspace_status reports it for a workspace: waits for
 * `stream`, then HYPIC_OK or HYPIC_ERR_TIMEOUT (a bounded device-side wait of
 * that build gave up).  The word lives in the shared static scratch block, so
 * overlapping no-alloc builds share it too.
 */
int hypic_noalloc_status(hypic_stream stream);

/*
 * Compose: the running state of every (layer, head) over the request
 * order[0..n_order), starting from S_init (NULL = zero):
 *     for e in 0..n_order-1, s = order[e]:
 *         S_prefix_out[l][e][h] = S                      (if non-NULL)
 *         if seam_w > 0: re-run the first min(w, len_s) tokens of s from S,
 *             writing o_out[l][e][j][h][:] = S_j^T q_j and advancing S
 *         S = T[l][s][h] S + S[l][s][h]                  (composition law)
 *     S_final[l][h] = S
 * (HYPIC pages: "线性层" -- left-multiply by T_C then add; "全注意力层" --
 * seams re-run under the full prefix, advancing the running state and passing
 * each seam token's output up.)  With conv_k > 0 a seam token's convolution
 * history is the previous entry's last raw tokens (zero before the request
 * start): the articles' "convolution state warm-up".
 *
 * T, S: the cache, as written by hypic_segment_build with the same desc and
 * n_seg.  tok: the request's tokens (may be NULL when seam_w == 0).
 * o_out: fp32 [L][n_order][w][H][d_v]; rows past a short seam are zeroed
 * (NULL allowed when seam_w == 0).  S_prefix_out: fp32 [L][n_order][H][d_k][d_v]
 * or NULL.  S_final: fp32 [L][H][d_k][d_v], may alias S_init.
 * n_order == 0 copies S_init (or zero) to S_final.
 */
int hypic_compose(const hypic_desc *desc, const hypic_tokens *tok,
                  const int64_t *seg_off, int32_t n_seg,
                  const int32_t *order, int32_t n_order,
                  const float *T, const float *S, const float *S_init,
                  float *S_prefix_out, float *S_final, float *o_out,
                  hypic_stream stream);

/*
 * Seam advance: every entry's seam re-run from a given state, all entries in
 * parallel (the seams of a request are independent once their prefix states
 * are known, e.g. from hypic_compose's S_prefix_out):
 *     for each e, l, h:  S = S_in[l][e][h];
 *         for the first min(w, len) tokens of order[e]: advance S, emit o
 *         o_out[l][e][j][h][:] = S_j^T q_j ;  S_out[l][e][h] = S
 * (HYPIC pages: "全注意力层" -- the linear layer computes the seam window's
 * T and S on the fly while advancing the running state and forwards each seam
 * token's output.)  Same conv history rule as hypic_compose.
 * S_in: fp32 [L][n_order][H][d_k][d_v]; o_out: fp32 [L][n_order][w][H][d_v];
 * S_out: same layout as S_in or NULL; S_out may alias S_in.
 * Gated delta seams (alpha = 1: DeltaNet) are computed in closed form, all
 * tokens of a seam in one pass over S in fp32 (equal to the token-by-token
 * recurrence up to rounding); the other modes step token by token.  At
 * d = 128 with seam_w <= 8 the kernel is persistent and pipelined; its
 * device-side waits are bounded, and if one gives up the outputs are left
 * incomplete instead of the kernel hanging and hypic_async_status reports it.
 */
int hypic_seam_advance(const hypic_desc *desc, const hypic_tokens *tok,
                       const int64_t *seg_off, int32_t n_seg,
                       const int32_t *order, int32_t n_order,
                       const float *S_in, float *o_out, float *S_out,
                       hypic_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* HYPIC_H */
