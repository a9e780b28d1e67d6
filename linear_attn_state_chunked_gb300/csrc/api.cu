// api.cu -- the C ABI of include/hypic.h: host-side validation, the
// longest-first work order of the build, and kernel launches on the caller's
// stream.  No device memory is allocated here.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "kernels.h"

using namespace hypic;

namespace {

thread_local char g_err[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_desc(const hypic_desc *d)
{
    if (!d) return fail(HYPIC_ERR_INVALID_ARG, "desc is NULL");
    if (d->mode < HYPIC_GATED_DELTA || d->mode > HYPIC_KDA)
        return fail(HYPIC_ERR_INVALID_ARG, "unknown mode %d", d->mode);
    if (d->in_dtype != HYPIC_F32 && d->in_dtype != HYPIC_BF16)
        return fail(HYPIC_ERR_DTYPE, "unknown in_dtype %d", d->in_dtype);
    if (d->n_layers < 1 || d->n_heads < 1 || (int64_t)d->n_layers * d->n_heads > 65536)
        return fail(HYPIC_ERR_SHAPE, "n_layers=%d n_heads=%d out of range", d->n_layers, d->n_heads);
    if (d->d_k != d->d_v)
        return fail(HYPIC_ERR_UNSUPPORTED, "d_k (%d) != d_v (%d)", d->d_k, d->d_v);
    if (d->d_k != 16 && d->d_k != 32 && d->d_k != 64 && d->d_k != 128)
        return fail(HYPIC_ERR_UNSUPPORTED, "d_k=%d not in {16, 32, 64, 128}", d->d_k);
    if (d->seam_w < 0 || d->seam_w > 64)
        return fail(HYPIC_ERR_SHAPE, "seam_w=%d not in [0, 64]", d->seam_w);
    if (d->conv_k != 0 && (d->conv_k < 2 || d->conv_k > 4))
        return fail(HYPIC_ERR_UNSUPPORTED, "conv_k=%d not in {0, 2, 3, 4}", d->conv_k);
    if (d->conv_act != HYPIC_ACT_NONE && d->conv_act != HYPIC_ACT_SILU)
        return fail(HYPIC_ERR_INVALID_ARG, "unknown conv_act %d", d->conv_act);
    if (d->conv_act != HYPIC_ACT_NONE && d->conv_k == 0)
        return fail(HYPIC_ERR_INVALID_ARG, "conv_act %d without a conv (conv_k = 0)", d->conv_act);
    if (d->conv_k > 0 && d->seam_w < d->conv_k - 1)
        return fail(HYPIC_ERR_UNSUPPORTED,
                    "conv_k=%d needs seam_w >= %d so that cached bodies are prefix-independent",
                    d->conv_k, d->conv_k - 1);
    return HYPIC_OK;
}

int check_tokens(const hypic_desc *d, const hypic_tokens *t, bool need_q)
{
    if (!t) return fail(HYPIC_ERR_INVALID_ARG, "tokens is NULL");
    if (t->n_tokens < 0 || t->n_tokens >= ((int64_t)1 << 31))
        return fail(HYPIC_ERR_SHAPE, "n_tokens=%lld out of range", (long long)t->n_tokens);
    struct { const void *p; const char *name; bool need; } ps[] = {
        {t->q, "q", need_q},
        {t->k, "k", true},
        {t->v, "v", true},
        {t->alpha, "alpha", true},
        {t->beta, "beta", d->mode == HYPIC_GATED_DELTA || d->mode == HYPIC_KDA},
        {t->conv_w, "conv_w", d->conv_k > 0},
    };
    for (auto &x : ps) {
        if (!x.need) continue;
        if (!x.p) return fail(HYPIC_ERR_INVALID_ARG, "tokens.%s is NULL", x.name);
        if (!aligned(x.p, 16)) return fail(HYPIC_ERR_INVALID_ARG, "tokens.%s is not 16-byte aligned", x.name);
    }
    return HYPIC_OK;
}

int check_segments(const int64_t *seg_off, int32_t n_seg, int64_t n_tokens)
{
    if (n_seg < 0 || n_seg > HYPIC_MAX_SEGMENTS)
        return fail(HYPIC_ERR_SHAPE, "n_seg=%d not in [0, %d]", n_seg, HYPIC_MAX_SEGMENTS);
    if (!seg_off) return fail(HYPIC_ERR_INVALID_ARG, "seg_off is NULL");
    if (seg_off[0] < 0) return fail(HYPIC_ERR_SHAPE, "seg_off[0]=%lld < 0", (long long)seg_off[0]);
    for (int32_t i = 0; i < n_seg; ++i)
        if (seg_off[i + 1] < seg_off[i])
            return fail(HYPIC_ERR_SHAPE, "seg_off decreases at %d (%lld > %lld)", i,
                        (long long)seg_off[i], (long long)seg_off[i + 1]);
    if (seg_off[n_seg] > n_tokens)
        return fail(HYPIC_ERR_SHAPE, "seg_off[n_seg]=%lld > n_tokens=%lld", (long long)seg_off[n_seg],
                    (long long)n_tokens);
    return HYPIC_OK;
}

int check_order(const int32_t *order, int32_t n_order, int32_t n_seg)
{
    if (n_order < 0 || n_order > HYPIC_MAX_SEGMENTS)
        return fail(HYPIC_ERR_SHAPE, "n_order=%d not in [0, %d]", n_order, HYPIC_MAX_SEGMENTS);
    if (n_order > 0 && !order) return fail(HYPIC_ERR_INVALID_ARG, "order is NULL");
    for (int32_t i = 0; i < n_order; ++i)
        if (order[i] < 0 || order[i] >= n_seg)
            return fail(HYPIC_ERR_SHAPE, "order[%d]=%d not in [0, %d)", i, order[i], n_seg);
    return HYPIC_OK;
}

int check_out(const void *p, const char *name)
{
    if (!p) return fail(HYPIC_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, 16)) return fail(HYPIC_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return HYPIC_OK;
}

Dims make_dims(const hypic_desc *d)
{
    return Dims{d->n_layers, d->n_heads, d->d_k, d->seam_w, d->conv_k, d->mode, d->in_dtype, d->conv_act};
}

TokPtrs make_tok(const hypic_tokens *t)
{
    TokPtrs p{};
    if (t) {
        p.q = t->q; p.k = t->k; p.v = t->v; p.alpha = t->alpha; p.beta = t->beta;
        p.conv_w = t->conv_w;
        p.N = (int32_t)t->n_tokens;
    }
    return p;
}

void fill_offsets(SegTable &tab, const int64_t *seg_off, int32_t n_seg)
{
    tab.n_seg = n_seg;
    for (int32_t i = 0; i <= n_seg; ++i) tab.off[i] = (int32_t)seg_off[i];
}

// Request table of a build: segment offsets, and the items' order longest
// body first (ties: lower index first), the greedy LPT order.
void fill_build_table(SegTable &tab, const int64_t *seg_off, int32_t n_seg, int w)
{
    fill_offsets(tab, seg_off, n_seg);
    auto body = [&](int s) {
        const int64_t len = seg_off[s + 1] - seg_off[s];
        return len - std::min<int64_t>(w, len);
    };
    std::vector<int32_t> idx(n_seg);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return body(a) > body(b); });
    for (int32_t i = 0; i < n_seg; ++i) tab.perm[i] = idx[i];
    tab.n_perm = n_seg;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(HYPIC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One status word per device for the calls that take no workspace (compose,
// seam advance): a kernel whose bounded device-side wait gives up ORs 1 into
// it, and hypic_async_status reads and clears it.  The word is a static device
// variable (every GPU that loads the library holds it until exit); its device
// address is looked up once per device, with that device current.
__device__ int g_async_status;
constexpr int kMaxDevices = 64;
std::once_flag g_status_once[kMaxDevices];
int *g_status_ptr[kMaxDevices];
cudaError_t g_status_err[kMaxDevices];

int async_status_ptr(int **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(HYPIC_ERR_UNSUPPORTED, "device %d beyond the %d devices served", dev, kMaxDevices);
    std::call_once(g_status_once[dev], [dev]() {
        void *p = nullptr;
        g_status_err[dev] = cudaGetSymbolAddress(&p, g_async_status);
        g_status_ptr[dev] = static_cast<int *>(p);
    });
    if (g_status_err[dev] != cudaSuccess || !g_status_ptr[dev])
        return cuda_fail(g_status_err[dev], "status word address");
    *out = g_status_ptr[dev];
    return HYPIC_OK;
}

}  // namespace

namespace hypic {
// The device status word of the current device (api.cu); for selftest.cu.
int async_status_word(int **out) { return async_status_ptr(out); }
}  // namespace hypic

namespace hypic {
int report_error(int code, const char *msg) { return fail(code, "%s", msg); }
}  // namespace hypic

extern "C" {

int hypic_version(void) { return HYPIC_ABI_VERSION; }

const char *hypic_last_error(void) { return g_err; }

size_t hypic_workspace_size(const hypic_desc *desc)
{
    (void)desc;
    return 256;
}

int hypic_segment_build(const hypic_desc *desc, const hypic_tokens *tok, const int64_t *seg_off,
                        int32_t n_seg, float *T_out, float *S_out, void *workspace,
                        size_t workspace_bytes, hypic_stream stream)
{
    g_err[0] = 0;
    int rc;
    if ((rc = check_desc(desc))) return rc;
    if ((rc = check_tokens(desc, tok, false))) return rc;
    if ((rc = check_segments(seg_off, n_seg, tok->n_tokens))) return rc;
    if ((rc = check_out(T_out, "T_out"))) return rc;
    if ((rc = check_out(S_out, "S_out"))) return rc;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < hypic_workspace_size(desc))
        return fail(HYPIC_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes",
                    hypic_workspace_size(desc));
    // every build starts from a clear status word, whichever kernel runs
    {
        cudaError_t e = cudaMemsetAsync(static_cast<char *>(workspace) + 128, 0, sizeof(int), (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "status word clear");
    }
    if (n_seg == 0) return HYPIC_OK;

    static thread_local SegTable tab;
    fill_build_table(tab, seg_off, n_seg, desc->seam_w);

    BuildArgs a{};
    a.dm = make_dims(desc);
    a.tok = make_tok(tok);
    a.T_out = T_out;
    a.S_out = S_out;
    a.status = reinterpret_cast<int *>(static_cast<char *>(workspace) + 128);
    // Gated delta at d = 128 with bf16 inputs runs on the tensor cores (tf32
    // products, 2e-3 class); everything else, including every fp32-input
    // request (1e-5 class), runs the token-serial fp32 recurrence.
    cudaError_t e = build_tc_supported(a.dm) ? launch_build_tc(a, tab, (cudaStream_t)stream)
                                             : launch_build_rec(a, tab, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "segment build launch");
    return HYPIC_OK;
}

int hypic_segment_forward(const hypic_desc *desc, const hypic_tokens *tok, const int64_t *seg_off,
                          int32_t n_seg, float *o_out, float *T_out, float *S_out, hypic_stream stream)
{
    g_err[0] = 0;
    int rc;
    if ((rc = check_desc(desc))) return rc;
    if ((rc = check_tokens(desc, tok, true))) return rc;
    if ((rc = check_segments(seg_off, n_seg, tok->n_tokens))) return rc;
    if ((rc = check_out(o_out, "o_out"))) return rc;
    if (T_out && !aligned(T_out, 16)) return fail(HYPIC_ERR_INVALID_ARG, "T_out is not 16-byte aligned");
    if (S_out && !aligned(S_out, 16)) return fail(HYPIC_ERR_INVALID_ARG, "S_out is not 16-byte aligned");
    if (n_seg == 0) return HYPIC_OK;

    static thread_local SegTable tab;
    fill_build_table(tab, seg_off, n_seg, desc->seam_w);
    BuildArgs a{};
    a.dm = make_dims(desc);
    a.tok = make_tok(tok);
    a.T_out = T_out;
    a.S_out = S_out;
    a.o_out = o_out;
    // the outputs come from the exact-fp32 token-serial build, for every mode
    cudaError_t e = launch_build_rec(a, tab, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "segment forward launch");
    return HYPIC_OK;
}

int hypic_workspace_status(const void *workspace, hypic_stream stream)
{
    g_err[0] = 0;
    if (!workspace || !aligned(workspace, 256))
        return fail(HYPIC_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int word = 0;
    e = cudaMemcpy(&word, static_cast<const char *>(workspace) + 128, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word != 0) return fail(HYPIC_ERR_TIMEOUT, "a device-side wait of the last build gave up (status %d)", word);
    return HYPIC_OK;
}

int hypic_async_status(hypic_stream stream)
{
    g_err[0] = 0;
    int *word = nullptr;
    int rc;
    if ((rc = async_status_ptr(&word))) return rc;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int v = 0;
    e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (v == 0) return HYPIC_OK;
    e = cudaMemset(word, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return fail(HYPIC_ERR_TIMEOUT, "a device-side wait of a compose or seam-advance call gave up (status %d)", v);
}

int hypic_compose(const hypic_desc *desc, const hypic_tokens *tok, const int64_t *seg_off,
                  int32_t n_seg, const int32_t *order, int32_t n_order, const float *T,
                  const float *S, const float *S_init, float *S_prefix_out, float *S_final,
                  float *o_out, hypic_stream stream)
{
    g_err[0] = 0;
    int rc;
    if ((rc = check_desc(desc))) return rc;
    const bool seams = desc->seam_w > 0 && n_order > 0;
    if (seams && (rc = check_tokens(desc, tok, true))) return rc;
    if ((rc = check_segments(seg_off, n_seg, seams ? tok->n_tokens : INT64_MAX))) return rc;
    if ((rc = check_order(order, n_order, n_seg))) return rc;
    if (n_order > 0) {
        if ((rc = check_out(T, "T"))) return rc;
        if ((rc = check_out(S, "S"))) return rc;
    }
    if (S_init && !aligned(S_init, 16)) return fail(HYPIC_ERR_INVALID_ARG, "S_init is not 16-byte aligned");
    if (S_prefix_out && !aligned(S_prefix_out, 16))
        return fail(HYPIC_ERR_INVALID_ARG, "S_prefix_out is not 16-byte aligned");
    if ((rc = check_out(S_final, "S_final"))) return rc;
    if (seams && (rc = check_out(o_out, "o_out"))) return rc;

    static thread_local SegTable tab;
    fill_offsets(tab, seg_off, n_seg);
    for (int32_t i = 0; i < n_order; ++i) tab.perm[i] = order[i];
    tab.n_perm = n_order;

    ComposeArgs a{};
    a.dm = make_dims(desc);
    if (!seams) a.dm.w = 0;
    a.tok = make_tok(seams ? tok : nullptr);
    a.T = T;
    a.S = S;
    a.S_init = S_init;
    a.S_prefix = S_prefix_out;
    a.S_final = S_final;
    a.o_out = o_out;
    if ((rc = async_status_ptr(&a.status))) return rc;
    cudaError_t e = launch_compose(a, tab, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "compose launch");
    return HYPIC_OK;
}

int hypic_seam_advance(const hypic_desc *desc, const hypic_tokens *tok, const int64_t *seg_off,
                       int32_t n_seg, const int32_t *order, int32_t n_order, const float *S_in,
                       float *o_out, float *S_out, hypic_stream stream)
{
    g_err[0] = 0;
    int rc;
    if ((rc = check_desc(desc))) return rc;
    if ((rc = check_tokens(desc, tok, true))) return rc;
    if ((rc = check_segments(seg_off, n_seg, tok->n_tokens))) return rc;
    if ((rc = check_order(order, n_order, n_seg))) return rc;
    if (desc->seam_w == 0 || n_order == 0) return HYPIC_OK;
    if ((rc = check_out(S_in, "S_in"))) return rc;
    if ((rc = check_out(o_out, "o_out"))) return rc;
    if (S_out && !aligned(S_out, 16)) return fail(HYPIC_ERR_INVALID_ARG, "S_out is not 16-byte aligned");

    static thread_local SegTable tab;
    fill_offsets(tab, seg_off, n_seg);
    for (int32_t i = 0; i < n_order; ++i) tab.perm[i] = order[i];
    tab.n_perm = n_order;

    SeamArgs a{};
    a.dm = make_dims(desc);
    a.tok = make_tok(tok);
    a.S_in = S_in;
    a.o_out = o_out;
    a.S_out = S_out;
    if ((rc = async_status_ptr(&a.status))) return rc;
    cudaError_t e = launch_seam(a, tab, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "seam advance launch");
    return HYPIC_OK;
}

}  // extern "C"
