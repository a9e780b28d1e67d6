/*
 * oracle.c -- plain, sequential fp64 CPU reference for the linear-attention
 * hot path of position-independent caching (HYPIC).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Everything here is the plain definition, token by token, in double
 * precision, with no chunking, blocking or reordering:
 *
 *  - The recurrence (article “小红书联合北大、上交提出 HYPIC：混合注意力大模型首
 *    Token 延迟降低 3.25 倍，实现位置无关缓存”, section "线性层"; article
 *    “Xiaohongshu, Peking University, Shanghai Jiao Tong University Unveil
 *    HYPIC to Slash First Token Latency by 3.25x in Hybrid Attention
 *    Models”, paragraph on linear layers): per token the state is
 *    advanced by the transition A_t and a rank-1 write,
 *        S_t = A_t S_{t-1} + W_t ,   o_t = S_t^T q_t ,
 *    in the gated-delta convention
 *        A_t = alpha_t (I - beta_t k_t k_t^T),   W_t = beta_t k_t v_t^T,
 *    with the two named specialisations
 *        scalar decay (RetNet):    A_t = gamma I,          W_t = k_t v_t^T
 *        diagonal gate (Mamba2/GLA): A_t = diag(alpha_t),  W_t = k_t v_t^T,
 *    and the delta rule with a per-channel decay (the KDA family, named by
 *    the first article's "线性层" section without a formula; read as decay
 *    first, then erase and write):
 *        KDA:  A_t = (I - beta_t k_t k_t^T) diag(alpha_t),  W_t = beta_t k_t v_t^T.
 *  - The cached pair of a segment C (same sections): T_C is the ordered
 *    product A_L ... A_1 of the segment's transitions, applied one token at a
 *    time to T = I; S(C|0) is the recurrence's final state from S = 0.
 *  - Composition (same sections): S(C1 C2) = T(C2) S(C1) + S(C2), a dense
 *    matrix product and a sum.
 *
 * Layouts (all row-major, contiguous, one "chain" = one independent
 * (layer, head) problem, chains stacked on the outermost axis):
 *    q, k : [n_chain][n][dk]      v : [n_chain][n][dv]
 *    a    : mode 0/1: [n_chain][n]   mode 2/3: [n_chain][n][dk]
 *    b    : [n_chain][n]  (modes 0 and 3; may be NULL otherwise)
 *    S    : [n_chain][dk][dv]      T : [n_chain][dk][dk]
 * Independent chains run in parallel under OpenMP; each chain is a plain
 * sequential loop.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { ORC_GATED_DELTA = 0, ORC_SCALAR_DECAY = 1, ORC_DIAG_GATE = 2, ORC_KDA = 3 };

/* S <- A_t S + W_t for one token.  X is [dk][ncol]; v may be NULL (then the
 * write term is absent, which is how T is propagated).  u is scratch [ncol]. */
static void apply_token(int mode, int dk, int ncol, double *X,
                        const double *k, const double *v, const double *a,
                        double b, double *u)
{
    if (mode == ORC_GATED_DELTA) {
        double alpha = a[0];
        /* u = X^T k */
        for (int j = 0; j < ncol; ++j) u[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) u[j] += k[i] * X[(size_t)i * ncol + j];
        /* X = alpha (X - b k u^T) + b k v^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) {
                double x = X[(size_t)i * ncol + j];
                x = alpha * (x - b * k[i] * u[j]);
                if (v) x += b * k[i] * v[j];
                X[(size_t)i * ncol + j] = x;
            }
    } else if (mode == ORC_SCALAR_DECAY) {
        double gamma = a[0];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) {
                double x = gamma * X[(size_t)i * ncol + j];
                if (v) x += k[i] * v[j];
                X[(size_t)i * ncol + j] = x;
            }
    } else if (mode == ORC_KDA) {
        /* X = diag(alpha) X, then X = X - b k (X^T k)^T + b k v^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) X[(size_t)i * ncol + j] *= a[i];
        for (int j = 0; j < ncol; ++j) u[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) u[j] += k[i] * X[(size_t)i * ncol + j];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) {
                double x = X[(size_t)i * ncol + j] - b * k[i] * u[j];
                if (v) x += b * k[i] * v[j];
                X[(size_t)i * ncol + j] = x;
            }
    } else { /* ORC_DIAG_GATE */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < ncol; ++j) {
                double x = a[i] * X[(size_t)i * ncol + j];
                if (v) x += k[i] * v[j];
                X[(size_t)i * ncol + j] = x;
            }
    }
}

static const double *alpha_at(int mode, int dk, int64_t n, const double *a,
                              int c, int64_t t)
{
    if (mode == ORC_DIAG_GATE || mode == ORC_KDA) return a + ((size_t)c * n + t) * dk;
    return a + (size_t)c * n + t;
}

/*
 * Run the recurrence over n tokens for every chain, starting from S (in/out).
 * If o != NULL, o[c][t] = S_t^T q_t after token t's update.
 * If n_rec > 0, S_rec[c][r] is the state just BEFORE token rec_at[r]
 * (rec_at[r] == n records the final state).
 */
int orc_recurrence(int mode, int dk, int dv, int64_t n, int n_chain,
                   const double *q, const double *k, const double *v,
                   const double *a, const double *b, double *S, double *o,
                   int n_rec, const int64_t *rec_at, double *S_rec)
{
    if (dk <= 0 || dv <= 0 || n < 0 || n_chain < 0) return 1;
    for (int r = 0; r < n_rec; ++r)
        if (rec_at[r] < 0 || rec_at[r] > n) return 2;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int c = 0; c < n_chain; ++c) {
        double *X = S + (size_t)c * dk * dv;
        double *u = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!u) { err = 3; continue; }
        for (int64_t t = 0; t <= n; ++t) {
            for (int r = 0; r < n_rec; ++r)
                if (rec_at[r] == t)
                    memcpy(S_rec + ((size_t)c * n_rec + r) * dk * dv, X,
                           sizeof(double) * (size_t)dk * dv);
            if (t == n) break;
            const double *kt = k + ((size_t)c * n + t) * dk;
            const double *vt = v + ((size_t)c * n + t) * dv;
            double bt = (mode == ORC_GATED_DELTA || mode == ORC_KDA) ? b[(size_t)c * n + t] : 0.0;
            apply_token(mode, dk, dv, X, kt, vt, alpha_at(mode, dk, n, a, c, t), bt, u);
            if (o) {
                const double *qt = q + ((size_t)c * n + t) * dk;
                double *ot = o + ((size_t)c * n + t) * dv;
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += X[(size_t)i * dv + j] * qt[i];
                    ot[j] = acc;
                }
            }
        }
        free(u);
    }
    return err;
}

/*
 * The cached pair of each chain's n tokens: T = A_n ... A_1 (applied token by
 * token to the identity) and S = final state from zero.
 */
int orc_pair(int mode, int dk, int dv, int64_t n, int n_chain,
             const double *k, const double *v, const double *a,
             const double *b, double *T, double *S)
{
    if (dk <= 0 || dv <= 0 || n < 0 || n_chain < 0) return 1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int c = 0; c < n_chain; ++c) {
        double *Tc = T + (size_t)c * dk * dk;
        double *Sc = S + (size_t)c * dk * dv;
        int w = dk > dv ? dk : dv;
        double *u = (double *)malloc(sizeof(double) * (size_t)w);
        if (!u) { err = 3; continue; }
        memset(Tc, 0, sizeof(double) * (size_t)dk * dk);
        for (int i = 0; i < dk; ++i) Tc[(size_t)i * dk + i] = 1.0;
        memset(Sc, 0, sizeof(double) * (size_t)dk * dv);
        for (int64_t t = 0; t < n; ++t) {
            const double *kt = k + ((size_t)c * n + t) * dk;
            const double *vt = v + ((size_t)c * n + t) * dv;
            const double *at = alpha_at(mode, dk, n, a, c, t);
            double bt = (mode == ORC_GATED_DELTA || mode == ORC_KDA) ? b[(size_t)c * n + t] : 0.0;
            apply_token(mode, dk, dk, Tc, kt, NULL, at, bt, u);
            apply_token(mode, dk, dv, Sc, kt, vt, at, bt, u);
        }
        free(u);
    }
    return err;
}

/* S_out[c] = T[c] S_in[c] + S_c[c]  (dense product; S_out may not alias S_in). */
int orc_compose(int dk, int dv, int n_chain, const double *T, const double *Sc,
                const double *S_in, double *S_out)
{
    if (dk <= 0 || dv <= 0 || n_chain < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int c = 0; c < n_chain; ++c) {
        const double *Tm = T + (size_t)c * dk * dk;
        const double *Cm = Sc + (size_t)c * dk * dv;
        const double *Xm = S_in + (size_t)c * dk * dv;
        double *Ym = S_out + (size_t)c * dk * dv;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double acc = Cm[(size_t)i * dv + j];
                for (int l = 0; l < dk; ++l)
                    acc += Tm[(size_t)i * dk + l] * Xm[(size_t)l * dv + j];
                Ym[(size_t)i * dv + j] = acc;
            }
    }
    return 0;
}
