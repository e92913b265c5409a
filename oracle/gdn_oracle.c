/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle for the gated delta rule and
 * for plain causal linear attention.  TEST INFRASTRUCTURE ONLY: nothing on
 * the product (CUDA) path includes, links or calls this file; only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg load it.
 *
 * Sources (the web pages this project restates):
 *  - "Как ускорить LLM на длинном контексте" (tgstat post of the RnD ML team),
 *    section "Linear attention": the plain state rule S_t = S_{t-1} + v_t k_t^T,
 *    one recurrent step of O(1) memory per token.
 *  - forpes.ru survey of linear attention and linearization, section
 *    "Введение": linear attention has a recurrent form over a fixed-size state
 *    matrix; GatedDeltaNet is named among the gated variants (its update table
 *    did not survive extraction).  The gated delta rule used here is
 *        S_t = a_t * S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t
 *    with a_t = exp(log_alpha_t) the scalar gate and b_t the write strength.
 *  - "Метод SparseGDN ускоряет префилл Gated Delta Networks…", section
 *    "Чем дорог префилл в Gated Delta Networks…": prefill is computed per chunk
 *    of fixed size -- an intra-chunk delta-system solve, a sequential per-head
 *    pass over chunks, and the state at each chunk start feeding that chunk's
 *    outputs.  Section "Схема встраивания селектора…": the per-chunk update is
 *    an affine map S -> A_c S + B_c applied chunk after chunk.
 *
 * Conventions (readings of the pages, stated once):
 *  - S is d_v x d_k (S_t = ... + v_t k_t^T).  The stored state is h = S^T,
 *    laid out [d_k][d_v] row-major.
 *  - o_t uses the state AFTER token t's update (the diagonal of the causal
 *    mask is included).  No 1/sqrt(d) scaling of q: callers pre-scale.
 *  - Tensors are token-major and packed: x[t][head][feature]; sequences are
 *    delimited by cu_seqlens[0..n_seqs] (cu[0] = 0, non-decreasing).
 *  - log_alpha == NULL means a_t = 1; beta == NULL means b_t = 1;
 *    h0 == NULL means a zero initial state; hT may be NULL.
 *
 * Everything is double precision with plain loops, so that the arithmetic
 * can be read against the formulas above.  (seq, head) chains are
 * independent and run in parallel with OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS -1
#define ORACLE_ERR_SEQLENS -2
#define ORACLE_ERR_NOMEM -3

static int check_seqlens(const int64_t *cu, int n_seqs)
{
    if (n_seqs < 0 || cu == NULL || cu[0] != 0) return 0;
    for (int s = 0; s < n_seqs; ++s)
        if (cu[s + 1] < cu[s]) return 0;
    return 1;
}

static int set_threads(int n_threads)
{
#ifdef _OPENMP
    return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

int oracle_num_threads(int n_threads) { return set_threads(n_threads); }

/*
 * Token-by-token recurrence, the definition of the method.
 *   delta_rule = 1:  S <- a S - b (a S k) k^T + b v k^T   (= a S (I - b k k^T) + b v k^T)
 *   delta_rule = 0:  S <- a S + b v k^T                   (plain rule when a = b = 1)
 *   o_t = S q_t after the update.
 */
int oracle_recurrent(const double *q, const double *k, const double *v,
                     const double *log_alpha, const double *beta,
                     const double *h0, const int64_t *cu, int n_seqs,
                     int H, int dk, int dv, int delta_rule,
                     double *o, double *hT, int n_threads)
{
    if (!q || !k || !v || !o || H <= 0 || dk <= 0 || dv <= 0) return ORACLE_ERR_ARGS;
    if (!check_seqlens(cu, n_seqs)) return ORACLE_ERR_SEQLENS;
    const int n_chains = n_seqs * H;
    const int nt = set_threads(n_threads);
    int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int c = 0; c < n_chains; ++c) {
        const int s = c / H, hd = c % H;
        double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        double *Sk = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!S || !Sk) {
            free(S); free(Sk);
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
            continue;
        }
        /* S = h0^T */
        for (int j = 0; j < dv; ++j)
            for (int i = 0; i < dk; ++i)
                S[(size_t)j * dk + i] =
                    h0 ? h0[(((size_t)s * H + hd) * dk + i) * dv + j] : 0.0;

        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
            const size_t row = (size_t)t * H + hd;
            const double *qt = q + row * dk;
            const double *kt = k + row * dk;
            const double *vt = v + row * dv;
            const double a = log_alpha ? exp(log_alpha[row]) : 1.0;
            const double b = beta ? beta[row] : 1.0;

            /* (S k_t), taken from the state before this token's update */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dk + i] * kt[i];
                Sk[j] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                for (int i = 0; i < dk; ++i) {
                    double x = a * S[(size_t)j * dk + i];
                    if (delta_rule) x -= b * (a * Sk[j]) * kt[i];
                    x += b * vt[j] * kt[i];
                    S[(size_t)j * dk + i] = x;
                }
            }
            /* o_t = S_t q_t */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dk + i] * qt[i];
                o[row * dv + j] = acc;
            }
        }
        if (hT)
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    hT[(((size_t)s * H + hd) * dk + i) * dv + j] = S[(size_t)j * dk + i];
        free(S);
        free(Sk);
    }
    return status;
}

/* Number of chunks of size C in each sequence (the last may be partial). */
static int64_t chunks_of(int64_t len, int C) { return (len + C - 1) / C; }

int64_t oracle_num_chunks(const int64_t *cu, int n_seqs, int C)
{
    int64_t n = 0;
    for (int s = 0; s < n_seqs; ++s) n += chunks_of(cu[s + 1] - cu[s], C);
    return n;
}

/*
 * Chunk-wise evaluation, following the stages the SparseGDN article lists for
 * chunked GDN prefill: within each chunk a delta system is solved (quadratic
 * in the chunk size), then the state is carried from chunk to chunk, and each
 * chunk's outputs use the state at the chunk start.  In the notation of the
 * token recurrence, with g the within-chunk running sum of log_alpha and h
 * the state (h = S^T) at the chunk start:
 *
 *   A[i][j] = b_i exp(g_i - g_j) (k_i . k_j)       for j < i, else 0
 *   Tm      = (I + A)^(-1)                          (forward substitution)
 *   w       = Tm (b * exp(g) * K),   u = Tm (b * V)
 *   v_new   = u - w h
 *   o_i     = exp(g_i) q_i^T h + sum_{j<=i} exp(g_i - g_j) (q_i . k_j) v_new_j
 *   h      <- exp(g_last) h + sum_j exp(g_last - g_j) k_j v_new_j^T
 *
 * (These follow from unrolling the token recurrence inside one chunk; with
 * delta_rule = 0 the system is trivial: A = 0, w = 0, v_new = b * V.)
 * Optional per-chunk outputs (any may be NULL), indexed by the global chunk
 * number n (chunks numbered sequence by sequence):
 *   A_out, Tm_out : [n][H][C][C]   (rows past a partial chunk's end are 0 / identity)
 *   w_out         : [t][H][dk],  u_out : [t][H][dv],  g_out : [t][H]
 *
 * band > 0 selects the block-adjacent solver of the SparseGDN article
 * ("Двухуровневая разреженность SparseGDN…", first observation: the solver
 * restricts the delta system to links between neighbouring blocks, a fixed,
 * input-independent approximation).  Read here as: Tm is kept on the
 * diagonal blocks of `band` tokens and on the blocks directly below them,
 * both exactly as the full inverse has them, and is zero on blocks two or
 * more apart.  band = 0 is the exact solve.
 */
static int chunked_impl(const double *q, const double *k, const double *v,
                        const double *log_alpha, const double *beta,
                        const double *h0, const int64_t *cu, int n_seqs,
                        int H, int dk, int dv, int C, int delta_rule, int band,
                        double *o, double *hT,
                        double *A_out, double *Tm_out, double *w_out, double *u_out,
                        double *g_out, int n_threads)
{
    if (!q || !k || !v || !o || H <= 0 || dk <= 0 || dv <= 0 || C <= 0)
        return ORACLE_ERR_ARGS;
    if (!check_seqlens(cu, n_seqs)) return ORACLE_ERR_SEQLENS;
    const int n_chains = n_seqs * H;
    const int nt = set_threads(n_threads);
    int status = ORACLE_OK;

    /* first global chunk number of each sequence */
    int64_t *chunk0 = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_seqs + 1));
    if (!chunk0) return ORACLE_ERR_NOMEM;
    chunk0[0] = 0;
    for (int s = 0; s < n_seqs; ++s) chunk0[s + 1] = chunk0[s] + chunks_of(cu[s + 1] - cu[s], C);

#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int c = 0; c < n_chains; ++c) {
        const int s = c / H, hd = c % H;
        const size_t CC = (size_t)C * C;
        double *h = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        double *g = (double *)malloc(sizeof(double) * (size_t)C);
        double *A = (double *)malloc(sizeof(double) * CC);
        double *Tm = (double *)malloc(sizeof(double) * CC);
        double *w = (double *)malloc(sizeof(double) * (size_t)C * dk);
        double *u = (double *)malloc(sizeof(double) * (size_t)C * dv);
        double *vn = (double *)malloc(sizeof(double) * (size_t)C * dv);
        double *hn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        if (!h || !g || !A || !Tm || !w || !u || !vn || !hn) {
            free(h); free(g); free(A); free(Tm); free(w); free(u); free(vn); free(hn);
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
            continue;
        }
        for (size_t x = 0; x < (size_t)dk * dv; ++x)
            h[x] = h0 ? h0[((size_t)s * H + hd) * dk * dv + x] : 0.0;

        const int64_t L = cu[s + 1] - cu[s];
        for (int64_t ch = 0; ch < chunks_of(L, C); ++ch) {
            const int64_t t0 = cu[s] + ch * C;
            const int n = (int)((L - ch * C) < C ? (L - ch * C) : C); /* valid tokens */
#define ROW(t) ((size_t)(t0 + (t)) * H + hd)
            /* g: running sum of log_alpha within the chunk */
            double run = 0.0;
            for (int i = 0; i < n; ++i) {
                run += log_alpha ? log_alpha[ROW(i)] : 0.0;
                g[i] = run;
            }
            /* A: decay-masked, beta-scaled K K^T, strictly lower */
            memset(A, 0, sizeof(double) * CC);
            if (delta_rule)
                for (int i = 0; i < n; ++i)
                    for (int j = 0; j < i; ++j) {
                        double kk = 0.0;
                        for (int x = 0; x < dk; ++x) kk += k[ROW(i) * dk + x] * k[ROW(j) * dk + x];
                        const double bi = beta ? beta[ROW(i)] : 1.0;
                        A[(size_t)i * C + j] = bi * exp(g[i] - g[j]) * kk;
                    }
            /* Tm = (I + A)^-1 by forward substitution, row by row:
               Tm[i][:] = e_i - sum_{j<i} A[i][j] Tm[j][:] */
            memset(Tm, 0, sizeof(double) * CC);
            for (int i = 0; i < C; ++i) {
                for (int col = 0; col < C; ++col) {
                    double x = (i == col) ? 1.0 : 0.0;
                    for (int j = 0; j < i; ++j) x -= A[(size_t)i * C + j] * Tm[(size_t)j * C + col];
                    Tm[(size_t)i * C + col] = x;
                }
            }
            /* block-adjacent solver: drop the blocks of Tm two or more blocks below
               the diagonal */
            if (band > 0)
                for (int i = 0; i < C; ++i)
                    for (int col = 0; col < C; ++col)
                        if (i / band - col / band >= 2) Tm[(size_t)i * C + col] = 0.0;
            /* w = Tm (b e^g K), u = Tm (b V) */
            for (int i = 0; i < n; ++i) {
                for (int x = 0; x < dk; ++x) {
                    double acc = 0.0;
                    if (delta_rule)
                        for (int j = 0; j <= i; ++j) {
                            const double bj = beta ? beta[ROW(j)] : 1.0;
                            acc += Tm[(size_t)i * C + j] * bj * exp(g[j]) * k[ROW(j) * dk + x];
                        }
                    w[(size_t)i * dk + x] = acc;
                }
                for (int y = 0; y < dv; ++y) {
                    double acc = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        const double bj = beta ? beta[ROW(j)] : 1.0;
                        acc += Tm[(size_t)i * C + j] * bj * v[ROW(j) * dv + y];
                    }
                    u[(size_t)i * dv + y] = acc;
                }
            }
            /* v_new = u - w h */
            for (int i = 0; i < n; ++i)
                for (int y = 0; y < dv; ++y) {
                    double acc = u[(size_t)i * dv + y];
                    for (int x = 0; x < dk; ++x) acc -= w[(size_t)i * dk + x] * h[(size_t)x * dv + y];
                    vn[(size_t)i * dv + y] = acc;
                }
            /* outputs from the chunk-start state plus the intra-chunk part */
            for (int i = 0; i < n; ++i)
                for (int y = 0; y < dv; ++y) {
                    double inter = 0.0;
                    for (int x = 0; x < dk; ++x) inter += q[ROW(i) * dk + x] * h[(size_t)x * dv + y];
                    double intra = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        double qk = 0.0;
                        for (int x = 0; x < dk; ++x) qk += q[ROW(i) * dk + x] * k[ROW(j) * dk + x];
                        intra += exp(g[i] - g[j]) * qk * vn[(size_t)j * dv + y];
                    }
                    o[ROW(i) * dv + y] = exp(g[i]) * inter + intra;
                }
            /* carry the state to the next chunk start */
            const double gl = n > 0 ? g[n - 1] : 0.0;
            for (int x = 0; x < dk; ++x)
                for (int y = 0; y < dv; ++y) {
                    double acc = exp(gl) * h[(size_t)x * dv + y];
                    for (int j = 0; j < n; ++j)
                        acc += exp(gl - g[j]) * k[ROW(j) * dk + x] * vn[(size_t)j * dv + y];
                    hn[(size_t)x * dv + y] = acc;
                }
            memcpy(h, hn, sizeof(double) * (size_t)dk * dv);

            const int64_t gch = chunk0[s] + ch;
            if (A_out) memcpy(A_out + ((size_t)gch * H + hd) * CC, A, sizeof(double) * CC);
            if (Tm_out) memcpy(Tm_out + ((size_t)gch * H + hd) * CC, Tm, sizeof(double) * CC);
            for (int i = 0; i < n; ++i) {
                if (w_out) memcpy(w_out + ROW(i) * dk, w + (size_t)i * dk, sizeof(double) * dk);
                if (u_out) memcpy(u_out + ROW(i) * dv, u + (size_t)i * dv, sizeof(double) * dv);
                if (g_out) g_out[ROW(i)] = g[i];
            }
#undef ROW
        }
        if (hT) memcpy(hT + ((size_t)s * H + hd) * dk * dv, h, sizeof(double) * (size_t)dk * dv);
        free(h); free(g); free(A); free(Tm); free(w); free(u); free(vn); free(hn);
    }
    free(chunk0);
    return status;
}

int oracle_chunked(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta,
                   const double *h0, const int64_t *cu, int n_seqs,
                   int H, int dk, int dv, int C, int delta_rule,
                   double *o, double *hT,
                   double *A_out, double *Tm_out, double *w_out, double *u_out,
                   double *g_out, int n_threads)
{
    return chunked_impl(q, k, v, log_alpha, beta, h0, cu, n_seqs, H, dk, dv, C, delta_rule, 0,
                        o, hT, A_out, Tm_out, w_out, u_out, g_out, n_threads);
}

int oracle_chunked_band(const double *q, const double *k, const double *v,
                        const double *log_alpha, const double *beta,
                        const double *h0, const int64_t *cu, int n_seqs,
                        int H, int dk, int dv, int C, int delta_rule, int band,
                        double *o, double *hT,
                        double *A_out, double *Tm_out, double *w_out, double *u_out,
                        double *g_out, int n_threads)
{
    if (band <= 0) return ORACLE_ERR_ARGS;
    return chunked_impl(q, k, v, log_alpha, beta, h0, cu, n_seqs, H, dk, dv, C, delta_rule, band,
                        o, hT, A_out, Tm_out, w_out, u_out, g_out, n_threads);
}
