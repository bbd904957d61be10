/*
 * Plain FP64 CPU oracle for GatedDeltaNet speculative verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file; only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark load it.
 * It shares no code, header or constant with the CUDA path.
 *
 * What it computes (each function cites the passage it follows):
 *
 *   oracle_gdn_recurrent   the gated delta rule, token by token
 *       S_t = S_{t-1} * alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *       o_t = q_scale * S_t q_t,  alpha_t = exp(g_t)
 *     ("Native three-step MTP", What changed: FP32 sigmoid gates and the
 *     GDN state update; the recurrence itself is the gated delta rule of the
 *     task statement).  The product S (alpha (I - beta k k^T)) is expanded as
 *     alpha S - alpha beta (S k) k^T, i.e. S <- alpha S + beta (v - alpha S k) k^T,
 *     which is the same matrix with O(d_v d_k) work per token.
 *     S is d_v x d_k, row-major: S[a][j], a over values, j over keys.
 *
 *   oracle_gdn_chunked     the same recurrence evaluated chunk by chunk in
 *     the WY/UT form ("Run chained MTP drafting in the batch Engine",
 *     Correctness fix: the chunked GatedDeltaNet plan publishes only the
 *     final state).  Within a chunk with start state S0 and G = cumsum(g):
 *       A[t][i] = beta_t e^{G_t - G_i} k_t.k_i (i < t),  T = (I + A)^{-1}
 *       W  = T diag(beta e^G) K,   Ut = T diag(beta) V,   U = Ut - W S0^T
 *       O  = diag(e^G) Q S0^T + (M o Q K^T) U,  M[t][i] = e^{G_t - G_i}, i <= t
 *       S' = e^{G_last} S0 + U^T diag(e^{G_last - G}) K
 *     Derivation: unrolling S_t = alpha_t S_{t-1} + u_t k_t^T with
 *     u_t = beta_t (v_t - alpha_t S_{t-1} k_t) inside the chunk gives
 *     (I + A) U = diag(beta) V - diag(beta e^G) K S0^T.
 *
 *   oracle_argmax_bf16     greedy choice per logits row: a scan with strict
 *     '>' over bf16 values widened exactly to float, lowest index on ties,
 *     the first NaN wins ("Native three-step MTP", Apply...: greedy requests;
 *     "Run chained MTP drafting", Quality follow-up: greedy trajectories).
 *
 * Units are independent (request, v-head) pairs; OpenMP spreads them over
 * the host cores without changing any unit's arithmetic order.
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Recurrent form.  For unit u the rows are [roff[u], roff[u+1]) of the packed
 * arrays q,k [R][dk], v [R][dv], g,beta [R]; S [units][dv][dk] holds S_0 on
 * entry and the state after the last row on exit; ckpt [R][dv][dk] (may be
 * NULL) receives the state after every row; o [R][dv].
 */
void oracle_gdn_recurrent(int dk, int dv, int units, const int64_t *roff,
                          const double *q, const double *k, const double *v,
                          const double *g, const double *beta, double q_scale,
                          double *S, double *ckpt, double *o)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < units; ++u) {
        double *s = S + (size_t)u * dv * dk;
        double *sk = (double *)malloc(sizeof(double) * (size_t)dv);
        for (int64_t t = roff[u]; t < roff[u + 1]; ++t) {
            const double *kt = k + (size_t)t * dk;
            const double *qt = q + (size_t)t * dk;
            const double *vt = v + (size_t)t * dv;
            const double alpha = exp(g[t]);
            const double b = beta[t];
            /* S_{t-1} k_t */
            for (int a = 0; a < dv; ++a) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += s[(size_t)a * dk + j] * kt[j];
                sk[a] = acc;
            }
            /* S_t = alpha S_{t-1} + beta (v_t - alpha S_{t-1} k_t) k_t^T */
            for (int a = 0; a < dv; ++a) {
                const double ua = b * (vt[a] - alpha * sk[a]);
                for (int j = 0; j < dk; ++j)
                    s[(size_t)a * dk + j] = alpha * s[(size_t)a * dk + j] + ua * kt[j];
            }
            /* o_t = q_scale * S_t q_t */
            for (int a = 0; a < dv; ++a) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += s[(size_t)a * dk + j] * qt[j];
                o[(size_t)t * dv + a] = q_scale * acc;
            }
            if (ckpt) memcpy(ckpt + (size_t)t * dv * dk, s, sizeof(double) * (size_t)dv * dk);
        }
        free(sk);
    }
}

/*
 * WY/UT quantities of one chunk of n rows (k [n][dk], v [n][dv], g, beta [n]):
 * G (cumsum of g), T = (I + A)^{-1} [n][n], W [n][dk], Ut [n][dv].
 * T is obtained by forward substitution on the unit lower-triangular I + A:
 *   T[t][t] = 1,  T[t][i] = -sum_{m=i}^{t-1} A[t][m] T[m][i]  (i < t).
 */
void oracle_gdn_chunk_wy(int dk, int dv, int n, const double *k, const double *v,
                         const double *g, const double *beta,
                         double *G, double *T, double *W, double *Ut)
{
    double run = 0.0;
    for (int t = 0; t < n; ++t) {
        run += g[t];
        G[t] = run;
    }
    double *A = (double *)calloc((size_t)n * n, sizeof(double));
    for (int t = 0; t < n; ++t)
        for (int i = 0; i < t; ++i) {
            double kk = 0.0;
            for (int j = 0; j < dk; ++j) kk += k[(size_t)t * dk + j] * k[(size_t)i * dk + j];
            A[(size_t)t * n + i] = beta[t] * exp(G[t] - G[i]) * kk;
        }
    memset(T, 0, sizeof(double) * (size_t)n * n);
    for (int t = 0; t < n; ++t) {
        T[(size_t)t * n + t] = 1.0;
        for (int i = 0; i < t; ++i) {
            double acc = 0.0;
            for (int m = i; m < t; ++m) acc += A[(size_t)t * n + m] * T[(size_t)m * n + i];
            T[(size_t)t * n + i] = -acc;
        }
    }
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < dk; ++j) {
            double acc = 0.0;
            for (int i = 0; i <= t; ++i)
                acc += T[(size_t)t * n + i] * beta[i] * exp(G[i]) * k[(size_t)i * dk + j];
            W[(size_t)t * dk + j] = acc;
        }
        for (int a = 0; a < dv; ++a) {
            double acc = 0.0;
            for (int i = 0; i <= t; ++i)
                acc += T[(size_t)t * n + i] * beta[i] * v[(size_t)i * dv + a];
            Ut[(size_t)t * dv + a] = acc;
        }
    }
    free(A);
}

/*
 * Chunked form with chunk length C (the last chunk of a unit may be shorter).
 * Same argument layout as oracle_gdn_recurrent, without checkpoints: the
 * chunked form only publishes the state at the end of the unit's rows.
 */
void oracle_gdn_chunked(int dk, int dv, int units, const int64_t *roff, int C,
                        const double *q, const double *k, const double *v,
                        const double *g, const double *beta, double q_scale,
                        double *S, double *o)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < units; ++u) {
        double *s = S + (size_t)u * dv * dk;
        double *G = (double *)malloc(sizeof(double) * (size_t)C);
        double *T = (double *)malloc(sizeof(double) * (size_t)C * C);
        double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
        double *Ut = (double *)malloc(sizeof(double) * (size_t)C * dv);
        double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
        double *snew = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        for (int64_t c0 = roff[u]; c0 < roff[u + 1]; c0 += C) {
            const int n = (int)((roff[u + 1] - c0) < C ? (roff[u + 1] - c0) : C);
            const double *kc = k + (size_t)c0 * dk;
            const double *qc = q + (size_t)c0 * dk;
            const double *vc = v + (size_t)c0 * dv;
            oracle_gdn_chunk_wy(dk, dv, n, kc, vc, g + c0, beta + c0, G, T, W, Ut);
            /* U = Ut - W S0^T */
            for (int t = 0; t < n; ++t)
                for (int a = 0; a < dv; ++a) {
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += W[(size_t)t * dk + j] * s[(size_t)a * dk + j];
                    U[(size_t)t * dv + a] = Ut[(size_t)t * dv + a] - acc;
                }
            /* O = diag(e^G) Q S0^T + (M o Q K^T) U */
            for (int t = 0; t < n; ++t) {
                for (int a = 0; a < dv; ++a) {
                    double inter = 0.0;
                    for (int j = 0; j < dk; ++j) inter += qc[(size_t)t * dk + j] * s[(size_t)a * dk + j];
                    double intra = 0.0;
                    for (int i = 0; i <= t; ++i) {
                        double qk = 0.0;
                        for (int j = 0; j < dk; ++j) qk += qc[(size_t)t * dk + j] * kc[(size_t)i * dk + j];
                        intra += exp(G[t] - G[i]) * qk * U[(size_t)i * dv + a];
                    }
                    o[(size_t)(c0 + t) * dv + a] = q_scale * (exp(G[t]) * inter + intra);
                }
            }
            /* S' = e^{G_last} S0 + U^T diag(e^{G_last - G}) K */
            const double Gl = G[n - 1];
            for (int a = 0; a < dv; ++a)
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < n; ++i)
                        acc += U[(size_t)i * dv + a] * exp(Gl - G[i]) * kc[(size_t)i * dk + j];
                    snew[(size_t)a * dk + j] = exp(Gl) * s[(size_t)a * dk + j] + acc;
                }
            memcpy(s, snew, sizeof(double) * (size_t)dv * dk);
        }
        free(G); free(T); free(W); free(Ut); free(U); free(snew);
    }
}

static float bf16_bits_to_float(uint16_t h)
{
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/*
 * Greedy choice per row of bf16 logits: rows x vocab values at row stride
 * `stride` (elements).  out[r] = index of the first maximum, or of the first
 * NaN if the row holds one; -1 for an empty row.
 */
void oracle_argmax_bf16(int64_t rows, int64_t vocab, int64_t stride,
                        const uint16_t *x, int32_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *row = x + r * stride;
        int64_t best = -1;
        float bestv = 0.0f;
        for (int64_t i = 0; i < vocab; ++i) {
            const float f = bf16_bits_to_float(row[i]);
            if (isnan(f)) { best = i; break; }
            if (best < 0 || f > bestv) { best = i; bestv = f; }
        }
        out[r] = (int32_t)best;
    }
}
