/*
 * KDA forward oracle: the per-token gated delta-rule recurrence in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is part of the oracle that the CUDA
 * path is checked against.  It shares no code, header, table or constant with
 * the CUDA library, and the product path never links or calls it; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes (page "PyPTO-Gym chunk_kda operator: an NPU forward of
 * chunked gated delta-rule linear attention"):
 *   - section "算子定位与算法背景" (operator placement and background): per
 *     token, first the per-dimension gate decay S <- S * exp(g), then the
 *     delta update S <- S + outer(beta*k, v - k.S), then the read-out
 *     o = q.S.  S is the K x V state, g lives in the log domain (g <= 0).
 *   - section "算法原理" step M1: q is multiplied by `scale`.
 *   - section "算子签名与 I/O 规格" (signature and I/O): the initial and final
 *     state use the [N, H, V, K] layout, i.e. the transpose of the K x V state;
 *     scale None means K^-0.5 (the caller resolves that, this file takes a
 *     number); fixed-length inputs form N = B sequences of length T, varlen
 *     inputs (B == 1) are delimited by cu_seqlens.
 *   - section "测试与验证体系" (tests): the optional in-kernel q/k
 *     normalisation is a per-token L2 normalisation over the K dimension with
 *     eps = 1e-6, read here as x / sqrt(sum(x^2) + 1e-6).
 *
 * Precision: every arithmetic step is double.  Inputs arrive as float
 * (bf16 q/k/v widened exactly, fp32 g/beta/h0).  The unit loop (one sequence
 * times one head) is the natural parallel grain; OpenMP spreads it over the
 * host cores when the file is built with -fopenmp.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define KDA_ORACLE_OK 0
#define KDA_ORACLE_BAD_ARG 1
#define KDA_ORACLE_BAD_CU 2
#define KDA_ORACLE_NO_MEM 3

/* Number of host threads OpenMP would use (1 when built without OpenMP). */
int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Run the recurrence for every selected (sequence, head) unit.
 *
 *   q, k      float [B*T, H, K]  (bf16 values widened exactly)
 *   v         float [B*T, H, V]
 *   g         float [B*T, H, K]  log-domain gate
 *   beta      float [B*T, H]
 *   scale     multiplier applied to q (after the optional normalisation)
 *   h0        float [N, H, V, K] or NULL (zero initial state)
 *   cu        int32 [N+1] token offsets, or NULL for fixed length (N == B)
 *   l2norm    nonzero: normalise q and k per token before use
 *   unit_mask uint8 [N*H] (index n*H + h) or NULL for all units; units whose
 *             byte is 0 are skipped and their outputs left untouched
 *   o         double [B*T, H, V]  written for the selected units
 *   ht        double [N, H, V, K] written for the selected units, or NULL
 */
int kda_oracle_recurrent(const float *q, const float *k, const float *v,
                         const float *g, const float *beta, double scale,
                         const float *h0, const int32_t *cu, int B, int T,
                         int H, int K, int V, int N, int l2norm,
                         const uint8_t *unit_mask, double *o, double *ht) {
    if (!q || !k || !v || !g || !beta || !o) return KDA_ORACLE_BAD_ARG;
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1 || N < 0) return KDA_ORACLE_BAD_ARG;
    if (cu == NULL) {
        if (N != B) return KDA_ORACLE_BAD_ARG;
    } else {
        if (B != 1) return KDA_ORACLE_BAD_ARG;
        if (cu[0] != 0 || cu[N] != T) return KDA_ORACLE_BAD_CU;
        for (int n = 0; n < N; ++n)
            if (cu[n + 1] < cu[n]) return KDA_ORACLE_BAD_CU;
    }

    const long long units = (long long)N * H;
    int status = KDA_ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (long long unit = 0; unit < units; ++unit) {
        if (unit_mask && !unit_mask[unit]) continue;
        const int n = (int)(unit / H);
        const int h = (int)(unit % H);
        const long long bos = cu ? (long long)cu[n] : (long long)n * T;
        const long long eos = cu ? (long long)cu[n + 1] : (long long)(n + 1) * T;

        /* S is K x V, row-major: S[d * V + j]. */
        double *S = (double *)malloc(sizeof(double) * (size_t)K * (size_t)V);
        double *xq = (double *)malloc(sizeof(double) * (size_t)K);
        double *xk = (double *)malloc(sizeof(double) * (size_t)K);
        double *kS = (double *)malloc(sizeof(double) * (size_t)V);
        if (!S || !xq || !xk || !kS) {
            free(S); free(xq); free(xk); free(kS);
#pragma omp atomic write
            status = KDA_ORACLE_NO_MEM;
            continue;
        }

        /* Initial state: the [V, K] slab transposed into the K x V state. */
        for (int d = 0; d < K; ++d)
            for (int j = 0; j < V; ++j)
                S[(size_t)d * V + j] =
                    h0 ? (double)h0[(((size_t)n * H + h) * V + j) * K + d] : 0.0;

        for (long long t = bos; t < eos; ++t) {
            const size_t rowK = ((size_t)t * H + h) * (size_t)K;
            const size_t rowV = ((size_t)t * H + h) * (size_t)V;

            for (int d = 0; d < K; ++d) {
                xq[d] = (double)q[rowK + d];
                xk[d] = (double)k[rowK + d];
            }
            if (l2norm) {
                double sq = 0.0, sk = 0.0;
                for (int d = 0; d < K; ++d) {
                    sq += xq[d] * xq[d];
                    sk += xk[d] * xk[d];
                }
                const double iq = 1.0 / sqrt(sq + 1e-6);
                const double ik = 1.0 / sqrt(sk + 1e-6);
                for (int d = 0; d < K; ++d) {
                    xq[d] *= iq;
                    xk[d] *= ik;
                }
            }

            /* 1. decay: S <- diag(exp(g_t)) S */
            for (int d = 0; d < K; ++d) {
                const double a = exp((double)g[rowK + d]);
                double *Srow = S + (size_t)d * V;
                for (int j = 0; j < V; ++j) Srow[j] *= a;
            }

            /* 2. delta update: S <- S + beta * k (v - S^T k)^T */
            for (int j = 0; j < V; ++j) kS[j] = 0.0;
            for (int d = 0; d < K; ++d) {
                const double kd = xk[d];
                const double *Srow = S + (size_t)d * V;
                for (int j = 0; j < V; ++j) kS[j] += kd * Srow[j];
            }
            const double b = (double)beta[(size_t)t * H + h];
            for (int j = 0; j < V; ++j) kS[j] = b * ((double)v[rowV + j] - kS[j]);
            for (int d = 0; d < K; ++d) {
                const double kd = xk[d];
                double *Srow = S + (size_t)d * V;
                for (int j = 0; j < V; ++j) Srow[j] += kd * kS[j];
            }

            /* 3. read-out: o_t = S^T (scale * q) */
            double *orow = o + rowV;
            for (int j = 0; j < V; ++j) orow[j] = 0.0;
            for (int d = 0; d < K; ++d) {
                const double qd = scale * xq[d];
                const double *Srow = S + (size_t)d * V;
                for (int j = 0; j < V; ++j) orow[j] += qd * Srow[j];
            }
        }

        if (ht) {
            for (int j = 0; j < V; ++j)
                for (int d = 0; d < K; ++d)
                    ht[(((size_t)n * H + h) * V + j) * K + d] = S[(size_t)d * V + j];
        }
        free(S); free(xq); free(xk); free(kS);
    }
    return status;
}
