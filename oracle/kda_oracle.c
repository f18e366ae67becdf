/*
 * TEST INFRASTRUCTURE ONLY.  The plain fp64 CPU oracle for the Kimi Delta
 * Attention (KDA) prefill forward.  Only tests/, the smoke check and the CPU
 * baseline leg of the benchmark may load this; the CUDA product path never does,
 * and the two share no code.
 *
 * What it computes (the gated delta rule as the method defines it):
 *   "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 01 RESULTS
 *   (every kernel is checked against a token-by-token fp64 recurrence) and
 *   section 03 REWARD HACKING (q and k are L2-normalised; an initial state enters;
 *   cu_seqlens packs variable-length sequences);
 *   "Autoresearch on Kimi Delta Attention", section THE MECHANISM (a fixed-size
 *   memory per head; each token reads the memory's prediction and writes only the
 *   correction; each key channel forgets at its own rate).
 *
 * For every sequence s and head h, with S a dk x dv matrix:
 *     S <- h0[s,h]               (zeros when h0 is NULL)
 *     for each token t of s, in order:
 *         qh = q_t / sqrt(|q_t|^2 + eps),  kh = k_t / sqrt(|k_t|^2 + eps)
 *         S  <- Diag(exp(g_t)) S                      (per key-channel decay)
 *         r  <- S^T kh                                 (what the memory predicts)
 *         S  <- S + beta_t kh (v_t - r)^T              (write only the correction)
 *         o_t = scale * S^T qh                         (read the updated state)
 *     hT[s,h] <- S
 * which is S_t = (I - beta_t kh kh^T) Diag(alpha_t) S_{t-1} + beta_t kh v_t^T.
 *
 * Layout (row-major, contiguous):
 *   q, k, g : [B, T, H, dk]      v, o : [B, T, H, dv]      beta : [B, T, H]
 *   h0, hT  : [N, H, dk, dv]
 * Fixed length: cu_seqlens == NULL, N = B, sequence b is batch row b.
 * Varlen: B == 1, cu_seqlens holds N+1 non-decreasing offsets into the T axis.
 * Returns 0 on success, -1 on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted mistakes, for the tests that show the pins can catch them.  The
 * normal build defines no KDA_ORACLE_MUTANT and every MUT(n) is 0. */
#ifndef KDA_ORACLE_MUTANT
#define KDA_ORACLE_MUTANT 0
#endif
#define MUT(n) (KDA_ORACLE_MUTANT == (n))

static void l2_normalise(const double* x, int64_t d, double eps, double* out) {
    double ss = 0.0;
    for (int64_t c = 0; c < d; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + eps);
    for (int64_t c = 0; c < d; ++c) out[c] = x[c] * inv;
}

/* One (sequence, head) chain: rows [bos, eos) of the batch row `b`. */
static void run_chain(const double* q, const double* k, const double* v,
                      const double* g, const double* beta, const double* h0,
                      int64_t b, int64_t bos, int64_t eos, int64_t s, int64_t h,
                      int64_t T, int64_t H, int64_t dk, int64_t dv,
                      double scale, double eps, double* o, double* hT,
                      double* S, double* qh, double* kh, double* r) {
    if (h0 && !MUT(7)) memcpy(S, h0 + (s * H + h) * dk * dv, sizeof(double) * dk * dv);
    else memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t = bos; t < eos; ++t) {
        int64_t row = (b * T + t) * H + h;          /* token-head index */
        l2_normalise(q + row * dk, dk, eps, qh);
        l2_normalise(k + row * dk, dk, eps, kh);
        if (MUT(5)) { /* normalisation dropped: raw vectors */
            for (int64_t c = 0; c < dk; ++c) { qh[c] = q[row * dk + c]; kh[c] = k[row * dk + c]; }
        }
        const double* gt = g + row * dk;
        const double* vt = v + row * dv;
        double bt = MUT(4) ? 1.0 : beta[row];
        double* ot = o + row * dv;

        /* S <- Diag(alpha) S */
        if (!MUT(1) && !MUT(6)) {
            for (int64_t i = 0; i < dk; ++i) {
                double a = exp(gt[i]);
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
            }
        }
        if (MUT(3)) { /* reads the state before this token's write */
            for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qh[i];
            for (int64_t j = 0; j < dv; ++j) ot[j] *= scale;
        }
        /* r = S^T kh */
        for (int64_t j = 0; j < dv; ++j) r[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) r[j] += S[i * dv + j] * kh[i];
        /* S <- S + beta kh (v - r)^T */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                S[i * dv + j] += bt * kh[i] * (MUT(2) ? vt[j] + r[j] : vt[j] - r[j]);
        if (MUT(6)) { /* decay applied after the write */
            for (int64_t i = 0; i < dk; ++i) {
                double a = exp(gt[i]);
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
            }
        }
        if (MUT(3)) continue;
        /* o_t = scale S^T qh */
        const double* rd = MUT(8) ? kh : qh;
        for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                ot[j] += (MUT(9) ? S[j * dv + i] : S[i * dv + j]) * rd[i];
        if (!MUT(10))
            for (int64_t j = 0; j < dv; ++j) ot[j] *= scale;
    }
    if (hT) memcpy(hT + (s * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

int kda_oracle_fwd(const double* q, const double* k, const double* v,
                   const double* g, const double* beta, const double* h0,
                   const int64_t* cu_seqlens, int64_t num_seqs,
                   int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                   double scale, double eps, double* o, double* hT, int nthreads) {
    if (!q || !k || !v || !g || !beta || !o) return -1;
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || num_seqs < 0) return -1;
    if (cu_seqlens) {
        if (B != 1) return -1;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
        for (int64_t s = 0; s < num_seqs; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    } else if (num_seqs != B) {
        return -1;
    }
    int64_t units = num_seqs * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
        double* qh = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kh = (double*)malloc(sizeof(double) * (size_t)dk);
        double* r = (double*)malloc(sizeof(double) * (size_t)dv);
        int ok = S && qh && kh && r;
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            if (!ok) continue;
            int64_t s = u / H, h = u % H;
            int64_t b = cu_seqlens ? 0 : s;
            int64_t bos = cu_seqlens ? cu_seqlens[s] : 0;
            int64_t eos = cu_seqlens ? cu_seqlens[s + 1] : T;
            run_chain(q, k, v, g, beta, h0, b, bos, eos, s, h, T, H, dk, dv,
                      scale, eps, o, hT, S, qh, kh, r);
        }
        free(S); free(qh); free(kh); free(r);
    }
    return failed ? -2 : 0;
}

/* Number of threads the OpenMP runtime would use (1 when built without it). */
int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
