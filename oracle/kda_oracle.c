/*
 * KDA oracle: plain fp64 CPU evaluation of the Kimi Delta Attention recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library. The product path
 * (the CUDA library) shares no code, header or constant with this file.
 *
 * What it computes. The orkas.ai page "Kimi K3 architecture" describes KDA in
 * prose: each KDA layer keeps a fixed-size state that is updated as the
 * sequence advances (section "Sequence: three quarters of the layers stopped
 * reading everything"), the state carries a decay (same section), the update
 * is serial and applies a token-dependent transition to the incoming state
 * (section "The bill arrives in the serving stack", first and second
 * bullets), and decoding updates the state in place (same section, third
 * bullet). The plainest formula that agrees with all of these is, per head,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * with S in R^{dk x dv}, g_t in R^{dk} the per-channel log-decay and beta_t a
 * scalar. This file evaluates exactly that, one token at a time, in fp64, in
 * the order the formula is written: decay first, then the delta-rule write,
 * then the read of the freshly written state. The only rewriting is the
 * expansion of the product: with S' = Diag(exp g) S,
 *     (I - beta k k^T) S' + beta k v^T = S' + k (beta (v - S'^T k))^T,
 * which avoids forming the dk x dk matrix. No chunking, blocking or
 * reordering is done.
 *
 * Inputs are read as the exact bytes handed to the GPU: q, k, v as bf16 or
 * fp32 (widened to fp64), g, beta and the initial state as fp32.
 *
 * Layouts (contiguous, row-major): q, k, g: [B, T, H, dk]; v, o: [B, T, H, dv];
 * beta: [B, T, H]; h0, hT: [B, H, dk, dv]. Decode uses T = 1 and N sequences.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* bf16 is the upper half of an IEEE fp32 word: widening is exact. */
static double load_elem(const void* p, int dtype, size_t i) {
    if (dtype == ORACLE_BF16) {
        uint32_t u = ((uint32_t)((const uint16_t*)p)[i]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float*)p)[i];
}

/*
 * One token of the recurrence on one head's state S[dk][dv] (fp64).
 * qi, ki, gi are dk-vectors, vi a dv-vector; kv and u are dv-sized scratch.
 * Writes o_t = S_t^T q_t to out[0..dv).
 */
static void kda_token(double* S, long dk, long dv, const double* qi, const double* ki,
                      const double* gi, const double* vi, double beta, double* kv,
                      double* u, double* out) {
    long i, j;
    /* S' = Diag(exp g_t) S_{t-1}: row i is channel i of the key space. */
    for (i = 0; i < dk; i++) {
        double a = exp(gi[i]);
        double* row = S + i * dv;
        for (j = 0; j < dv; j++) row[j] *= a;
    }
    /* kv = S'^T k_t */
    for (j = 0; j < dv; j++) kv[j] = 0.0;
    for (i = 0; i < dk; i++) {
        const double* row = S + i * dv;
        double kk = ki[i];
        for (j = 0; j < dv; j++) kv[j] += row[j] * kk;
    }
    /* u = beta_t (v_t - S'^T k_t) */
    for (j = 0; j < dv; j++) u[j] = beta * (vi[j] - kv[j]);
    /* S_t = S' + k_t u^T  ==  (I - beta k k^T) S' + beta k v^T */
    for (i = 0; i < dk; i++) {
        double* row = S + i * dv;
        double kk = ki[i];
        for (j = 0; j < dv; j++) row[j] += kk * u[j];
    }
    /* o_t = S_t^T q_t */
    for (j = 0; j < dv; j++) out[j] = 0.0;
    for (i = 0; i < dk; i++) {
        const double* row = S + i * dv;
        double qq = qi[i];
        for (j = 0; j < dv; j++) out[j] += row[j] * qq;
    }
}

/*
 * Prefill: runs the recurrence over T tokens for every (b, h).
 * h0 may be NULL (zero initial state). o and hT may be NULL (not written).
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int kda_oracle_prefill(const void* q, const void* k, const void* v, int qkv_dtype,
                       const float* g, const float* beta, const float* h0, double* o,
                       double* hT, long B, long T, long H, long dk, long dv, int nthreads) {
    long bh, nbh = B * H;
    int err = 0;
    if (!q || !k || !v || !g || !beta || B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (qkv_dtype != ORACLE_F32 && qkv_dtype != ORACLE_BF16) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (bh = 0; bh < nbh; bh++) {
        long b = bh / H, h = bh % H, t, i, j;
        size_t sz = (size_t)dk * dv;
        double* S = (double*)malloc(sz * sizeof(double));
        double* buf = (double*)malloc((size_t)(3 * dk + 4 * dv) * sizeof(double));
        if (!S || !buf) {
            free(S);
            free(buf);
            err |= 1;
            continue;
        }
        double *qi = buf, *ki = buf + dk, *gi = buf + 2 * dk;
        double *vi = buf + 3 * dk, *kv = vi + dv, *u = kv + dv, *out = u + dv;
        const size_t st_off = (size_t)(b * H + h) * sz;
        for (i = 0; i < (long)sz; i++) S[i] = h0 ? (double)h0[st_off + i] : 0.0;
        for (t = 0; t < T; t++) {
            size_t row = (size_t)((b * T + t) * H + h);
            for (i = 0; i < dk; i++) {
                qi[i] = load_elem(q, qkv_dtype, row * dk + i);
                ki[i] = load_elem(k, qkv_dtype, row * dk + i);
                gi[i] = (double)g[row * dk + i];
            }
            for (j = 0; j < dv; j++) vi[j] = load_elem(v, qkv_dtype, row * dv + j);
            kda_token(S, dk, dv, qi, ki, gi, vi, (double)beta[row], kv, u, out);
            if (o)
                for (j = 0; j < dv; j++) o[row * dv + j] = out[j];
        }
        if (hT)
            for (i = 0; i < (long)sz; i++) hT[st_off + i] = S[i];
        free(S);
        free(buf);
    }
    return err ? -2 : 0;
}

/*
 * Decode: one token per sequence, applied in place to S[N][H][dk][dv] (fp64).
 * q, k, g: [N, H, dk]; v, o: [N, H, dv]; beta: [N, H].
 */
int kda_oracle_decode(const void* q, const void* k, const void* v, int qkv_dtype,
                      const float* g, const float* beta, double* S, double* o, long N,
                      long H, long dk, long dv, int nthreads) {
    long nh, tot = N * H;
    int err = 0;
    if (!q || !k || !v || !g || !beta || !S || N < 0 || H < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (qkv_dtype != ORACLE_F32 && qkv_dtype != ORACLE_BF16) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(static) reduction(| : err)
    for (nh = 0; nh < tot; nh++) {
        long i, j;
        double* buf = (double*)malloc((size_t)(3 * dk + 4 * dv) * sizeof(double));
        if (!buf) {
            err |= 1;
            continue;
        }
        double *qi = buf, *ki = buf + dk, *gi = buf + 2 * dk;
        double *vi = buf + 3 * dk, *kv = vi + dv, *u = kv + dv, *out = u + dv;
        for (i = 0; i < dk; i++) {
            qi[i] = load_elem(q, qkv_dtype, (size_t)nh * dk + i);
            ki[i] = load_elem(k, qkv_dtype, (size_t)nh * dk + i);
            gi[i] = (double)g[(size_t)nh * dk + i];
        }
        for (j = 0; j < dv; j++) vi[j] = load_elem(v, qkv_dtype, (size_t)nh * dv + j);
        kda_token(S + (size_t)nh * dk * dv, dk, dv, qi, ki, gi, vi, (double)beta[nh], kv, u,
                  out);
        if (o)
            for (j = 0; j < dv; j++) o[(size_t)nh * dv + j] = out[j];
        free(buf);
    }
    return err ? -2 : 0;
}

/* Number of threads the OpenMP runtime will use (for reporting). */
int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
