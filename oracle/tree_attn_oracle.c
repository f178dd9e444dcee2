/*
 * Float64 CPU oracle for single-query (decode) softmax attention and for the
 * partial states that Tree Attention merges.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the "obviously correct" restatement
 * that the CUDA library is checked against.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline / reference leg may load it; the
 * product path never calls it and shares no code, header or constant with it.
 *
 * Sources (web pages on Tree Attention, arXiv:2408.04093):
 *  - "Tree Attention Guide: Topology-Aware LLM Decoding" (aifetchly blog),
 *    section "Core Innovation 2: Mathematical Formulation of Online Softmax on
 *    Trees": the softmax over the whole sequence is defined with the global
 *    maximum logit (the Softmax(S)_j equation), and the merged tuple must equal
 *    that result exactly.
 *  - Same page, "Core Innovation 1", item 2 "Local Independent Partial
 *    Attention": the partial state of one KV slice is m = max(q K^T),
 *    l = sum exp(q K^T - m), o = sum exp(q K^T - m) V.
 *  - Same page, implementation listing ("local_attention"): logits are scaled
 *    by 1/sqrt(d_head) before the maximum is taken.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - scale: the caller passes it; 1/sqrt(d) unless stated otherwise.
 *  - GQA: query head h reads KV head h / (Hq/Hkv) (contiguous grouping).
 *  - lse = m + ln(l) in natural-log units; an empty sequence gives out = 0,
 *    lse = -inf (the identity state (o=0, l=0, m=-inf) normalised).
 *  - valid cache positions are [0, seqlens[b]); no causal mask (one query).
 *
 * Inputs are the exact stored values (FP32, or BF16 bit patterns) widened to
 * double; every sum is a plain left-to-right double sum.
 *
 * Layouts (all row-major, dense):
 *   q      [B][Hq][d]
 *   k, v   [B][Hkv][S][d]
 *   out    [B][Hq][d]      (double)
 *   lse    [B][Hq]         (double)
 *   partials: o [B][Hq][P][d], m and l [B][Hq][P]   (double)
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

/* Widen one stored element to double.  A BF16 value is the upper 16 bits of
 * an IEEE binary32, so widening is a 16-bit shift followed by a float read. */
static double widen(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    uint16_t bits = ((const uint16_t *)base)[idx];
    uint32_t word = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static int check_args(int B, int Hq, int Hkv, int d, int64_t S, int q_dtype, int kv_dtype)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || S < 0)
        return -3;
    if (Hq % Hkv != 0)
        return -3;
    if ((q_dtype != ORACLE_F32 && q_dtype != ORACLE_BF16) ||
        (kv_dtype != ORACLE_F32 && kv_dtype != ORACLE_BF16))
        return -4;
    return 0;
}

/* The definition: out[b,h,:] = sum_t softmax(s)_t V[b,g,t,:] with
 * s_t = scale * <q[b,h,:], K[b,g,t,:]>, g = h / (Hq/Hkv); lse = M + ln L.
 * Two passes over the tokens: logits and their maximum first, then the
 * exponentials, their sum and the weighted sum of V rows. */
int oracle_attention_f64(int B, int Hq, int Hkv, int d, int64_t S,
                         const void *q, int q_dtype,
                         const void *k, const void *v, int kv_dtype,
                         const int32_t *seqlens, double scale,
                         double *out, double *lse, int nthreads)
{
    int rc = check_args(B, Hq, Hkv, d, S, q_dtype, kv_dtype);
    if (rc)
        return rc;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > S)
            return -8;
    const int G = Hq / Hkv;
    const int64_t BH = (int64_t)B * Hq;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (int64_t bh = 0; bh < BH; ++bh) {
        const int b = (int)(bh / Hq);
        const int h = (int)(bh % Hq);
        const int g = h / G;
        const int64_t N = seqlens[b];
        const int64_t qoff = bh * d;
        const int64_t kvoff = ((int64_t)b * Hkv + g) * S * d;
        double *o = out + bh * d;
        if (N == 0) {
            for (int i = 0; i < d; ++i)
                o[i] = 0.0;
            lse[bh] = -INFINITY;
            continue;
        }
        double *s = (double *)malloc((size_t)N * sizeof(double));
        if (!s) {
            bad = 1;
            continue;
        }
        /* pass 1: scaled logits and their maximum */
        double M = -INFINITY;
        for (int64_t t = 0; t < N; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += widen(q, q_dtype, qoff + i) * widen(k, kv_dtype, kvoff + t * d + i);
            s[t] = scale * acc;
            if (s[t] > M)
                M = s[t];
        }
        /* pass 2: exponentials relative to the global maximum */
        double L = 0.0;
        for (int i = 0; i < d; ++i)
            o[i] = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            double w = exp(s[t] - M);
            L += w;
            for (int i = 0; i < d; ++i)
                o[i] += w * widen(v, kv_dtype, kvoff + t * d + i);
        }
        for (int i = 0; i < d; ++i)
            o[i] = o[i] / L;
        lse[bh] = M + log(L);
        free(s);
    }
    return bad ? -6 : 0;
}

/* Partial states of the local attention step, one per (b, h, p):
 * split p of batch row b covers tokens [starts[b*P+p], ends[b*P+p]) clipped
 * to [0, seqlens[b]).  m = max of the scaled logits in the slice,
 * l = sum exp(s - m), o = sum exp(s - m) V.  An empty slice yields the
 * identity state o = 0, l = 0, m = -inf. */
int oracle_partials_f64(int B, int Hq, int Hkv, int d, int64_t S,
                        const void *q, int q_dtype,
                        const void *k, const void *v, int kv_dtype,
                        const int32_t *seqlens, double scale,
                        int P, const int64_t *starts, const int64_t *ends,
                        double *po, double *pm, double *pl, int nthreads)
{
    int rc = check_args(B, Hq, Hkv, d, S, q_dtype, kv_dtype);
    if (rc)
        return rc;
    if (P <= 0)
        return -5;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > S)
            return -8;
    const int G = Hq / Hkv;
    const int64_t work = (int64_t)B * Hq * P;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (int64_t w = 0; w < work; ++w) {
        const int p = (int)(w % P);
        const int64_t bh = w / P;
        const int b = (int)(bh / Hq);
        const int h = (int)(bh % Hq);
        const int g = h / G;
        int64_t t0 = starts[(int64_t)b * P + p];
        int64_t t1 = ends[(int64_t)b * P + p];
        if (t0 < 0)
            t0 = 0;
        if (t1 > seqlens[b])
            t1 = seqlens[b];
        const int64_t qoff = bh * d;
        const int64_t kvoff = ((int64_t)b * Hkv + g) * S * d;
        double *o = po + w * d;
        for (int i = 0; i < d; ++i)
            o[i] = 0.0;
        if (t1 <= t0) {
            pm[w] = -INFINITY;
            pl[w] = 0.0;
            continue;
        }
        const int64_t n = t1 - t0;
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
            bad = 1;
            continue;
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += widen(q, q_dtype, qoff + i) * widen(k, kv_dtype, kvoff + (t0 + t) * d + i);
            s[t] = scale * acc;
            if (s[t] > m)
                m = s[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            double e = exp(s[t] - m);
            l += e;
            for (int i = 0; i < d; ++i)
                o[i] += e * widen(v, kv_dtype, kvoff + (t0 + t) * d + i);
        }
        pm[w] = m;
        pl[w] = l;
        free(s);
    }
    return bad ? -6 : 0;
}

/* Several queries per sequence (multi-query decode, e.g. verifying nq draft
 * tokens): q is [B][Hq][nq][d] and query i of row b sits at position
 * N_b - nq + i.  With `causal`, it attends to tokens [0, N_b - nq + i]
 * (max(0, N_b - nq + 1 + i) tokens); without, every query attends to all N_b.
 * For each (b, h, i) the result is the definition above over that token
 * range; out is [B][Hq][nq][d], lse [B][Hq][nq].  A query with no tokens
 * gives out = 0, lse = -inf. */
int oracle_attention_multi_f64(int B, int Hq, int Hkv, int d, int64_t S, int nq, int causal,
                               const void *q, int q_dtype,
                               const void *k, const void *v, int kv_dtype,
                               const int32_t *seqlens, double scale,
                               double *out, double *lse, int nthreads)
{
    int rc = check_args(B, Hq, Hkv, d, S, q_dtype, kv_dtype);
    if (rc)
        return rc;
    if (nq < 1)
        return -3;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > S)
            return -8;
    const int G = Hq / Hkv;
    const int64_t work = (int64_t)B * Hq * nq;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (int64_t w = 0; w < work; ++w) {
        const int i = (int)(w % nq);
        const int64_t bh = w / nq;
        const int b = (int)(bh / Hq);
        const int h = (int)(bh % Hq);
        const int g = h / G;
        int64_t n = seqlens[b];
        if (causal) {
            n = n - nq + 1 + i;
            if (n < 0)
                n = 0;
        }
        const int64_t qoff = w * d;
        const int64_t kvoff = ((int64_t)b * Hkv + g) * S * d;
        double *o = out + w * d;
        if (n == 0) {
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            lse[w] = -INFINITY;
            continue;
        }
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
            bad = 1;
            continue;
        }
        double M = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += widen(q, q_dtype, qoff + c) * widen(k, kv_dtype, kvoff + t * d + c);
            s[t] = scale * acc;
            if (s[t] > M)
                M = s[t];
        }
        double L = 0.0;
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            double e = exp(s[t] - M);
            L += e;
            for (int c = 0; c < d; ++c)
                o[c] += e * widen(v, kv_dtype, kvoff + t * d + c);
        }
        for (int c = 0; c < d; ++c)
            o[c] = o[c] / L;
        lse[w] = M + log(L);
        free(s);
    }
    return bad ? -6 : 0;
}

/* FP8 E4M3 (the "fn" variant: no infinities) widened to double from its
 * definition: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN. */
double oracle_e4m3_to_double(uint8_t x)
{
    const int sign = (x >> 7) & 1;
    const int e = (x >> 3) & 0xF;
    const int m = x & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Decode attention over an FP8 E4M3 cache with one scale per KV head:
 * K[b,g,t,i] = k_scale[g] * e4m3(k8[b,g,t,i]), V likewise with v_scale; q in
 * FP32 or BF16.  Otherwise the definition of oracle_attention_f64, with nq
 * queries per row as in oracle_attention_multi_f64 (nq = 1 for one). */
int oracle_attention_e4m3_f64(int B, int Hq, int Hkv, int d, int64_t S, int nq, int causal,
                              const void *q, int q_dtype, const uint8_t *k8, const uint8_t *v8,
                              const float *k_scale, const float *v_scale,
                              const int32_t *seqlens, double scale,
                              double *out, double *lse, int nthreads)
{
    int rc = check_args(B, Hq, Hkv, d, S, q_dtype, ORACLE_F32);
    if (rc)
        return rc;
    if (nq < 1)
        return -3;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > S)
            return -8;
    const int G = Hq / Hkv;
    const int64_t work = (int64_t)B * Hq * nq;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (int64_t w = 0; w < work; ++w) {
        const int i = (int)(w % nq);
        const int64_t bh = w / nq;
        const int b = (int)(bh / Hq);
        const int h = (int)(bh % Hq);
        const int g = h / G;
        int64_t n = seqlens[b];
        if (causal) {
            n = n - nq + 1 + i;
            if (n < 0)
                n = 0;
        }
        const double ks = (double)k_scale[g], vs = (double)v_scale[g];
        const int64_t qoff = w * d;
        const int64_t kvoff = ((int64_t)b * Hkv + g) * S * d;
        double *o = out + w * d;
        if (n == 0) {
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            lse[w] = -INFINITY;
            continue;
        }
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
            bad = 1;
            continue;
        }
        double M = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += widen(q, q_dtype, qoff + c) * (ks * oracle_e4m3_to_double(k8[kvoff + t * d + c]));
            s[t] = scale * acc;
            if (s[t] > M)
                M = s[t];
        }
        double L = 0.0;
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            double e = exp(s[t] - M);
            L += e;
            for (int c = 0; c < d; ++c)
                o[c] += e * (vs * oracle_e4m3_to_double(v8[kvoff + t * d + c]));
        }
        for (int c = 0; c < d; ++c)
            o[c] = o[c] / L;
        lse[w] = M + log(L);
        free(s);
    }
    return bad ? -6 : 0;
}

/* Number of OpenMP threads a call with nthreads <= 0 would use (1 when the
 * oracle was built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
