/*
 * orthros_ref.c -- plain CPU oracle for the Orthros attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the package smoke check and the benchmark's CPU
 * baseline do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (Orthros: Phase-Aware Heterogeneous Attention for Efficient
 * Transformers, paperz.arrangedbits.com full text):
 *   - Sec. 3.1, base query  q_t  = alpha  (.) q_t  + beta    (element-wise affine)
 *   - Sec. 3.1, output query q'_t = alpha' (.) q'_t + beta'
 *   - Sec. 3.1, Eq. 4: sliding-window attention of every position t over keys
 *     max(1, t-w+1) .. t (1-indexed; here 0-indexed: max(0, t-w+1) .. t)
 *   - Sec. 3.1, Eq. 5: full causal cross-attention of every output position t
 *     over keys 1 .. t (0-indexed: 0 .. t), against the same K/V
 *   - Sec. 3.2 "Decoding": the base token first appends its K/V to the cache,
 *     then runs Eq. 4; the output token runs Eq. 5 over the whole history.
 *   - Sec. 2.1, Eq. 1: the logit is q k^T / sqrt(d_h) (the scale is an argument).
 *   - Alg. 1, lines 6-7: heads are split after the affine, so alpha/beta hold
 *     one value per (query head, channel); grouped K/V heads follow the
 *     contiguous-group convention kv = h / (Hq / Hkv).
 *   - The backward of Eq. 4 / Eq. 5 and of the affines (training on the
 *     pre-training and fine-tuning regimes of Sec. 3.2 runs exactly these rows):
 *     the chain rule through softmax attention, written out per row (recompute
 *     p, then ds = p (dO.v - dO.o)); no formula for it is printed in the paper.
 *
 * Arithmetic: inputs are float (bf16 inputs are widened exactly by the caller);
 * every intermediate and every output is double. Softmax is the two-pass exact
 * form: max, then sum of exp(s - max). lse = max + ln(sum), natural log.
 * No blocking, fusion, online rescaling or reordering beyond the definition.
 *
 * Parallelism: OpenMP over independent (sequence, head, row) units only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_EINVAL 1
#define REF_ENOMEM 2

/*
 * One query row against the key range [lo, hi] (inclusive).
 * krow[j] / vrow[j] point at key / value j of the right K/V head.
 * qa is the already-affined query (double). Writes o[0..d) and *lse.
 * w is scratch of length hi - lo + 1.
 */
static void attend_row(const double *qa, const float *const *krow,
                       const float *const *vrow, int lo, int hi, int d,
                       double scale, double *o, double *lse, double *w)
{
    double m = -INFINITY;
    for (int j = lo; j <= hi; ++j) {
        const float *kj = krow[j];
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += qa[c] * (double)kj[c];
        double s = scale * dot;
        w[j - lo] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int j = lo; j <= hi; ++j) {
        double p = exp(w[j - lo] - m);
        const float *vj = vrow[j];
        l += p;
        for (int c = 0; c < d; ++c)
            o[c] += p * (double)vj[c];
    }
    for (int c = 0; c < d; ++c)
        o[c] /= l;
    *lse = m + log(l);
}

/* Sec. 3.1: scale-offset affine of one raw query row. */
static void affine(const float *qraw, const float *alpha, const float *beta,
                   int d, double *qa)
{
    for (int c = 0; c < d; ++c)
        qa[c] = (double)alpha[c] * (double)qraw[c] + (double)beta[c];
}

static int check_common(int B, int T, int Hq, int Hkv, int d, int window)
{
    if (B < 0 || T < 0 || Hq < 1 || Hkv < 1 || d < 1 || window < 1)
        return REF_EINVAL;
    if (Hq % Hkv != 0)
        return REF_EINVAL;
    return REF_OK;
}

/*
 * Prefill over B sequences of T tokens (Sec. 3.2 regimes PT / SFT / Prefill).
 *
 * q       [B, T, Hq, d]     raw (pre-affine) queries of the base tokens
 * k, v    [B, T, Hkv, d]
 * alpha_base, beta_base, alpha_out, beta_out   [Hq, d]
 * out_indptr [B+1], out_positions [n_out]: output rows of sequence b are
 *         out_positions[out_indptr[b] .. out_indptr[b+1]), positions in [0, T)
 * q_out   [n_out, Hq, d] raw output-stream queries, or NULL: then the raw
 *         query of output row r is q[b, out_positions[r]] (one shared Q
 *         projection, Alg. 1 line 5 with X_cross duplicated from X, Alg. 2).
 * base_rows, n_base_rows: if base_rows is NULL every position is computed and
 *         o_base is [B, T, Hq, d], lse_base [B, Hq, T]; otherwise only the
 *         listed positions are computed (for every b and h) and the outputs are
 *         compact: o_base [B, n_base_rows, Hq, d], lse_base [B, Hq, n_base_rows].
 *         n_base_rows = 0 with a non-NULL list computes no base rows.
 * o_out [n_out, Hq, d], lse_out [n_out, Hq]  (may be NULL when n_out == 0)
 */
int orthros_ref_prefill(const float *q, const float *k, const float *v,
                        const float *alpha_base, const float *beta_base,
                        const float *alpha_out, const float *beta_out,
                        const int32_t *out_indptr, const int32_t *out_positions,
                        const float *q_out, int B, int T, int Hq, int Hkv,
                        int d, int window, double scale,
                        const int32_t *base_rows, int n_base_rows,
                        double *o_base, double *lse_base, double *o_out,
                        double *lse_out, int nthreads)
{
    if (check_common(B, T, Hq, Hkv, d, window) != REF_OK)
        return REF_EINVAL;
    const int g = Hq / Hkv;
    const int nrows = base_rows ? n_base_rows : T;
    for (int i = 0; base_rows && i < n_base_rows; ++i)
        if (base_rows[i] < 0 || base_rows[i] >= T)
            return REF_EINVAL;
    const int n_out = out_indptr ? out_indptr[B] : 0;
    for (int b = 0; out_indptr && b < B; ++b)
        for (int r = out_indptr[b]; r < out_indptr[b + 1]; ++r)
            if (out_positions[r] < 0 || out_positions[r] >= T)
                return REF_EINVAL;

    /* key / value row tables: krow[b][kv][j] */
    const size_t ntab = (size_t)B * Hkv * (size_t)(T > 0 ? T : 1);
    const float **krow = (const float **)malloc(ntab * sizeof(*krow));
    const float **vrow = (const float **)malloc(ntab * sizeof(*vrow));
    if (!krow || !vrow) {
        free(krow);
        free(vrow);
        return REF_ENOMEM;
    }
    for (int b = 0; b < B; ++b)
        for (int kv = 0; kv < Hkv; ++kv)
            for (int j = 0; j < T; ++j) {
                size_t tab = ((size_t)b * Hkv + kv) * T + j;
                size_t off = (((size_t)b * T + j) * Hkv + kv) * (size_t)d;
                krow[tab] = k + off;
                vrow[tab] = v + off;
            }

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = REF_OK;

    /* base stream: Eq. 4 at every (b, h, listed position) */
    const long long nbase = (long long)B * Hq * nrows;
#pragma omp parallel
    {
        double *qa = (double *)malloc(sizeof(double) * d);
        double *o = (double *)malloc(sizeof(double) * d);
        double *w = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
        const int ok = qa && o && w;
        if (!ok) {
#pragma omp atomic write
            err = REF_ENOMEM;
        }
        {
#pragma omp for schedule(dynamic, 16)
            for (long long u = 0; u < nbase; ++u) {
                if (!ok)
                    continue;
                const int i = (int)(u % nrows);
                const int h = (int)((u / nrows) % Hq);
                const int b = (int)(u / ((long long)nrows * Hq));
                const int t = base_rows ? base_rows[i] : i;
                const int kv = h / g;
                const size_t qoff = (((size_t)b * T + t) * Hq + h) * (size_t)d;
                affine(q + qoff, alpha_base + (size_t)h * d,
                       beta_base + (size_t)h * d, d, qa);
                const int lo = t - window + 1 > 0 ? t - window + 1 : 0;
                const size_t tab = ((size_t)b * Hkv + kv) * T;
                double lse;
                attend_row(qa, krow + tab, vrow + tab, lo, t, d, scale, o, &lse, w);
                const size_t orow = (((size_t)b * nrows + i) * Hq + h) * (size_t)d;
                memcpy(o_base + orow, o, sizeof(double) * d);
                lse_base[((size_t)b * Hq + h) * nrows + i] = lse;
            }
        }
        free(qa);
        free(o);
        free(w);
    }

    /* output stream: Eq. 5 at every output row */
    const long long nout_units = (long long)n_out * Hq;
#pragma omp parallel
    {
        double *qa = (double *)malloc(sizeof(double) * d);
        double *o = (double *)malloc(sizeof(double) * d);
        double *w = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
        const int ok = qa && o && w;
        if (!ok) {
#pragma omp atomic write
            err = REF_ENOMEM;
        }
        {
#pragma omp for schedule(dynamic, 4)
            for (long long u = 0; u < nout_units; ++u) {
                if (!ok)
                    continue;
                const int r = (int)(u / Hq);
                const int h = (int)(u % Hq);
                int b = 0;
                while (out_indptr[b + 1] <= r)
                    ++b;
                const int t = out_positions[r];
                const int kv = h / g;
                const float *qraw =
                    q_out ? q_out + ((size_t)r * Hq + h) * (size_t)d
                          : q + (((size_t)b * T + t) * Hq + h) * (size_t)d;
                affine(qraw, alpha_out + (size_t)h * d,
                       beta_out + (size_t)h * d, d, qa);
                const size_t tab = ((size_t)b * Hkv + kv) * T;
                double lse;
                attend_row(qa, krow + tab, vrow + tab, 0, t, d, scale, o, &lse, w);
                memcpy(o_out + ((size_t)r * Hq + h) * (size_t)d, o,
                       sizeof(double) * d);
                lse_out[(size_t)r * Hq + h] = lse;
            }
        }
        free(qa);
        free(o);
        free(w);
    }

    free(krow);
    free(vrow);
    return err;
}

/*
 * One decoding step (Sec. 3.2 "Decoding", Sec. 3.1 decoupled pair) for B
 * sequences over a paged cache.
 *
 * q, q_out        [B, Hq, d] raw queries of the base / output token
 *                 (q_out NULL: the output token's raw query equals q)
 * k_new, v_new    [B, Hkv, d]
 * k_cache, v_cache [num_pages, page_size, Hkv, d]; token j of sequence b lives
 *                 in page block_table[b * max_pages + j / page_size], slot
 *                 j % page_size. MODIFIED: the new K/V is written at position
 *                 L = cache_lens[b] before either query runs.
 * cache_lens      [B] lengths before the append (not modified)
 * base row: keys max(0, L-w+1) .. L;  output row: keys 0 .. L.
 * o_base, o_out [B, Hq, d]; lse_base, lse_out [B, Hq]
 */
int orthros_ref_decode(const float *q, const float *q_out, const float *k_new,
                       const float *v_new, float *k_cache, float *v_cache,
                       const int32_t *block_table, int max_pages, int page_size,
                       int num_pages, const int32_t *cache_lens,
                       const float *alpha_base, const float *beta_base,
                       const float *alpha_out, const float *beta_out, int B,
                       int Hq, int Hkv, int d, int window, double scale,
                       double *o_base, double *lse_base, double *o_out,
                       double *lse_out, int nthreads)
{
    if (check_common(B, 1, Hq, Hkv, d, window) != REF_OK || page_size < 1 ||
        max_pages < 1 || num_pages < 1)
        return REF_EINVAL;
    const int g = Hq / Hkv;
    const size_t tok = (size_t)Hkv * d; /* floats per token in a page */
    int maxlen = 1;
    for (int b = 0; b < B; ++b) {
        const int L = cache_lens[b];
        if (L < 0 || L / page_size >= max_pages)
            return REF_EINVAL;
        for (int p = 0; p <= L / page_size; ++p) {
            const int pg = block_table[(size_t)b * max_pages + p];
            if (pg < 0 || pg >= num_pages)
                return REF_EINVAL;
        }
        if (L + 1 > maxlen)
            maxlen = L + 1;
    }

    /* append first: the base token updates the KV cache */
    for (int b = 0; b < B; ++b) {
        const int L = cache_lens[b];
        const int pg = block_table[(size_t)b * max_pages + L / page_size];
        const size_t off = ((size_t)pg * page_size + L % page_size) * tok;
        memcpy(k_cache + off, k_new + (size_t)b * tok, sizeof(float) * tok);
        memcpy(v_cache + off, v_new + (size_t)b * tok, sizeof(float) * tok);
    }

    const float **krow = (const float **)malloc(sizeof(*krow) * (size_t)B * Hkv * maxlen);
    const float **vrow = (const float **)malloc(sizeof(*vrow) * (size_t)B * Hkv * maxlen);
    if (!krow || !vrow) {
        free(krow);
        free(vrow);
        return REF_ENOMEM;
    }
    for (int b = 0; b < B; ++b)
        for (int kv = 0; kv < Hkv; ++kv)
            for (int j = 0; j <= cache_lens[b]; ++j) {
                const int pg = block_table[(size_t)b * max_pages + j / page_size];
                const size_t off =
                    ((size_t)pg * page_size + j % page_size) * tok + (size_t)kv * d;
                krow[((size_t)b * Hkv + kv) * maxlen + j] = k_cache + off;
                vrow[((size_t)b * Hkv + kv) * maxlen + j] = v_cache + off;
            }

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = REF_OK;
    const long long nunits = (long long)B * Hq * 2;
#pragma omp parallel
    {
        double *qa = (double *)malloc(sizeof(double) * d);
        double *w = (double *)malloc(sizeof(double) * maxlen);
        const int ok = qa && w;
        if (!ok) {
#pragma omp atomic write
            err = REF_ENOMEM;
        }
        {
#pragma omp for schedule(dynamic, 1)
            for (long long u = 0; u < nunits; ++u) {
                if (!ok)
                    continue;
                const int stream = (int)(u % 2); /* 0 base, 1 output */
                const int h = (int)((u / 2) % Hq);
                const int b = (int)(u / (2LL * Hq));
                const int L = cache_lens[b];
                const int kv = h / g;
                const size_t qoff = ((size_t)b * Hq + h) * (size_t)d;
                const size_t tab = ((size_t)b * Hkv + kv) * maxlen;
                double lse;
                if (stream == 0) {
                    affine(q + qoff, alpha_base + (size_t)h * d,
                           beta_base + (size_t)h * d, d, qa);
                    const int lo = L - window + 1 > 0 ? L - window + 1 : 0;
                    attend_row(qa, krow + tab, vrow + tab, lo, L, d, scale,
                               o_base + qoff, &lse, w);
                    lse_base[(size_t)b * Hq + h] = lse;
                } else {
                    affine((q_out ? q_out : q) + qoff, alpha_out + (size_t)h * d,
                           beta_out + (size_t)h * d, d, qa);
                    attend_row(qa, krow + tab, vrow + tab, 0, L, d, scale,
                               o_out + qoff, &lse, w);
                    lse_out[(size_t)b * Hq + h] = lse;
                }
            }
        }
        free(qa);
        free(w);
    }
    free(krow);
    free(vrow);
    return err;
}

/*
 * One continuous-batching step over the paged cache: Sec. 3.2 runs every
 * regime as the same computation (prefill then decoding agree exactly with
 * one longer prefill), so a step may append several tokens to a sequence (a
 * prefill chunk) or one (a decoding step) or none. Sequence b appends
 * n_b = new_indptr[b+1] - new_indptr[b] tokens (rows new_indptr[b] .. of
 * k_new/v_new/q) at positions L_b .. L_b + n_b - 1, L_b = cache_lens[b]; then
 *   - every new token's base row attends keys max(0, t-w+1) .. t (Eq. 4);
 *   - every output row r of sequence b (out_indptr, out_positions) at a
 *     position t in [0, L_b + n_b) attends keys 0 .. t (Eq. 5), with raw
 *     query q_out[r], or, when q_out is NULL, the q of the new token at t
 *     (t must then be a new position).
 * q [n_new,Hq,d], k_new/v_new [n_new,Hkv,d]; outputs o_base [n_new,Hq,d],
 * lse_base [n_new,Hq], o_out [n_out,Hq,d], lse_out [n_out,Hq]. The caches are
 * modified (the appends).
 */
int orthros_ref_extend(const float *q, const float *q_out, const float *k_new,
                       const float *v_new, float *k_cache, float *v_cache,
                       const int32_t *block_table, int max_pages, int page_size,
                       int num_pages, const int32_t *cache_lens,
                       const int32_t *new_indptr, const int32_t *out_indptr,
                       const int32_t *out_positions,
                       const float *alpha_base, const float *beta_base,
                       const float *alpha_out, const float *beta_out, int B,
                       int Hq, int Hkv, int d, int window, double scale,
                       double *o_base, double *lse_base, double *o_out,
                       double *lse_out, int nthreads)
{
    if (check_common(B, 1, Hq, Hkv, d, window) != REF_OK || page_size < 1 ||
        max_pages < 1 || num_pages < 1)
        return REF_EINVAL;
    const int g = Hq / Hkv;
    const size_t tok = (size_t)Hkv * d;
    int maxlen = 1;
    for (int b = 0; b < B; ++b) {
        const int L = cache_lens[b], n = new_indptr[b + 1] - new_indptr[b];
        if (L < 0 || n < 0 || (long long)L + n > (long long)max_pages * page_size)
            return REF_EINVAL;
        for (int p = 0; p * page_size < L + n; ++p) {
            const int pg = block_table[(size_t)b * max_pages + p];
            if (pg < 0 || pg >= num_pages)
                return REF_EINVAL;
        }
        for (int r = out_indptr[b]; r < out_indptr[b + 1]; ++r) {
            const int t = out_positions[r];
            if (t < 0 || t >= L + n || (!q_out && t < L))
                return REF_EINVAL;
        }
        if (L + n > maxlen)
            maxlen = L + n;
    }
    /* append first: the base tokens update the KV cache */
    for (int b = 0; b < B; ++b)
        for (int i = new_indptr[b]; i < new_indptr[b + 1]; ++i) {
            const int t = cache_lens[b] + (i - new_indptr[b]);
            const int pg = block_table[(size_t)b * max_pages + t / page_size];
            const size_t off = ((size_t)pg * page_size + t % page_size) * tok;
            memcpy(k_cache + off, k_new + (size_t)i * tok, sizeof(float) * tok);
            memcpy(v_cache + off, v_new + (size_t)i * tok, sizeof(float) * tok);
        }
    const float **krow = (const float **)malloc(sizeof(*krow) * (size_t)B * Hkv * maxlen);
    const float **vrow = (const float **)malloc(sizeof(*vrow) * (size_t)B * Hkv * maxlen);
    if (!krow || !vrow) {
        free(krow);
        free(vrow);
        return REF_ENOMEM;
    }
    for (int b = 0; b < B; ++b) {
        const int len = cache_lens[b] + new_indptr[b + 1] - new_indptr[b];
        for (int kv = 0; kv < Hkv; ++kv)
            for (int j = 0; j < len; ++j) {
                const int pg = block_table[(size_t)b * max_pages + j / page_size];
                const size_t off = ((size_t)pg * page_size + j % page_size) * tok + (size_t)kv * d;
                krow[((size_t)b * Hkv + kv) * maxlen + j] = k_cache + off;
                vrow[((size_t)b * Hkv + kv) * maxlen + j] = v_cache + off;
            }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int n_new = new_indptr[B], n_out = out_indptr[B];
    const long long nunits = ((long long)n_new + n_out) * Hq;
    int err = REF_OK;
#pragma omp parallel
    {
        double *qa = (double *)malloc(sizeof(double) * d);
        double *w = (double *)malloc(sizeof(double) * maxlen);
        const int ok = qa && w;
        if (!ok) {
#pragma omp atomic write
            err = REF_ENOMEM;
        }
#pragma omp for schedule(dynamic, 8)
        for (long long u = 0; u < nunits; ++u) {
            if (!ok)
                continue;
            const int h = (int)(u % Hq);
            const long long row = u / Hq;
            const int kv = h / g;
            double lse;
            if (row < n_new) { /* base row of a new token */
                const int i = (int)row;
                int b = 0;
                while (new_indptr[b + 1] <= i)
                    ++b;
                const int t = cache_lens[b] + (i - new_indptr[b]);
                const size_t qoff = ((size_t)i * Hq + h) * (size_t)d;
                const size_t tab = ((size_t)b * Hkv + kv) * maxlen;
                affine(q + qoff, alpha_base + (size_t)h * d, beta_base + (size_t)h * d, d, qa);
                const int lo = t - window + 1 > 0 ? t - window + 1 : 0;
                attend_row(qa, krow + tab, vrow + tab, lo, t, d, scale, o_base + qoff, &lse, w);
                lse_base[(size_t)i * Hq + h] = lse;
            } else { /* output row */
                const int r = (int)(row - n_new);
                int b = 0;
                while (out_indptr[b + 1] <= r)
                    ++b;
                const int t = out_positions[r];
                const size_t roff = ((size_t)r * Hq + h) * (size_t)d;
                const size_t tab = ((size_t)b * Hkv + kv) * maxlen;
                const float *qraw = q_out ? q_out + roff
                                          : q + ((size_t)(new_indptr[b] + t - cache_lens[b]) * Hq + h) * (size_t)d;
                affine(qraw, alpha_out + (size_t)h * d, beta_out + (size_t)h * d, d, qa);
                attend_row(qa, krow + tab, vrow + tab, 0, t, d, scale, o_out + roff, &lse, w);
                lse_out[(size_t)r * Hq + h] = lse;
            }
        }
        free(qa);
        free(w);
    }
    free(krow);
    free(vrow);
    return err;
}

/*
 * The projection feeding the hot path (Alg. 1 lines 4-5; Sec. 3.1): the base
 * tokens' hidden rows x and the output tokens' rows x' go through one shared
 * Q/K/V weight, y = x W (W [d_model, (Hq + 2 Hkv) d] stored transposed as
 * w_t [(Hq + 2 Hkv) d, d_model]); the query part gets its stream's affine,
 * q = alpha (.) y_Q + beta, and the base tokens' K/V parts are the cache
 * entries (only the base stream writes the cache). Rows 0 .. n_base-1 of x
 * are base tokens, rows n_base .. n_base+n_out-1 output tokens.
 * Outputs (double): q_base [n_base,Hq,d], q_out [n_out,Hq,d], k, v
 * [n_base,Hkv,d]; when k_cache is given, base row i is also written (as float)
 * to page block_table[token_seq[i]][token_pos[i] / page_size], slot
 * token_pos[i] % page_size.
 */
int orthros_ref_qkv_project(const float *x, int n_base, int n_out, int d_model,
                            const float *w_t, int Hq, int Hkv, int d,
                            const float *alpha_base, const float *beta_base,
                            const float *alpha_out, const float *beta_out,
                            double *q_base, double *q_out, double *k, double *v,
                            float *k_cache, float *v_cache, const int32_t *block_table,
                            int max_pages, int page_size, int num_pages,
                            const int32_t *token_seq, const int32_t *token_pos, int nthreads)
{
    if (n_base < 0 || n_out < 0 || d_model < 1 || Hq < 1 || Hkv < 1 || d < 1)
        return REF_EINVAL;
    const int Nq = Hq * d, Nkv = Hkv * d, N = Nq + 2 * Nkv;
    if (k_cache) {
        for (int i = 0; i < n_base; ++i) {
            const int t = token_pos[i];
            if (t < 0 || t / page_size >= max_pages)
                return REF_EINVAL;
            const int pg = block_table[(size_t)token_seq[i] * max_pages + t / page_size];
            if (pg < 0 || pg >= num_pages)
                return REF_EINVAL;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const long long rows = (long long)n_base + n_out;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long r = 0; r < rows; ++r) {
        const int base = r < n_base;
        const float *xr = x + (size_t)r * d_model;
        for (int j = 0; j < (base ? N : Nq); ++j) {
            const float *wj = w_t + (size_t)j * d_model;
            double y = 0.0;
            for (int c = 0; c < d_model; ++c)
                y += (double)xr[c] * (double)wj[c];
            if (j < Nq) {
                if (base)
                    q_base[(size_t)r * Nq + j] = (double)alpha_base[j] * y + (double)beta_base[j];
                else
                    q_out[(size_t)(r - n_base) * Nq + j] = (double)alpha_out[j] * y + (double)beta_out[j];
            } else if (j < Nq + Nkv) {
                k[(size_t)r * Nkv + (j - Nq)] = y;
            } else {
                v[(size_t)r * Nkv + (j - Nq - Nkv)] = y;
            }
        }
    }
    if (k_cache) {
        for (int i = 0; i < n_base; ++i) {
            const int t = token_pos[i];
            const int pg = block_table[(size_t)token_seq[i] * max_pages + t / page_size];
            const size_t off = ((size_t)pg * page_size + t % page_size) * (size_t)Nkv;
            for (int c = 0; c < Nkv; ++c) {
                k_cache[off + c] = (float)k[(size_t)i * Nkv + c];
                v_cache[off + c] = (float)v[(size_t)i * Nkv + c];
            }
        }
    }
    return REF_OK;
}

/*
 * Gradient of one query row's output (Eq. 4 / Eq. 5) given dO: recomputes the
 * row's exact softmax in double, then
 *   D = dO . o,  dp_j = dO . v_j,  ds_j = p_j (dp_j - D),
 *   dqa += scale sum_j ds_j k_j,  dk_j += scale ds_j qa,  dv_j += p_j dO.
 * krow/vrow/dkrow/dvrow[j] point at key j's rows. w is scratch (hi-lo+1).
 */
static void attend_row_backward(const double *qa, const float *dO, const float *const *krow,
                                const float *const *vrow, double *const *dkrow, double *const *dvrow,
                                int lo, int hi, int d, double scale, double *dqa, double *w, double *o)
{
    double m = -INFINITY;
    for (int j = lo; j <= hi; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += qa[c] * (double)krow[j][c];
        w[j - lo] = scale * dot;
        if (w[j - lo] > m)
            m = w[j - lo];
    }
    double l = 0.0;
    for (int j = lo; j <= hi; ++j) {
        w[j - lo] = exp(w[j - lo] - m);
        l += w[j - lo];
    }
    for (int c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int j = lo; j <= hi; ++j) {
        w[j - lo] /= l; /* p_j */
        for (int c = 0; c < d; ++c)
            o[c] += w[j - lo] * (double)vrow[j][c];
    }
    double D = 0.0;
    for (int c = 0; c < d; ++c)
        D += (double)dO[c] * o[c];
    for (int c = 0; c < d; ++c)
        dqa[c] = 0.0;
    for (int j = lo; j <= hi; ++j) {
        const double p = w[j - lo];
        double dp = 0.0;
        for (int c = 0; c < d; ++c)
            dp += (double)dO[c] * (double)vrow[j][c];
        const double ds = p * (dp - D);
        for (int c = 0; c < d; ++c) {
            dqa[c] += scale * ds * (double)krow[j][c];
            dkrow[j][c] += scale * ds * qa[c];
            dvrow[j][c] += p * (double)dO[c];
        }
    }
}

/*
 * Backward of orthros_ref_prefill: gradients of a loss L given dL/do_base
 * (do_base [B,T,Hq,d]) and dL/do_out (do_out [n_out,Hq,d]); lse is treated as
 * an output the loss does not use.
 *
 * Outputs (double, overwritten): dq [B,T,Hq,d] (raw base queries; also
 * receives the output rows' gradient when q_out is NULL, since those rows
 * read q at their position), dk, dv [B,T,Hkv,d], dq_out [n_out,Hq,d] (only
 * when q_out is given), d_alpha_base, d_beta_base, d_alpha_out, d_beta_out
 * [Hq,d]. Through the affine q = alpha (.) q_raw + beta (Sec. 3.1):
 * dq_raw = alpha (.) dqa, dalpha += dqa (.) q_raw, dbeta += dqa.
 * Only rows (of either stream) at positions in [row_lo, row_hi) contribute:
 * the full gradient is [0, T). A range [t0, T) still gives the exact dk, dv of
 * every key j >= t0 (no row before t0 sees such a key) and the exact dq of the
 * rows in the range, at a fraction of the cost on long sequences.
 * Parallel over kv heads only (each owns its K/V, query heads and affine rows).
 */
int orthros_ref_prefill_backward(const float *q, const float *k, const float *v,
                                 const float *alpha_base, const float *beta_base,
                                 const float *alpha_out, const float *beta_out,
                                 const int32_t *out_indptr, const int32_t *out_positions,
                                 const float *q_out, int B, int T, int Hq, int Hkv,
                                 int d, int window, double scale,
                                 const float *do_base, const float *do_out, int row_lo, int row_hi,
                                 double *dq, double *dk, double *dv, double *dq_out,
                                 double *d_alpha_base, double *d_beta_base,
                                 double *d_alpha_out, double *d_beta_out, int nthreads)
{
    if (check_common(B, T, Hq, Hkv, d, window) != REF_OK)
        return REF_EINVAL;
    const int g = Hq / Hkv;
    const int n_out = out_indptr ? out_indptr[B] : 0;
    for (int b = 0; out_indptr && b < B; ++b)
        for (int r = out_indptr[b]; r < out_indptr[b + 1]; ++r)
            if (out_positions[r] < 0 || out_positions[r] >= T)
                return REF_EINVAL;
    memset(dq, 0, sizeof(double) * (size_t)B * T * Hq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * T * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)B * T * Hkv * d);
    if (dq_out)
        memset(dq_out, 0, sizeof(double) * (size_t)n_out * Hq * d);
    memset(d_alpha_base, 0, sizeof(double) * (size_t)Hq * d);
    memset(d_beta_base, 0, sizeof(double) * (size_t)Hq * d);
    memset(d_alpha_out, 0, sizeof(double) * (size_t)Hq * d);
    memset(d_beta_out, 0, sizeof(double) * (size_t)Hq * d);
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = REF_OK;
    const size_t tt = T > 0 ? (size_t)T : 1;
#pragma omp parallel
    {
        const float **krow = (const float **)malloc(sizeof(*krow) * tt);
        const float **vrow = (const float **)malloc(sizeof(*vrow) * tt);
        double **dkrow = (double **)malloc(sizeof(*dkrow) * tt);
        double **dvrow = (double **)malloc(sizeof(*dvrow) * tt);
        double *qa = (double *)malloc(sizeof(double) * d);
        double *dqa = (double *)malloc(sizeof(double) * d);
        double *o = (double *)malloc(sizeof(double) * d);
        double *w = (double *)malloc(sizeof(double) * tt);
        const int ok = krow && vrow && dkrow && dvrow && qa && dqa && o && w;
        if (!ok) {
#pragma omp atomic write
            err = REF_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int kv = 0; kv < Hkv; ++kv) {
            if (!ok)
                continue;
            for (int b = 0; b < B; ++b) {
                for (int j = 0; j < T; ++j) {
                    const size_t off = (((size_t)b * T + j) * Hkv + kv) * (size_t)d;
                    krow[j] = k + off;
                    vrow[j] = v + off;
                    dkrow[j] = dk + off;
                    dvrow[j] = dv + off;
                }
                for (int h = kv * g; h < (kv + 1) * g; ++h) {
                    /* base stream, Eq. 4 */
                    for (int t = row_lo > 0 ? row_lo : 0; t < T && t < row_hi; ++t) {
                        const size_t qoff = (((size_t)b * T + t) * Hq + h) * (size_t)d;
                        affine(q + qoff, alpha_base + (size_t)h * d, beta_base + (size_t)h * d, d, qa);
                        const int lo = t - window + 1 > 0 ? t - window + 1 : 0;
                        attend_row_backward(qa, do_base + qoff, krow, vrow, dkrow, dvrow, lo, t, d, scale, dqa, w, o);
                        for (int c = 0; c < d; ++c) {
                            dq[qoff + c] += (double)alpha_base[(size_t)h * d + c] * dqa[c];
                            d_alpha_base[(size_t)h * d + c] += dqa[c] * (double)q[qoff + c];
                            d_beta_base[(size_t)h * d + c] += dqa[c];
                        }
                    }
                    /* output stream, Eq. 5 */
                    for (int r = out_indptr ? out_indptr[b] : 0; out_indptr && r < out_indptr[b + 1]; ++r) {
                        const int t = out_positions[r];
                        if (t < row_lo || t >= row_hi)
                            continue;
                        const size_t roff = ((size_t)r * Hq + h) * (size_t)d;
                        const size_t qoff = (((size_t)b * T + t) * Hq + h) * (size_t)d;
                        const float *qraw = q_out ? q_out + roff : q + qoff;
                        affine(qraw, alpha_out + (size_t)h * d, beta_out + (size_t)h * d, d, qa);
                        attend_row_backward(qa, do_out + roff, krow, vrow, dkrow, dvrow, 0, t, d, scale, dqa, w, o);
                        for (int c = 0; c < d; ++c) {
                            const double gq = (double)alpha_out[(size_t)h * d + c] * dqa[c];
                            if (q_out)
                                dq_out[roff + c] += gq;
                            else
                                dq[qoff + c] += gq;
                            d_alpha_out[(size_t)h * d + c] += dqa[c] * (double)qraw[c];
                            d_beta_out[(size_t)h * d + c] += dqa[c];
                        }
                    }
                }
            }
        }
        free(krow);
        free(vrow);
        free(dkrow);
        free(dvrow);
        free(qa);
        free(dqa);
        free(o);
        free(w);
    }
    return err;
}

/* Threads the OpenMP runtime would use (reported next to the CPU timing). */
int orthros_ref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
