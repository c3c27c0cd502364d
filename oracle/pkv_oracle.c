/*
 * pkv_oracle.c -- CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The CUDA library
 * never calls it and shares no code, header or constant with it.
 *
 * What it computes, written as the plain definition:
 *
 *  kv_store   For every new token t with out_loc[t] >= 0, the K and V rows of t
 *             ([Hkv, d] bf16 each) are copied bit for bit into pool slot
 *             out_loc[t] (mini-sglang "Engine Class", forward_batch: a batch
 *             carries out_loc; miniVLLM "Engine Architecture", prepare_prefill
 *             and prepare_decode: slot_mapping is the physical cache slot each
 *             new token is written to).  The pool is [num_pages, page_size,
 *             Hkv, d] (miniVLLM "Engine Architecture", allocate_kv_cache), so
 *             slot s is row s of the pool viewed as [num_pages*page_size, Hkv, d].
 *
 *  attention  For request r with n_r = cu_seqlens_q[r+1] - cu_seqlens_q[r]
 *             new tokens and seq_lens[r] = c_r + n_r tokens in total (c_r of
 *             them cached before this step: miniVLLM prepare_prefill skips
 *             num_cached_tokens), new token i sits at absolute position c_r + i
 *             and attends to key positions j = 0 .. c_r + i.  Key position j
 *             lives in physical page page_table[r, j / page_size] at offset
 *             j % page_size (mini-sglang "Engine Class", page_table maps
 *             logical to physical KV locations; miniVLLM block_tables map
 *             logical block to physical block).  Query head h reads KV head
 *             h / (Hq / Hkv) (grouped-query attention: miniVLLM "LLMEngine",
 *             num_heads / num_kv_heads).  With s_j = scale * <q, k_j>:
 *                 o = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m),  m = max_j s_j
 *             computed in two passes (max, then exponentials) in double
 *             precision from the exact bf16 values.  Decode is the case n_r = 1.
 *             The natural-log log-sum-exp m + log(sum_j exp(s_j - m)) of each
 *             row is returned too.
 *
 * Every function returns 0 on success or a positive error code; nothing is
 * written for a call that fails its argument checks.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_EARG = 1,       /* bad sizes or null pointers */
    ORACLE_EPAGE = 2,      /* a page id outside [0, num_pages) */
    ORACLE_ESEQLEN = 3,    /* seq_len larger than the page table row holds */
    ORACLE_ECUSEQ = 4,     /* cu_seqlens_q not monotone or beyond seq_lens */
    ORACLE_ESLOT = 5,      /* out_loc beyond the pool */
    ORACLE_ENOMEM = 6,
};

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int pkv_oracle_kv_store(const uint16_t *k_new, const uint16_t *v_new,
                        const int32_t *out_loc, int64_t T,
                        uint16_t *k_cache, uint16_t *v_cache,
                        int64_t num_slots, int Hkv, int d)
{
    if (T < 0 || Hkv <= 0 || d <= 0 || num_slots < 0)
        return ORACLE_EARG;
    if (T > 0 && (!k_new || !v_new || !out_loc || !k_cache || !v_cache))
        return ORACLE_EARG;
    for (int64_t t = 0; t < T; ++t)
        if (out_loc[t] >= num_slots)
            return ORACLE_ESLOT;
    const int64_t row = (int64_t)Hkv * d;
    for (int64_t t = 0; t < T; ++t) {
        if (out_loc[t] < 0)
            continue; /* padding token: nothing to store */
        const int64_t s = out_loc[t];
        memcpy(k_cache + s * row, k_new + t * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_cache + s * row, v_new + t * row, (size_t)row * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* Request that owns flat new-token index t (cu is monotone, cu[0] = 0). */
static int owner_of(const int32_t *cu, int B, int64_t t)
{
    int lo = 0, hi = B; /* answer in [lo, hi) with cu[r] <= t < cu[r+1] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (cu[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

/* One output row: new token t, query head h. */
static int attend_row(const uint16_t *q, const int32_t *cu, int B,
                      const uint16_t *k_cache, const uint16_t *v_cache,
                      int64_t num_pages, int page_size,
                      const int32_t *page_table, int64_t pt_stride,
                      const int32_t *seq_lens, int Hq, int Hkv, int d,
                      double scale, int64_t t, int h,
                      double *s, double *o, double *lse)
{
    const int r = owner_of(cu, B, t);
    const int64_t n = (int64_t)cu[r + 1] - cu[r];
    const int64_t c = (int64_t)seq_lens[r] - n;
    const int64_t i = t - cu[r];
    const int64_t nkeys = c + i + 1;
    const int g = h / (Hq / Hkv);
    const uint16_t *qrow = q + (t * Hq + h) * (int64_t)d;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const int64_t page = page_table[(int64_t)r * pt_stride + j / page_size];
        if (page < 0 || page >= num_pages)
            return ORACLE_EPAGE;
        const int64_t slot = page * page_size + j % page_size;
        const uint16_t *krow = k_cache + (slot * Hkv + g) * (int64_t)d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += bf16_value(qrow[e]) * bf16_value(krow[e]);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double l = 0.0;
    for (int e = 0; e < d; ++e)
        o[e] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const int64_t page = page_table[(int64_t)r * pt_stride + j / page_size];
        const int64_t slot = page * page_size + j % page_size;
        const uint16_t *vrow = v_cache + (slot * Hkv + g) * (int64_t)d;
        const double p = exp(s[j] - m);
        l += p;
        for (int e = 0; e < d; ++e)
            o[e] += p * bf16_value(vrow[e]);
    }
    for (int e = 0; e < d; ++e)
        o[e] /= l;
    if (lse)
        *lse = m + log(l);
    return ORACLE_OK;
}

/*
 * Attention for the rows listed in rows[0..n_rows) (each t*Hq + h), or for all
 * Tq*Hq rows when rows is NULL (then Tq = cu_seqlens_q[B]).  out receives
 * n_rows*d doubles in list order; lse (optional) n_rows doubles.
 * n_threads > 1 splits the rows over OpenMP threads.
 */
int pkv_oracle_attention(const uint16_t *q, const int32_t *cu_seqlens_q, int B,
                         const uint16_t *k_cache, const uint16_t *v_cache,
                         int64_t num_pages, int page_size,
                         const int32_t *page_table, int64_t pt_stride,
                         const int32_t *seq_lens, int Hq, int Hkv, int d,
                         double scale, const int64_t *rows, int64_t n_rows,
                         double *out, double *lse, int n_threads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0 || num_pages < 0 ||
        pt_stride < 0 || Hq % Hkv != 0)
        return ORACLE_EARG;
    if (B == 0)
        return ORACLE_OK;
    if (!q || !cu_seqlens_q || !k_cache || !v_cache || !page_table || !seq_lens || !out)
        return ORACLE_EARG;
    if (cu_seqlens_q[0] != 0)
        return ORACLE_ECUSEQ;
    int64_t max_keys = 0;
    for (int r = 0; r < B; ++r) {
        const int64_t n = (int64_t)cu_seqlens_q[r + 1] - cu_seqlens_q[r];
        if (n < 0 || seq_lens[r] < n)
            return ORACLE_ECUSEQ;
        if ((int64_t)seq_lens[r] > pt_stride * page_size)
            return ORACLE_ESEQLEN;
        if (seq_lens[r] > max_keys)
            max_keys = seq_lens[r];
    }
    const int64_t Tq = cu_seqlens_q[B];
    const int64_t total = rows ? n_rows : Tq * Hq;
    if (rows) {
        for (int64_t k = 0; k < n_rows; ++k)
            if (rows[k] < 0 || rows[k] >= Tq * Hq)
                return ORACLE_EARG;
    }
    if (n_threads < 1)
        n_threads = 1;

    int status = ORACLE_OK;
#ifdef _OPENMP
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double *s = (double *)malloc((size_t)(max_keys > 0 ? max_keys : 1) * sizeof(double));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_ENOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t k = 0; k < total; ++k) {
            if (!s)
                continue;
            const int64_t row = rows ? rows[k] : k;
            const int rc = attend_row(q, cu_seqlens_q, B, k_cache, v_cache, num_pages,
                                      page_size, page_table, pt_stride, seq_lens, Hq, Hkv,
                                      d, scale, row / Hq, (int)(row % Hq), s,
                                      out + k * d, lse ? lse + k : NULL);
            if (rc != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                status = rc;
            }
        }
        free(s);
    }
    return status;
}

int pkv_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
