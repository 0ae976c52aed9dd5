/*
 * Float64 CPU oracle for paged grouped-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (textbook definition, no blocking, no fusion, no reordering):
 *
 *   For every sequence b and query head h:
 *     kv      = h / G,  G = Hq / Hkv            (contiguous head groups)
 *     k_t,v_t = the t-th logical token of sequence b, for t in [0, L_b),
 *               found in physical block block_table[b][t / bs] at slot t % bs
 *     s_t     = scale * sum_d q[b,h,d] * k_t[d]
 *     out     = sum_t exp(s_t - max s) v_t / sum_t exp(s_t - max s)
 *
 * Passages followed:
 *   - "Modern LLM Inference - Workloads, Bottlenecks, and Optimization
 *     Techniques" (Stanford LLM lecture 11 notes), section "Why Cross-Layer
 *     Attention Shares K/V but Not Q", equation Attention(Q,K,V) =
 *     softmax(Q K^T / sqrt(d)) V.  The 1/sqrt(d) factor is the `scale` argument.
 *   - same notes, section 4.1 "Grouped-Query Attention": N query heads share K
 *     key/value heads, each KV head serving one group of query heads.
 *   - "The Ultimate Guide to LLM Inference Optimization - Part 2", section
 *     "Grouped Query Attention" (num heads divisible by num kv groups) and
 *     section "Paged Attention" (fixed-size blocks, e.g. 16 tokens, and a block
 *     table mapping a request's logical sequence to physical blocks).
 *   - itinai.com page on packed variable-length batches and GQA: the 5-D query
 *     layout [batch, seq, groups, per-group heads, dim] with a singleton KV head
 *     axis, which fixes the contiguous grouping kv = h / G.
 *   - "Advanced Optimizations: MQA, GQA, and PagedAttention", section
 *     "PagedAttention: The OS Analogy": the model sees a continuous logical
 *     sequence while the data is scattered over physical blocks.
 *
 * Extension (oracle_decode_ex_f64): q_len query tokens per sequence, the last
 * q_len cached tokens, each attending causally to the tokens up to its own
 * position, optionally only to the most recent `window` of them.  Passages:
 * speculative decoding checks several drafted tokens at once ("Modern LLM
 * Inference ...", section 7.1); local attention restricts each token to the
 * most recent K tokens (same notes, section 4.4 "Local Attention").
 *
 * Extension (oracle_decode_q8_f64): quantized K/V pages holding 8-bit codes,
 * e4m3 floats or signed int8 integers, each standing for a scale times its
 * value; one scale per KV head, or one per physical block and KV head (the
 * scale of a token is the one of the block it is stored in).  Passages: int8
 * and fp8 quantization ("Modern LLM Inference ...", section 6) and KV cache
 * compression ("The Ultimate Guide ... Part 2", section "KV Cache
 * Compression").
 *
 * Readings where the pages are silent:
 *   - seq_lens[b] counts the cached tokens; the single decode query attends to
 *     all of them (no causal mask for one query token).
 *   - With q_len query tokens, query i is the token at position
 *     L - q_len + i and attends to positions [lo, L - q_len + i]; window W > 0
 *     gives lo = max(0, L - q_len + i - W + 1) (the query's own token counts
 *     as one of the W).  An empty range gives zeros.
 *   - L_b == 0 gives an all-zero output row.
 *   - A block id outside [0, num_blocks) or L_b outside [0, max_blocks*bs]
 *     gives NaN for the affected rows and a non-zero return code.
 *   - Inputs are read in their stored type and widened exactly to double
 *     (bf16 -> float is exact by appending 16 zero bits; float -> double is
 *     exact).  All arithmetic is double with libm exp().
 *
 * Parallelised over (b, h) rows with OpenMP when compiled with -fopenmp; each
 * row is computed by one thread in the order written above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_FP8_E4M3 = 2, ORACLE_INT8 = 3 };
enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_BLOCK_ID = 2, ORACLE_ERR_SEQ_LEN = 3 };

/*
 * An 8-bit float with 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa
 * bits, no infinities, all-ones exponent and mantissa = NaN: normal values
 * (-1)^s 2^(e-7) (1 + m/8), subnormal (e = 0) values (-1)^s 2^-6 (m/8).
 */
static double e4m3_value(uint8_t v)
{
    const int sign = v >> 7, e = (v >> 3) & 15, m = v & 7;
    double x;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) {
        x = ldexp((double)m / 8.0, -6);
    } else {
        x = ldexp(1.0 + (double)m / 8.0, e - 7);
    }
    return sign ? -x : x;
}

/* Exact widening of element `idx` of a float32, bfloat16, e4m3 or int8 array
 * (an int8 code is a two's-complement integer in [-128, 127]). */
static double load_elem(const void *base, int64_t idx, int dtype)
{
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[idx];
    }
    if (dtype == ORACLE_FP8_E4M3) {
        return e4m3_value(((const uint8_t *)base)[idx]);
    }
    if (dtype == ORACLE_INT8) {
        return (double)((const int8_t *)base)[idx];
    }
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * One output row out[0..D) for sequence b, query token i of q_len, query head
 * h.  Query i sits at position p = L - q_len + i of the sequence (the q_len
 * new tokens are the last ones in the cache) and attends to tokens
 * [lo, p], lo = max(0, p - window + 1) when window > 0, else 0 (causal, and
 * local attention keeps only the most recent `window` tokens).  An empty range
 * gives zeros.  Returns a status.
 *
 * Quantized pages: a stored K (V) element stands for a scale times its code
 * value.  Without scale arrays the scale is 1; with scale_per_block == 0 it
 * is k_scale[kv] (one per KV head); with scale_per_block == 1 it is
 * k_scale[phys * Hkv + kv], one per physical block and KV head, so tokens of
 * one sequence in different blocks may carry different scales.
 */
static int decode_row(const void *q, const void *k_pool, const void *v_pool,
                      const float *k_scale, const float *v_scale, int scale_per_block,
                      const int32_t *block_table, const int32_t *seq_lens, int dtype,
                      int kv_dtype,
                      int q_len, int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                      int max_blocks, int window, double scale, int b, int i, int h, double *out)
{
    const int G = Hq / Hkv;
    const int kv = h / G;
    const int64_t L = seq_lens[b];
    int d;

    if (L < 0 || L > (int64_t)max_blocks * block_size) {
        for (d = 0; d < D; ++d) out[d] = NAN;
        return ORACLE_ERR_SEQ_LEN;
    }
    for (d = 0; d < D; ++d) out[d] = 0.0;
    const int64_t p = L - q_len + i;
    int64_t lo = 0;
    if (window > 0 && p - window + 1 > 0) lo = p - window + 1;
    const int64_t n = p - lo + 1;
    if (n <= 0) return ORACLE_OK;

    /* Gather: physical (block, slot) of every attended token, checked first,
     * and the K / V scales of that token's block. */
    int64_t *row_base = (int64_t *)malloc((size_t)n * sizeof(int64_t));
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double *ks = (double *)malloc((size_t)n * sizeof(double));
    double *vs = (double *)malloc((size_t)n * sizeof(double));
    if (!row_base || !s || !ks || !vs) {
        free(row_base);
        free(s);
        free(ks);
        free(vs);
        for (d = 0; d < D; ++d) out[d] = NAN;
        return ORACLE_ERR_ARG;
    }
    for (int64_t t = 0; t < n; ++t) {
        const int64_t tok = lo + t;
        int64_t phys = block_table[(int64_t)b * max_blocks + tok / block_size];
        int64_t slot = tok % block_size;
        if (phys < 0 || phys >= num_blocks) {
            free(row_base);
            free(s);
            free(ks);
            free(vs);
            for (d = 0; d < D; ++d) out[d] = NAN;
            return ORACLE_ERR_BLOCK_ID;
        }
        /* pool layout [num_blocks, block_size, Hkv, D] */
        row_base[t] = ((phys * block_size + slot) * Hkv + kv) * (int64_t)D;
        const int64_t sc_idx = scale_per_block ? phys * Hkv + kv : kv;
        ks[t] = k_scale ? (double)k_scale[sc_idx] : 1.0;
        vs[t] = v_scale ? (double)v_scale[sc_idx] : 1.0;
    }

    /* Scores s_t = scale * <q, k_t>; q layout [B, q_len, Hq, D]. */
    const int64_t q_base = (((int64_t)b * q_len + i) * Hq + h) * (int64_t)D;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (d = 0; d < D; ++d) {
            dot += load_elem(q, q_base + d, dtype) *
                   (ks[t] * load_elem(k_pool, row_base[t] + d, kv_dtype));
        }
        s[t] = scale * dot;
    }

    /* Softmax weights, max-subtracted for range, then the weighted mean of V. */
    double m = s[0];
    for (int64_t t = 1; t < n; ++t) {
        if (s[t] > m) m = s[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        s[t] = exp(s[t] - m);
        z += s[t];
    }
    for (int64_t t = 0; t < n; ++t) {
        for (d = 0; d < D; ++d) {
            out[d] += s[t] * (vs[t] * load_elem(v_pool, row_base[t] + d, kv_dtype));
        }
    }
    for (d = 0; d < D; ++d) out[d] /= z;

    free(row_base);
    free(s);
    free(ks);
    free(vs);
    return ORACLE_OK;
}

static int check_args(int dtype, int B, int Hq, int Hkv, int D, int block_size,
                      int64_t num_blocks, int max_blocks)
{
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_FP8_E4M3) return ORACLE_ERR_ARG;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return ORACLE_ERR_ARG;
    if (num_blocks < 0 || max_blocks < 0) return ORACLE_ERR_ARG;
    if (Hq % Hkv != 0) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/*
 * Selected rows.  rows[2*i], rows[2*i+1] = (b, h) of output row i; out is
 * [n_rows, D] doubles.  Returns the first non-zero row status, else 0.
 */
int oracle_decode_rows_f64(const void *q, const void *k_pool, const void *v_pool,
                           const int32_t *block_table, const int32_t *seq_lens, int dtype,
                           int B, int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                           int max_blocks, double scale, const int32_t *rows, int64_t n_rows,
                           double *out)
{
    int rc = check_args(dtype, B, Hq, Hkv, D, block_size, num_blocks, max_blocks);
    if (rc) return rc;
    for (int64_t i = 0; i < n_rows; ++i) {
        if (rows[2 * i] < 0 || rows[2 * i] >= B || rows[2 * i + 1] < 0 || rows[2 * i + 1] >= Hq)
            return ORACLE_ERR_ARG;
    }
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        int r = decode_row(q, k_pool, v_pool, NULL, NULL, 0, block_table, seq_lens, dtype, dtype,
                           1, Hq, Hkv, D,
                           block_size, num_blocks, max_blocks, 0, scale, rows[2 * i], 0,
                           rows[2 * i + 1], out + i * (int64_t)D);
        if (r) {
#pragma omp critical
            {
                if (!status) status = r;
            }
        }
    }
    return status;
}

/* Every row: out is [B, Hq, D] doubles. */
int oracle_decode_f64(const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *seq_lens, int dtype, int B,
                      int Hq, int Hkv, int D, int block_size, int64_t num_blocks, int max_blocks,
                      double scale, double *out)
{
    int rc = check_args(dtype, B, Hq, Hkv, D, block_size, num_blocks, max_blocks);
    if (rc) return rc;
    int status = ORACLE_OK;
    const int64_t n_rows = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        int r = decode_row(q, k_pool, v_pool, NULL, NULL, 0, block_table, seq_lens, dtype, dtype,
                           1, Hq, Hkv, D,
                           block_size, num_blocks, max_blocks, 0, scale, (int)(i / Hq), 0,
                           (int)(i % Hq), out + i * (int64_t)D);
        if (r) {
#pragma omp critical
            {
                if (!status) status = r;
            }
        }
    }
    return status;
}

/*
 * Several query tokens per sequence and an optional attention window:
 * q and out are [B, q_len, Hq, D]; seq_lens count every cached token, the
 * q_len query tokens included (they are the last q_len); window <= 0 means
 * no window.  With q_len = 1 and window = 0 this is oracle_decode_f64.
 */
static int decode_ex(const void *q, const void *k_pool, const void *v_pool, const float *k_scale,
                     const float *v_scale, int scale_per_block, const int32_t *block_table,
                     const int32_t *seq_lens,
                     int dtype, int kv_dtype, int B, int q_len, int Hq, int Hkv, int D,
                     int block_size, int64_t num_blocks, int max_blocks, int window,
                     double scale, double *out)
{
    int rc = check_args(dtype, B, Hq, Hkv, D, block_size, num_blocks, max_blocks);
    if (rc) return rc;
    if (q_len < 1) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
    const int64_t n_rows = (int64_t)B * q_len * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int h = (int)(r % Hq);
        const int i = (int)((r / Hq) % q_len);
        const int b = (int)(r / ((int64_t)Hq * q_len));
        int st = decode_row(q, k_pool, v_pool, k_scale, v_scale, scale_per_block, block_table,
                            seq_lens, dtype,
                            kv_dtype, q_len, Hq, Hkv, D,
                            block_size, num_blocks, max_blocks, window, scale, b, i, h,
                            out + r * (int64_t)D);
        if (st) {
#pragma omp critical
            {
                if (!status) status = st;
            }
        }
    }
    return status;
}

int oracle_decode_ex_f64(const void *q, const void *k_pool, const void *v_pool,
                         const int32_t *block_table, const int32_t *seq_lens, int dtype, int B,
                         int q_len, int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                         int max_blocks, int window, double scale, double *out)
{
    return decode_ex(q, k_pool, v_pool, NULL, NULL, 0, block_table, seq_lens, dtype, dtype, B, q_len,
                     Hq, Hkv, D, block_size, num_blocks, max_blocks, window, scale, out);
}

/*
 * 8-bit K/V pages: k_pool / v_pool hold 8-bit codes, `code` ORACLE_FP8_E4M3
 * (e4m3 bytes) or ORACLE_INT8 (signed integers); element (block, slot, head
 * kv, d) stands for a scale times the code's value.  scale_per_block == 0:
 * k_scale / v_scale hold one scale per KV head [Hkv]; 1: one per physical
 * block and KV head [num_blocks, Hkv].  q and out as in
 * oracle_decode_ex_f64, q in `q_dtype` (float32 or bfloat16).  Quantized KV
 * pages: "Modern LLM Inference ...", section 6 (int8 / fp8 quantization);
 * "The Ultimate Guide ... Part 2", "KV Cache Compression".
 */
int oracle_decode_q8_f64(const void *q, int q_dtype, const void *k_pool, const void *v_pool,
                         int code, const float *k_scale, const float *v_scale,
                         int scale_per_block, const int32_t *block_table,
                         const int32_t *seq_lens, int B, int q_len, int Hq, int Hkv, int D,
                         int block_size, int64_t num_blocks, int max_blocks, int window,
                         double scale, double *out)
{
    if (q_dtype != ORACLE_F32 && q_dtype != ORACLE_BF16) return ORACLE_ERR_ARG;
    if (code != ORACLE_FP8_E4M3 && code != ORACLE_INT8) return ORACLE_ERR_ARG;
    if (!k_scale || !v_scale || (scale_per_block != 0 && scale_per_block != 1))
        return ORACLE_ERR_ARG;
    return decode_ex(q, k_pool, v_pool, k_scale, v_scale, scale_per_block, block_table,
                     seq_lens, q_dtype, code, B, q_len, Hq, Hkv, D, block_size, num_blocks,
                     max_blocks, window, scale, out);
}

/* e4m3 pages with one scale per KV head (oracle_decode_q8_f64's first form). */
int oracle_decode_kv8_f64(const void *q, int q_dtype, const void *k_pool, const void *v_pool,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_table, const int32_t *seq_lens, int B, int q_len,
                          int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                          int max_blocks, int window, double scale, double *out)
{
    return oracle_decode_q8_f64(q, q_dtype, k_pool, v_pool, ORACLE_FP8_E4M3, k_scale, v_scale,
                                0, block_table, seq_lens, B, q_len, Hq, Hkv, D, block_size,
                                num_blocks, max_blocks, window, scale, out);
}

/* Threads OpenMP will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Use n threads from now on (n >= 1; ignored without OpenMP); returns the
 * count in effect.  Changes only how many rows run at once, never the
 * arithmetic of a row. */
int oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return oracle_num_threads();
}
