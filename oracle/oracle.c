/*
 * Paged KV-cache attention oracle: plain, slow, fp64, on the host.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file; only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *   - Attention(Q, K, V) = softmax(Q K^T / sqrt(d)) V, with the scale supplied
 *     by the caller (chengxuchu PyTorch #47, section 2.1).
 *   - Decode: the new token's K/V are first written into the cache, then the
 *     new query reads every cached K/V of its sequence (same page, section 2.2,
 *     and its pitfall 2).  So a decode query of a sequence with context length
 *     L attends to logical tokens 0 .. L-1.
 *   - Paging: fixed-size blocks that need not be contiguous, chained by a block
 *     table; the kernel "finds K/V through the block table" (ainews page,
 *     "PagedAttention"; chengxuchu #47 section 5.2; caffein.top "Paging").
 *     Logical token t of sequence s is row t % bs of physical block
 *     block_tables[s][t / bs]; layout of each cache is
 *     [num_blocks][num_kv_heads][bs][head_dim].
 *   - GQA: query head h reads kv head h / (Hq / Hkv) (chengxuchu #47, 2.3).
 *   - Chunked prefill: a prompt chunk of n tokens of a sequence whose cache
 *     holds L tokens after the append has its queries at positions
 *     L-n .. L-1; query j attends causally to tokens 0 .. L-n+j
 *     (caffein.top, "Chunked Prefill"; ainews page, continuous batching).
 *   - Copy-on-write: copy the whole forked block, K and V (ainews page,
 *     "PagedAttention", copy-on-write paragraph).
 *
 * The softmax is the textbook one: m = max_t x_t, w_t = exp(x_t - m),
 * out = sum_t w_t V_t / sum_t w_t, in double precision, one token at a time
 * in logical order.  A sequence with L = 0 gets an all-zero output row.
 *
 * Element types: 0 = IEEE binary32, 1 = bfloat16 (the upper 16 bits of a
 * binary32), 2 = fp8 E4M3 (quantised cache, chengxuchu #47 / the runtime
 * page on KV-cache memory, section 2.4: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 is subnormal, m * 2^-9; the code
 * S.1111.111 is NaN and there is no infinity, so the largest finite value
 * is 448).  An fp8 cache stores K / scale and V / scale with one scale per
 * kv head; reading multiplies back.  Every value is widened exactly to
 * double before use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG -1
#define ORC_BAD_INDEX -2

/* Value of an E4M3 code, from the format's definition. */
static double e4m3_value(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_e4m3_decode(uint8_t c) { return e4m3_value(c); }

/*
 * E4M3 code of a binary32 value: the nearest finite code, ties to the code
 * with an even mantissa (round to nearest even), magnitudes beyond 448 to
 * 448 (saturation); NaN to the NaN code.  Found by trying every code, the
 * plainest correct way.
 */
uint8_t oracle_e4m3_encode(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0;
    double a = fabs((double)f);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 127; c++) { /* every finite non-negative code */
        double err = fabs(e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

static double widen(const void *base, int64_t i, int dtype) {
    if (dtype == 2) return e4m3_value(((const uint8_t *)base)[i]);
    if (dtype == 0) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    } else {
        uint16_t h;
        uint32_t bits;
        float f;
        memcpy(&h, (const char *)base + 2 * i, 2);
        bits = ((uint32_t)h) << 16;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
}

static int elem_bytes(int dtype) { return dtype == 0 ? 4 : dtype == 1 ? 2 : 1; }

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the parallel loops that follow (n >= 1). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Write new tokens' K and V rows into their slots; slot < 0 is skipped. */
int oracle_kv_append(const void *k, const void *v, const int64_t *slot_mapping, int num_tokens,
                     void *k_cache, void *v_cache, int num_blocks, int num_kv_heads,
                     int block_size, int head_dim, int dtype) {
    int eb = elem_bytes(dtype);
    size_t row = (size_t)head_dim * eb;
    for (int i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return ORC_BAD_INDEX;
        int64_t blk = slot / block_size, r = slot % block_size;
        for (int g = 0; g < num_kv_heads; g++) {
            size_t src = ((size_t)i * num_kv_heads + g) * row;
            size_t dst = (((size_t)blk * num_kv_heads + g) * block_size + r) * row;
            memcpy((char *)k_cache + dst, (const char *)k + src, row);
            memcpy((char *)v_cache + dst, (const char *)v + src, row);
        }
    }
    return ORC_OK;
}

/*
 * Append into an fp8 E4M3 cache: each element x of token i, kv head g is
 * stored as the code of the binary32 quotient x / scale[g] (k_scale for K,
 * v_scale for V), x widened from in_dtype (0 binary32, 1 bfloat16).
 * Negative slots are skipped, as in oracle_kv_append.
 */
int oracle_kv_append_fp8(const void *k, const void *v, int in_dtype, const int64_t *slot_mapping,
                         int num_tokens, uint8_t *k_cache, uint8_t *v_cache, int num_blocks,
                         int num_kv_heads, int block_size, int head_dim, const float *k_scale,
                         const float *v_scale) {
    for (int i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return ORC_BAD_INDEX;
        int64_t blk = slot / block_size, r = slot % block_size;
        for (int g = 0; g < num_kv_heads; g++) {
            int64_t src = ((int64_t)i * num_kv_heads + g) * head_dim;
            int64_t dst = (((int64_t)blk * num_kv_heads + g) * block_size + r) * head_dim;
            for (int j = 0; j < head_dim; j++) {
                float xk = (float)widen(k, src + j, in_dtype), xv = (float)widen(v, src + j, in_dtype);
                k_cache[dst + j] = oracle_e4m3_encode(xk / k_scale[g]);
                v_cache[dst + j] = oracle_e4m3_encode(xv / v_scale[g]);
            }
        }
    }
    return ORC_OK;
}

/* Copy whole blocks (every kv head, every row) from src to dst, K and V. */
int oracle_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                       int num_blocks, int num_kv_heads, int block_size, int head_dim, int dtype) {
    size_t blk = (size_t)num_kv_heads * block_size * head_dim * elem_bytes(dtype);
    for (int i = 0; i < num_pairs; i++) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORC_BAD_INDEX;
        memmove((char *)k_cache + dst * blk, (const char *)k_cache + src * blk, blk);
        memmove((char *)v_cache + dst * blk, (const char *)v_cache + src * blk, blk);
    }
    return ORC_OK;
}

/*
 * Paged attention for one batch.  cu_q_lens == NULL means decode: sequence s
 * has exactly one query (row s of q) at position context_lens[s] - 1.
 * Otherwise sequence s owns query rows cu_q_lens[s] .. cu_q_lens[s+1]-1.
 * q is [rows][num_q_heads][head_dim]; out is [rows][num_q_heads][head_dim]
 * in double.
 */
int oracle_paged_attention(const void *q, int q_dtype, const void *k_cache, const void *v_cache,
                           int kv_dtype, const int32_t *block_tables, int max_blocks,
                           const int32_t *context_lens, const int32_t *cu_q_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, double scale, const float *k_scale, const float *v_scale,
                           double *out) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0) return ORC_BAD_ARG;
    int group = num_q_heads / num_kv_heads;
    int rows = cu_q_lens ? cu_q_lens[num_seqs] : num_seqs;
    /* map each query row to its sequence and absolute position */
    int *row_seq = (int *)malloc(sizeof(int) * (rows > 0 ? rows : 1));
    int *row_pos = (int *)malloc(sizeof(int) * (rows > 0 ? rows : 1));
    int status = ORC_OK;
    for (int s = 0; s < num_seqs; s++) {
        int L = context_lens[s];
        int first = cu_q_lens ? cu_q_lens[s] : s;
        int n = cu_q_lens ? cu_q_lens[s + 1] - cu_q_lens[s] : 1;
        if (L < 0 || L > max_blocks * block_size || (cu_q_lens && n > L)) status = ORC_BAD_ARG;
        for (int j = 0; j < n; j++) {
            row_seq[first + j] = s;
            row_pos[first + j] = L - n + j; /* decode: L - 1 */
        }
    }
    if (status != ORC_OK) {
        free(row_seq);
        free(row_pos);
        return status;
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t task = 0; task < (int64_t)rows * num_q_heads; task++) {
        int r = (int)(task / num_q_heads), h = (int)(task % num_q_heads);
        int s = row_seq[r], pos = row_pos[r];
        int g = h / group;
        int ntok = pos + 1; /* tokens 0 .. pos */
        double *o = out + ((size_t)r * num_q_heads + h) * head_dim;
        for (int j = 0; j < head_dim; j++) o[j] = 0.0;
        if (ntok <= 0) continue;
        double *x = (double *)malloc(sizeof(double) * ntok);
        /* per kv head dequantisation scales of an fp8 cache (1 otherwise) */
        const double ks = k_scale ? (double)k_scale[g] : 1.0, vs = v_scale ? (double)v_scale[g] : 1.0;
        const int32_t *table = block_tables + (size_t)s * max_blocks;
        int64_t qbase = ((int64_t)r * num_q_heads + h) * head_dim;
        /* logits x_t = scale * <q, K_t> */
        double m = -INFINITY;
        for (int t = 0; t < ntok; t++) {
            int32_t b = table[t / block_size];
            if (b < 0 || b >= num_blocks) {
                bad = 1;
                x[t] = -INFINITY;
                continue;
            }
            int64_t kbase = (((int64_t)b * num_kv_heads + g) * block_size + t % block_size) * head_dim;
            double acc = 0.0;
            for (int j = 0; j < head_dim; j++)
                acc += widen(q, qbase + j, q_dtype) * (widen(k_cache, kbase + j, kv_dtype) * ks);
            x[t] = scale * acc;
            if (x[t] > m) m = x[t];
        }
        /* softmax weights and the weighted sum of V rows */
        double den = 0.0;
        for (int t = 0; t < ntok; t++) {
            int32_t b = table[t / block_size];
            if (b < 0 || b >= num_blocks) continue;
            double w = exp(x[t] - m);
            den += w;
            int64_t vbase = (((int64_t)b * num_kv_heads + g) * block_size + t % block_size) * head_dim;
            for (int j = 0; j < head_dim; j++) o[j] += w * (widen(v_cache, vbase + j, kv_dtype) * vs);
        }
        for (int j = 0; j < head_dim; j++) o[j] /= den;
        free(x);
    }
    free(row_seq);
    free(row_pos);
    return bad ? ORC_BAD_INDEX : ORC_OK;
}
