/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle of the PagedAttention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline / reference legs use it.  It shares no source with the CUDA
 * library and includes none of its headers.
 *
 * What it computes, and from which passage of the pages:
 *
 *  - KV blocks and the block table ("Inside vLLM v0.7: How PagedAttention &
 *    Chunked Prefill Scaled 10x Token Serving", section "Architectural
 *    Blueprint 2: How PagedAttention Actually Works"; "Inside vLLM
 *    Architecture", section "The Block Table Mapping Subsystem"): token p of a
 *    sequence lives in logical block p / block_size at offset p % block_size;
 *    the block table maps the logical block to a physical block of the pool.
 *  - Exactness ("Inside vLLM Architecture", section "Semantic FAQ Section",
 *    question "Does PagedAttention change the mathematical output of the
 *    LLM?"): paging changes only where K and V live, not the result.  So the
 *    oracle first gathers each sequence's K and V into contiguous fp64 arrays
 *    and then evaluates plain softmax(q K^T * scale) V, two-pass, in fp64.
 *  - Chunked prefill ("Inside vLLM v0.7 ...", section "Architectural
 *    Blueprint 3: Chunked Prefill"; "High-Throughput LLM Serving with vLLM &
 *    PagedAttention", section "5. Chunked Prefill & Latency SLA Management"):
 *    a chunk of prompt rows at absolute positions q_start + r attends,
 *    causally, to the paged context positions 0 .. q_start + r.
 *  - FP8 KV cache ("High-Throughput LLM Serving ...", section "4. Production
 *    vLLM Docker Deployment with FP8 Quantization", flag --kv-cache-dtype
 *    fp8): the pages name no format; the reading taken is OCP E4M3 ("e4m3fn")
 *    with one fp32 scale per tensor, store code = e4m3(x / scale), load
 *    code * scale.
 *  - Copy-on-write ("High-Throughput LLM Serving ...", section "2. Virtual
 *    Memory Paging Applied to GPUs: PagedAttention"): a diverging branch gets
 *    a fresh physical block holding a copy of the shared one.
 *
 * Readings where the pages are silent (all listed in the design notes):
 * query head h reads KV head h / (Hq / Hkv); a sequence of length 0 yields a
 * zero output; a negative slot is a padding token and is skipped; the causal
 * boundary is inclusive.
 *
 * Layouts (all row-major, element counts not bytes):
 *   cache pools  [num_blocks][num_kv_heads][block_size][head_dim]
 *   q            [num_seqs][num_q_heads][head_dim]          (decode)
 *   q_chunk      [total_q][num_q_heads][head_dim]          (prefill)
 *   k, v input   token t, head h, element e at  t*token_stride + h*head_dim + e
 *   block_tables [num_seqs][max_blocks_per_seq] int32
 *   out          fp64, same shape as q
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_FP8_E4M3 = 2 };
enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_RANGE = 2, OR_ERR_NOMEM = 3 };

/* ---------------------------------------------------------------- scalars */

/* IEEE 754 binary16 -> double, from the format definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits, subnormals at exponent 0. */
double or_f16_to_double(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* f * 2^-10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return s ? -v : v;
}

/* bfloat16 -> double: a bfloat16 is the upper half of an IEEE binary32. */
double or_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit E4M3 ("e4m3fn") -> double: 1 sign bit, 4 exponent bits (bias 7),
 * 3 fraction bits; exponent 0 is subnormal (f * 2^-9); there is no infinity;
 * S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448. */
double or_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 0xf, f = c & 0x7;
    double v;
    if (e == 0xf && f == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -v : v;
}

/* fp32 -> OCP E4M3, round to nearest (ties to even), saturating finite values
 * to +-448.  NaN maps to the NaN code.  Every step below is exact in double:
 * x is a float, scaling by a power of two is exact, and nearbyint rounds to
 * the nearest integer with ties to even under the default rounding mode. */
uint8_t or_e4m3_encode(float x)
{
    uint8_t sign;
    double a, r;
    int e;
    if (isnan(x))
        return 0x7f;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e;                    /* satfinite */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; rounding up to 8 * 2^-9 = 2^-6
         * lands exactly on the smallest normal, whose code is 0x08. */
        r = nearbyint(a * 512.0);
        return sign | (uint8_t)r;
    }
    (void)frexp(a, &e);                        /* a = m * 2^e, m in [0.5,1) */
    e -= 1;                                    /* a = (1+f) * 2^e, f in [0,1) */
    r = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (r >= 8.0) {                            /* rounded up to next binade */
        r = 0.0;
        e += 1;
    }
    {
        int code = ((e + 7) << 3) | (int)r;
        if (code > 0x7e)
            code = 0x7e;                       /* 464 and up already handled */
        return sign | (uint8_t)code;
    }
}

/* Element of a stored KV/q array, converted exactly to double; fp8 codes are
 * dequantised with their tensor scale. */
static double elem(const void *base, int64_t idx, int dtype, float scale)
{
    switch (dtype) {
    case OR_F16:
        return or_f16_to_double(((const uint16_t *)base)[idx]);
    case OR_BF16:
        return or_bf16_to_double(((const uint16_t *)base)[idx]);
    default:
        return or_e4m3_to_double(((const uint8_t *)base)[idx]) * (double)scale;
    }
}

/* ------------------------------------------------------------ cache write */

/* For each token t with slot_mapping[t] >= 0:
 *   cache[slot / block_size][h][slot % block_size][:] = x[t][h][:]
 * (the address arithmetic of PagedKVCacheManager.allocate_slot in "Inside
 * vLLM Architecture", section "The Block Table Mapping Subsystem").  A cache
 * of the input dtype receives the bits unchanged; an fp8 cache receives
 * e4m3(fp32(x) / scale) with an IEEE fp32 division, scale = k_scales[h]
 * (resp. v_scales[h]) for KV head h: one value per head, or the same value
 * for every head when the cache has one scale per tensor. */
int or_reshape_and_cache(const void *k, const void *v, int in_dtype,
                         int64_t num_tokens, int64_t token_stride,
                         const int64_t *slot_mapping, void *k_cache,
                         void *v_cache, int64_t num_blocks, int block_size,
                         int num_kv_heads, int head_dim, int kv_dtype,
                         const float *k_scales, const float *v_scales)
{
    int64_t t;
    if (in_dtype != OR_F16 && in_dtype != OR_BF16)
        return OR_ERR_ARG;
    if (kv_dtype != in_dtype && kv_dtype != OR_FP8_E4M3)
        return OR_ERR_ARG;
    for (t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t], blk, off;
        int h, e, side;
        if (slot < 0)
            continue;
        blk = slot / block_size;
        off = slot % block_size;
        if (blk >= num_blocks)
            return OR_ERR_RANGE;
        for (side = 0; side < 2; ++side) {
            const uint16_t *src = (const uint16_t *)(side ? v : k);
            void *dst = side ? v_cache : k_cache;
            for (h = 0; h < num_kv_heads; ++h)
                for (e = 0; e < head_dim; ++e) {
                    float sc = side ? v_scales[h] : k_scales[h];
                    int64_t si = t * token_stride + (int64_t)h * head_dim + e;
                    int64_t di = ((blk * num_kv_heads + h) * block_size + off) *
                                     head_dim + e;
                    if (kv_dtype == OR_FP8_E4M3) {
                        float xf = (float)elem(src, si, in_dtype, 1.0f);
                        volatile float qv = xf / sc;   /* fp32, IEEE division */
                        ((uint8_t *)dst)[di] = or_e4m3_encode(qv);
                    } else {
                        ((uint16_t *)dst)[di] = src[si];
                    }
                }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------ copy blocks */

/* Copy-on-write: for each pair (src, dst), in order, the whole physical block
 * (every head, slot and element) of both pools is copied bit for bit. */
int or_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                   int64_t block_bytes, const int32_t *pairs, int64_t num_pairs)
{
    int64_t i;
    for (i = 0; i < num_pairs; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || d < 0 || s >= num_blocks || d >= num_blocks)
            return OR_ERR_RANGE;
        memmove((char *)k_cache + d * block_bytes,
                (char *)k_cache + s * block_bytes, (size_t)block_bytes);
        memmove((char *)v_cache + d * block_bytes,
                (char *)v_cache + s * block_bytes, (size_t)block_bytes);
    }
    return OR_OK;
}

/* ------------------------------------------------------------- attention */

/* Gather positions 0..len-1 of one sequence and one KV head into contiguous
 * fp64 rows: row p comes from physical block table[p / bs], slot p % bs. */
static int gather(const void *cache, int dtype, float scale, int64_t num_blocks,
                  int bs, int hkv, int d, const int32_t *table, int g,
                  int64_t len, double *dst)
{
    int64_t p;
    int e;
    for (p = 0; p < len; ++p) {
        int64_t blk = table[p / bs];
        if (blk < 0 || blk >= num_blocks)
            return OR_ERR_RANGE;
        for (e = 0; e < d; ++e) {
            int64_t idx = ((blk * hkv + g) * bs + p % bs) * (int64_t)d + e;
            dst[p * d + e] = elem(cache, idx, dtype, scale);
        }
    }
    return OR_OK;
}

/* softmax(scale * q . K^T) V over the first n gathered rows, two-pass fp64.
 * n == 0 gives a zero row. */
static void attend(const double *qrow, const double *K, const double *V,
                   int64_t n, int d, double scale, double *s, double *out)
{
    int64_t p;
    int e;
    double m = -INFINITY, den = 0.0;
    for (e = 0; e < d; ++e)
        out[e] = 0.0;
    if (n == 0)
        return;
    for (p = 0; p < n; ++p) {
        double acc = 0.0;
        for (e = 0; e < d; ++e)
            acc += qrow[e] * K[p * d + e];
        s[p] = scale * acc;
        if (s[p] > m)
            m = s[p];
    }
    for (p = 0; p < n; ++p) {
        s[p] = exp(s[p] - m);
        den += s[p];
    }
    for (p = 0; p < n; ++p)
        for (e = 0; e < d; ++e)
            out[e] += s[p] * V[p * d + e];
    for (e = 0; e < d; ++e)
        out[e] /= den;
}

/* Decode: one query row per sequence.  seq_ids (may be NULL = all) selects
 * which sequences to evaluate; rows of unselected sequences are untouched. */
int or_decode(const void *q, int q_dtype, int num_seqs, int num_q_heads,
              const void *k_cache, const void *v_cache, int64_t num_blocks,
              int block_size, int num_kv_heads, int head_dim, int kv_dtype,
              const float *k_scales, const float *v_scales, const int32_t *block_tables,
              int max_blocks_per_seq, const int32_t *seq_lens, float scale,
              const int32_t *seq_ids, int num_ids, double *out)
{
    int n = seq_ids ? num_ids : num_seqs;
    int G, err = OR_OK;
    int64_t job;
    if (num_q_heads % num_kv_heads)
        return OR_ERR_ARG;
    G = num_q_heads / num_kv_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (job = 0; job < (int64_t)n * num_kv_heads; ++job) {
        int i = seq_ids ? seq_ids[job / num_kv_heads] : (int)(job / num_kv_heads);
        int g = (int)(job % num_kv_heads), j, e;
        int64_t L = seq_lens[i];
        double *K, *V, *s, *qrow;
        if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            err = OR_ERR_RANGE;
            continue;
        }
        K = (double *)malloc(sizeof(double) * (size_t)(L * head_dim + 1));
        V = (double *)malloc(sizeof(double) * (size_t)(L * head_dim + 1));
        s = (double *)malloc(sizeof(double) * (size_t)(L + 1));
        qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!K || !V || !s || !qrow) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else if (gather(k_cache, kv_dtype, k_scales[g], num_blocks, block_size,
                          num_kv_heads, head_dim,
                          block_tables + (int64_t)i * max_blocks_per_seq, g, L,
                          K) ||
                   gather(v_cache, kv_dtype, v_scales[g], num_blocks, block_size,
                          num_kv_heads, head_dim,
                          block_tables + (int64_t)i * max_blocks_per_seq, g, L,
                          V)) {
#pragma omp atomic write
            err = OR_ERR_RANGE;
        } else {
            for (j = 0; j < G; ++j) {
                int h = g * G + j;
                int64_t row = (int64_t)i * num_q_heads + h;
                for (e = 0; e < head_dim; ++e)
                    qrow[e] = elem(q, row * head_dim + e, q_dtype, 1.0f);
                attend(qrow, K, V, L, head_dim, (double)scale, s,
                       out + row * head_dim);
            }
        }
        free(K);
        free(V);
        free(s);
        free(qrow);
    }
    return err;
}

/* Chunked prefill: chunk c owns query rows cu_q_lens[c] .. cu_q_lens[c+1]-1;
 * row r of the chunk sits at absolute position q_start[c] + r and attends to
 * positions 0 .. q_start[c] + r (inclusive) of sequence c through
 * block_tables[c].  The work is shared among threads by (chunk, KV head,
 * block of OR_PREFILL_ROWS rows); each job gathers the keys its last row
 * sees and evaluates its rows exactly as above, so the split changes no
 * result. */
#define OR_PREFILL_ROWS 64
int or_prefill(const void *q, int q_dtype, const int32_t *cu_q_lens,
               const int32_t *q_start, int num_chunks, int num_q_heads,
               const void *k_cache, const void *v_cache, int64_t num_blocks,
               int block_size, int num_kv_heads, int head_dim, int kv_dtype,
               const float *k_scales, const float *v_scales, const int32_t *block_tables,
               int max_blocks_per_seq, float scale, double *out)
{
    int G, c, err = OR_OK;
    int64_t job, nrb = 1;
    if (num_q_heads % num_kv_heads)
        return OR_ERR_ARG;
    G = num_q_heads / num_kv_heads;
    for (c = 0; c < num_chunks; ++c) {
        int64_t len = cu_q_lens[c + 1] - cu_q_lens[c];
        int64_t rb = (len + OR_PREFILL_ROWS - 1) / OR_PREFILL_ROWS;
        if (rb > nrb)
            nrb = rb;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (job = 0; job < (int64_t)num_chunks * num_kv_heads * nrb; ++job) {
        int c = (int)(job / ((int64_t)num_kv_heads * nrb));
        int g = (int)((job / nrb) % num_kv_heads), j, e;
        int64_t r, len = cu_q_lens[c + 1] - cu_q_lens[c];
        int64_t r0 = (job % nrb) * OR_PREFILL_ROWS;
        int64_t r1 = r0 + OR_PREFILL_ROWS < len ? r0 + OR_PREFILL_ROWS : len;
        int64_t ctx = (int64_t)q_start[c] + r1;
        double *K, *V, *s, *qrow;
        if (len < 0 || q_start[c] < 0 ||
            (int64_t)q_start[c] + len > (int64_t)max_blocks_per_seq * block_size) {
#pragma omp atomic write
            err = OR_ERR_RANGE;
            continue;
        }
        if (r0 >= len)
            continue;
        K = (double *)malloc(sizeof(double) * (size_t)(ctx * head_dim + 1));
        V = (double *)malloc(sizeof(double) * (size_t)(ctx * head_dim + 1));
        s = (double *)malloc(sizeof(double) * (size_t)(ctx + 1));
        qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!K || !V || !s || !qrow) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else if (gather(k_cache, kv_dtype, k_scales[g], num_blocks, block_size,
                          num_kv_heads, head_dim,
                          block_tables + (int64_t)c * max_blocks_per_seq, g,
                          ctx, K) ||
                   gather(v_cache, kv_dtype, v_scales[g], num_blocks, block_size,
                          num_kv_heads, head_dim,
                          block_tables + (int64_t)c * max_blocks_per_seq, g,
                          ctx, V)) {
#pragma omp atomic write
            err = OR_ERR_RANGE;
        } else {
            for (r = r0; r < r1; ++r)
                for (j = 0; j < G; ++j) {
                    int h = g * G + j;
                    int64_t row = ((int64_t)cu_q_lens[c] + r) * num_q_heads + h;
                    for (e = 0; e < head_dim; ++e)
                        qrow[e] = elem(q, row * head_dim + e, q_dtype, 1.0f);
                    attend(qrow, K, V, q_start[c] + r + 1, head_dim,
                           (double)scale, s, out + row * head_dim);
                }
        }
        free(K);
        free(V);
        free(s);
        free(qrow);
    }
    return err;
}

/* ------------------------------------------------------------- threading */

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
