/*
 * pagedkv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU statement of what the PagedAttention decode hot path
 * computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load this library; the product path never does.  It shares no code,
 * header, table or constant with the CUDA library: it has its own dtype codes, its
 * own element decoders and its own loops.
 *
 * Sources (four web pages about PagedAttention / vLLM):
 *  - "anthology-of-the-sota note-023", section Method: each sequence's KV cache is
 *    cut into fixed-size blocks of a fixed number of tokens; a per-sequence block
 *    table maps a logical block index to a physical block; the attention kernel
 *    gathers from those non-contiguous physical blocks.  Section Concepts: the
 *    kernel looks K/V up via the block table rather than in one contiguous buffer;
 *    copy-on-write gives a writer its own copy of a shared block.
 *  - "inferensys glossary: Paged Attention", paragraph 4: the gain comes from memory
 *    management alone and attention's arithmetic is left as it was.  So the
 *    result is exactly softmax(q K^T * scale) V over the gathered tokens.
 *  - "crackai.dev: Efficient Memory Management ... with PagedAttention", How It
 *    Works: pages hold the KV vectors of e.g. 16 tokens and are allocated as
 *    tokens are generated (the append); copy-on-write when a sharer diverges.
 *
 * Readings the pages leave open (they fix no layout, dtype or precision):
 *  - cache layout [num_blocks][num_kv_heads][block_size][head_dim];
 *    q and out [num_seqs][num_q_heads][head_dim];
 *    block_tables int32 [num_seqs][max_blocks_per_seq]; context_lens int32;
 *    slot = physical_block * block_size + offset (int64; negative = padding).
 *  - grouped-query attention: query head h reads KV head h / (num_q_heads/num_kv_heads).
 *  - an empty context (length 0) gives an all-zero output.
 *  - every element is decoded exactly to double; all arithmetic is in double.
 *
 * Parity pins (checked by the CPU test suite): the decoders against numpy/torch
 * conversions over all 65536 bit patterns; attention against brute force built from
 * contiguous per-sequence K/V, against a library softmax for identity block tables,
 * against closed forms (one token, two tokens, uniform keys), and under block
 * permutation / sharing invariants; append and block copy against a dictionary
 * model of the pool; the partition merge against the single pass.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 2, ORC_NO_MEMORY = 3 };

static size_t orc_elem_bytes(int dt) { return dt == ORC_F32 ? 4u : 2u; }

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double orc_half(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* zero / subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double orc_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double orc_load(const void* base, size_t i, int dt) {
    if (dt == ORC_F32) {
        float x;
        memcpy(&x, (const char*)base + 4 * i, 4);
        return (double)x;
    }
    uint16_t b;
    memcpy(&b, (const char*)base + 2 * i, 2);
    return dt == ORC_F16 ? orc_half(b) : orc_bf16(b);
}

int pkvo_decode(int32_t dtype, const void* src, int64_t n, double* dst) {
    if (dtype < 0 || dtype > 2 || n < 0 || (n && (!src || !dst))) return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_load(src, (size_t)i, dtype);
    return ORC_OK;
}

typedef struct {
    int32_t num_blocks, num_kv_heads, block_size, head_dim, dtype;
} orc_pool;

static int orc_pool_ok(const orc_pool* p) {
    return p->num_blocks > 0 && p->num_kv_heads > 0 && p->block_size > 0 && p->head_dim > 0 &&
           p->dtype >= 0 && p->dtype <= 2;
}

/* Element offset of (physical block b, kv head g, row r, dim 0) in a pool. */
static size_t orc_row(const orc_pool* p, int64_t b, int32_t g, int32_t r) {
    return (((size_t)b * p->num_kv_heads + g) * p->block_size + r) * p->head_dim;
}

/* Physical block holding logical token j of sequence s, or -1 if the table is bad. */
static int64_t orc_lookup(const orc_pool* p, const int32_t* tables, int32_t max_blocks, int32_t s,
                          int32_t j) {
    int32_t logical = j / p->block_size;
    if (logical >= max_blocks) return -1;
    int32_t b = tables[(size_t)s * max_blocks + logical];
    if (b < 0 || b >= p->num_blocks) return -1;
    return b;
}

/*
 * Attention of one query row (element offset qoff in q: the vector of sequence s,
 * query head h) over tokens [t0, t1) of the sequence:
 * scores s_j = scale * sum_d q[d] K_j[d]; m = max_j s_j; w_j = exp(s_j - m);
 * l = sum_j w_j; o[d] = sum_j w_j V_j[d] (NOT divided by l).  Returns ORC_OK or
 * ORC_BAD_INDEX.  For t1 <= t0: m = -inf, l = 0, o = 0.
 */
static int orc_head(const orc_pool* p, const void* q, size_t qoff, const void* kc, const void* vc,
                    const int32_t* tables, int32_t max_blocks, int32_t num_q_heads, int32_t s,
                    int32_t h, int32_t t0, int32_t t1, double scale, double* scores, double* m_out,
                    double* l_out, double* o) {
    const int32_t D = p->head_dim;
    const int32_t G = num_q_heads / p->num_kv_heads;
    const int32_t g = h / G;
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return ORC_OK;
    }
    double m = -INFINITY;
    for (int32_t j = t0; j < t1; ++j) {
        int64_t b = orc_lookup(p, tables, max_blocks, s, j);
        if (b < 0) return ORC_BAD_INDEX;
        size_t row = orc_row(p, b, g, j % p->block_size);
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += orc_load(q, qoff + d, p->dtype) * orc_load(kc, row + d, p->dtype);
        scores[j - t0] = scale * dot;
        if (scores[j - t0] > m) m = scores[j - t0];
    }
    double l = 0.0;
    for (int32_t j = t0; j < t1; ++j) {
        double w = exp(scores[j - t0] - m);
        size_t row = orc_row(p, orc_lookup(p, tables, max_blocks, s, j), g, j % p->block_size);
        l += w;
        for (int32_t d = 0; d < D; ++d) o[d] += w * orc_load(vc, row + d, p->dtype);
    }
    *m_out = m;
    *l_out = l;
    return ORC_OK;
}

static int orc_threads(int32_t requested) {
#ifdef _OPENMP
    return requested > 0 ? requested : omp_get_max_threads();
#else
    (void)requested;
    return 1;
#endif
}

/* Number of OpenMP threads a call with num_threads <= 0 would use. */
int32_t pkvo_max_threads(void) { return orc_threads(0); }

/*
 * out[s][h][:] = softmax_j(scale * q[s][h] . K_j) V_j over the context_lens[s] tokens
 * of sequence s, K_j / V_j read through block_tables from the pools.  Float64 result.
 */
int pkvo_attention_decode(const void* q, const void* k_cache, const void* v_cache, int32_t dtype,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, double scale, int32_t num_threads, double* out) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || num_seqs < 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads ||
        max_blocks_per_seq < 0 || (num_seqs && (!q || !k_cache || !v_cache || !context_lens || !out)))
        return ORC_BAD_ARG;
    int32_t max_len = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0) return ORC_BAD_ARG;
        if (context_lens[s] > max_len) max_len = context_lens[s];
    }
    if (max_len > 0 && !block_tables) return ORC_BAD_ARG;
    const int64_t pairs = (int64_t)num_seqs * num_q_heads;
    int status = ORC_OK;
#ifdef _OPENMP
#pragma omp parallel num_threads(orc_threads(num_threads))
#endif
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double m, l;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t i = 0; i < pairs; ++i) {
            int32_t s = (int32_t)(i / num_q_heads), h = (int32_t)(i % num_q_heads);
            double* o = out + (size_t)i * head_dim;
            if (!scores) {
                status = ORC_NO_MEMORY;
                continue;
            }
            int rc = orc_head(&p, q, (size_t)i * head_dim, k_cache, v_cache, block_tables,
                              max_blocks_per_seq, num_q_heads, s, h, 0, context_lens[s], scale,
                              scores, &m, &l, o);
            if (rc != ORC_OK) {
                status = rc;
                continue;
            }
            if (context_lens[s] > 0)
                for (int32_t d = 0; d < head_dim; ++d) o[d] /= l;
        }
        free(scores);
    }
    return status;
}

/*
 * Multi-token attention with a causal mask (prefill, chunked prefill): sequence s
 * brings n_s = query_start[s+1] - query_start[s] new tokens, the last n_s of its
 * context_lens[s] tokens (their K/V already written to the pool).  New token i sits
 * at position p = context_lens[s] - n_s + i and attends to tokens 0..p only.
 * q, out: [T][Hq][D], T = query_start[num_seqs]; sequence s's rows start at
 * query_start[s].  One new token per sequence is exactly decode.
 */
int pkvo_attention_prefill(const void* q, const void* k_cache, const void* v_cache, int32_t dtype,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, const int32_t* query_start,
                           int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks, double scale,
                           int32_t num_threads, double* out) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || num_seqs < 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads ||
        !query_start || (num_seqs && (!q || !k_cache || !v_cache || !context_lens || !out)))
        return ORC_BAD_ARG;
    int32_t max_len = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t n = query_start[s + 1] - query_start[s];
        if (n < 0 || context_lens[s] < n) return ORC_BAD_ARG;
        if (context_lens[s] > max_len) max_len = context_lens[s];
    }
    const int64_t rows = (int64_t)query_start[num_seqs] * num_q_heads;
    int status = ORC_OK;
#ifdef _OPENMP
#pragma omp parallel num_threads(orc_threads(num_threads))
#endif
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double m, l;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
        for (int64_t r = 0; r < rows; ++r) {
            const int32_t t = (int32_t)(r / num_q_heads), h = (int32_t)(r % num_q_heads);
            int32_t s = 0;
            while (query_start[s + 1] <= t) ++s;  /* the sequence owning token row t */
            const int32_t n = query_start[s + 1] - query_start[s];
            const int32_t pos = context_lens[s] - n + (t - query_start[s]);
            double* o = out + (size_t)r * head_dim;
            if (!scores) {
                status = ORC_NO_MEMORY;
                continue;
            }
            int rc = orc_head(&p, q, (size_t)r * head_dim, k_cache, v_cache, block_tables,
                              max_blocks_per_seq, num_q_heads, s, h, 0, pos + 1, scale, scores, &m,
                              &l, o);
            if (rc != ORC_OK) {
                status = rc;
                continue;
            }
            for (int32_t d = 0; d < head_dim; ++d) o[d] /= l;
        }
        free(scores);
    }
    return status;
}

/*
 * The same attention split into partitions of part_tokens consecutive logical tokens.
 * For partition pi of (s, h): m, l and the un-normalised o over tokens
 * [pi*part_tokens, min((pi+1)*part_tokens, len)).  Layout: m/l [S][Hq][max_parts],
 * o [S][Hq][max_parts][D].  Partitions past the end get m = -inf, l = 0, o = 0.
 */
int pkvo_attention_partitions(const void* q, const void* k_cache, const void* v_cache,
                              int32_t dtype, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int32_t num_blocks,
                              double scale, int32_t part_tokens, int32_t max_parts, double* m_out,
                              double* l_out, double* o_out) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || part_tokens <= 0 || max_parts <= 0 || num_q_heads % num_kv_heads)
        return ORC_BAD_ARG;
    double* scores = (double*)malloc(sizeof(double) * (size_t)part_tokens);
    if (!scores) return ORC_NO_MEMORY;
    int status = ORC_OK;
    for (int32_t s = 0; s < num_seqs && status == ORC_OK; ++s) {
        int32_t n = context_lens[s];
        if ((int64_t)max_parts * part_tokens < n) status = ORC_BAD_ARG;
        for (int32_t h = 0; h < num_q_heads && status == ORC_OK; ++h)
            for (int32_t pi = 0; pi < max_parts && status == ORC_OK; ++pi) {
                size_t k = ((size_t)s * num_q_heads + h) * max_parts + pi;
                int32_t t0 = pi * part_tokens;
                int32_t t1 = t0 + part_tokens < n ? t0 + part_tokens : n;
                status = orc_head(&p, q, ((size_t)s * num_q_heads + h) * head_dim, k_cache,
                                  v_cache, block_tables, max_blocks_per_seq, num_q_heads, s, h, t0,
                                  t1, scale, scores, &m_out[k], &l_out[k], o_out + k * head_dim);
            }
    }
    free(scores);
    return status;
}

/*
 * Combine partitions of one softmax: M = max_p m_p; c_p = exp(m_p - M);
 * out = sum_p c_p o_p / sum_p c_p l_p.  Partitions with l_p == 0 contribute nothing;
 * a row with no tokens at all gives zeros.  rows = S*Hq.
 */
int pkvo_merge_partitions(const double* m_in, const double* l_in, const double* o_in, int64_t rows,
                          int32_t max_parts, int32_t head_dim, double* out) {
    if (rows < 0 || max_parts <= 0 || head_dim <= 0) return ORC_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const double* m = m_in + r * max_parts;
        const double* l = l_in + r * max_parts;
        double M = -INFINITY;
        for (int32_t pi = 0; pi < max_parts; ++pi)
            if (l[pi] > 0.0 && m[pi] > M) M = m[pi];
        double* o = out + r * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (M == -INFINITY) continue;
        double L = 0.0;
        for (int32_t pi = 0; pi < max_parts; ++pi) {
            if (!(l[pi] > 0.0)) continue;
            double c = exp(m[pi] - M);
            L += c * l[pi];
            for (int32_t d = 0; d < head_dim; ++d) o[d] += c * o_in[(r * max_parts + pi) * head_dim + d];
        }
        for (int32_t d = 0; d < head_dim; ++d) o[d] /= L;
    }
    return ORC_OK;
}

/*
 * Cache append: new token t's K and V vectors go to slot slot_mapping[t], i.e. row
 * slot % block_size of physical block slot / block_size, for every KV head.  A
 * negative slot is padding and is skipped.  k, v: [T][Hkv][D].  Byte copies.
 */
int pkvo_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                   void* k_cache, void* v_cache, int32_t dtype, int32_t num_blocks,
                   int32_t num_kv_heads, int32_t block_size, int32_t head_dim) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || num_tokens < 0) return ORC_BAD_ARG;
    const size_t eb = orc_elem_bytes(dtype), row_bytes = eb * head_dim;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return ORC_BAD_INDEX;
        int64_t b = slot / block_size;
        int32_t r = (int32_t)(slot % block_size);
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            size_t src = ((size_t)t * num_kv_heads + g) * row_bytes;
            size_t dst = orc_row(&p, b, g, r) * eb;
            memcpy((char*)k_cache + dst, (const char*)k + src, row_bytes);
            memcpy((char*)v_cache + dst, (const char*)v + src, row_bytes);
        }
    }
    return ORC_OK;
}

/*
 * Copy-on-write block copy: for each (src, dst) pair, physical block dst of both
 * pools becomes a byte copy of block src (all KV heads, all rows).  Pairs are
 * applied in order.
 */
int pkvo_block_copy(const int64_t* pairs, int32_t num_pairs, void* k_cache, void* v_cache,
                    int32_t dtype, int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                    int32_t head_dim) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || num_pairs < 0) return ORC_BAD_ARG;
    const size_t block_bytes = orc_elem_bytes(dtype) * (size_t)num_kv_heads * block_size * head_dim;
    for (int32_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORC_BAD_INDEX;
        memcpy((char*)k_cache + dst * block_bytes, (const char*)k_cache + src * block_bytes, block_bytes);
        memcpy((char*)v_cache + dst * block_bytes, (const char*)v_cache + src * block_bytes, block_bytes);
    }
    return ORC_OK;
}

/*
 * The gather step alone: k_out[s][g][j][:] = row of logical token j of sequence s,
 * KV head g, for j < context_lens[s]; rows j >= len are left untouched.
 * k_out, v_out: [S][Hkv][max_len][D] in the cache dtype.  Byte copies.
 */
int pkvo_gather(const void* k_cache, const void* v_cache, int32_t dtype, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                int32_t num_blocks, int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                int32_t max_len, void* k_out, void* v_out) {
    orc_pool p = {num_blocks, num_kv_heads, block_size, head_dim, dtype};
    if (!orc_pool_ok(&p) || num_seqs < 0 || max_len < 0) return ORC_BAD_ARG;
    const size_t eb = orc_elem_bytes(dtype), row_bytes = eb * head_dim;
    for (int32_t s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0 || context_lens[s] > max_len) return ORC_BAD_ARG;
        for (int32_t j = 0; j < context_lens[s]; ++j) {
            int64_t b = orc_lookup(&p, block_tables, max_blocks_per_seq, s, j);
            if (b < 0) return ORC_BAD_INDEX;
            for (int32_t g = 0; g < num_kv_heads; ++g) {
                size_t dst = (((size_t)s * num_kv_heads + g) * max_len + j) * row_bytes;
                size_t src = orc_row(&p, b, g, j % block_size) * eb;
                memcpy((char*)k_out + dst, (const char*)k_cache + src, row_bytes);
                memcpy((char*)v_out + dst, (const char*)v_cache + src, row_bytes);
            }
        }
    }
    return ORC_OK;
}
