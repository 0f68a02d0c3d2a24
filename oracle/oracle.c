/*
 * FP64 CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition, written with scalar loops:
 *
 *   - oracle_append: the append step of "Project 17: Production Serving:
 *     Continuous Batching and PagedAttention" (llm-under-the-hood), Step 4
 *     "Implement the paged KV cache": token t's key/value rows are stored at
 *     (physical page, slot in page).  Here the slot comes from slot_mapping
 *     (slot = page * block_size + offset, negative = padding, skipped), the
 *     per-step metadata of "Continuous Batching" (infra.pidoku.co.in) §6
 *     "Under the hood".  A bit copy.
 *
 *   - oracle_decode: Step 6 "Implement attention over paged storage" of the
 *     same Project 17 page: walk the page table, gather each stored key,
 *     score = q.k / sqrt(head_dim), softmax over the sequence, weighted sum of
 *     the gathered values.  Read per query head (each query head has its own
 *     scores and softmax) with grouped KV heads: query head h reads KV head
 *     h / (Hq / Hkv).  Context length counts this step's appended token
 *     (tiny-vllm part 7, "Uploading the active arrays to the GPU": the new
 *     token's K/V is written first, then attention reads length + 1).
 *
 *   - oracle_prefill: the same per query token of a chunk, with the causal
 *     rule of chunked prefill ("Continuous Batching" §5 "Mixed batching"):
 *     query i of a chunk of q_len tokens sits at absolute position
 *     ctx - q_len + i and attends keys 0 .. that position, inclusive.
 *
 *   - oracle_dense: the same attention on contiguous [ctx, Hkv, d] K/V with no
 *     block table (the brute-force comparison the paged form must equal).
 *
 *   - oracle_decode_range / oracle_merge: attention restricted to a token range
 *     returned as (max, sum, unnormalised accumulator), and the log-sum-exp
 *     combination of such partials.  Used to check that splitting the KV
 *     range and merging reproduces the unsplit result.
 *
 * Element storage: 16-bit inputs are passed as raw bit patterns (uint16) plus
 * a dtype flag (0 = IEEE fp16, 1 = bfloat16); this file decodes them to
 * double exactly.  Arithmetic is double precision throughout, max-subtracted
 * softmax with exp() from libm.  A sequence with context length 0 yields an
 * all-zero output row.
 *
 * Cache layout: k_cache and v_cache are each [num_blocks][Hkv][block_size][d];
 * every gather goes through cache_index(), so a layout change is one line.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* Exact decode of an IEEE binary16 bit pattern. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(mant | 0x400), expo - 25); /* (1.m) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Exact decode of a bfloat16 bit pattern: it is the top half of a float32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const uint16_t *p, int64_t i, int dtype) {
    return dtype == ORACLE_BF16 ? bf16_bits_to_double(p[i]) : half_bits_to_double(p[i]);
}

/* Index of element (block, kv head, offset in block, dim) in a paged cache. */
static int64_t cache_index(int64_t block, int h, int off, int i, int Hkv, int bs, int d) {
    return (((block * Hkv) + h) * (int64_t)bs + off) * d + i;
}

/* Decode every element of a 16-bit array to double (for the Python side). */
void oracle_decode_bits(const uint16_t *bits, int64_t n, int dtype, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = elem(bits, i, dtype);
}

/*
 * Append: for every new token t and KV head h, copy k[t][h][:] and v[t][h][:]
 * into the cache at slot_mapping[t] (block = slot / bs, offset = slot % bs).
 * Negative slots are padding and write nothing.  Returns the number of
 * (token, head) rows written, or -1 if a slot points outside the pool.
 */
int64_t oracle_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                      uint16_t *k_cache, uint16_t *v_cache, int NB, int bs, int Hkv, int d) {
    int64_t written = 0;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t block = slot / bs;
        int off = (int)(slot % bs);
        if (block >= NB) return -1;
        for (int h = 0; h < Hkv; ++h) {
            for (int i = 0; i < d; ++i) {
                int64_t src = ((int64_t)t * Hkv + h) * d + i;
                int64_t dst = cache_index(block, h, off, i, Hkv, bs, d);
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
            ++written;
        }
    }
    return written;
}

/*
 * Softmax attention of one query row over the keys at logical positions
 * [t0, t1) of one sequence, reached through its block-table row.
 * Writes (m, l, acc[d]) with m = max score, l = sum exp(score - m),
 * acc = sum exp(score - m) * v.  An empty range gives m = -inf, l = 0, acc = 0.
 */
static void attend_range(const uint16_t *qrow, int dtype, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *table_row, int t0, int t1,
                         int g, int Hkv, int bs, int d, double scale, double *m_out,
                         double *l_out, double *acc) {
    double m = -INFINITY;
    for (int i = 0; i < d; ++i) acc[i] = 0.0;
    /* pass 1: scores and their maximum */
    for (int t = t0; t < t1; ++t) {
        int64_t block = table_row[t / bs];
        int off = t % bs;
        double x = 0.0;
        for (int i = 0; i < d; ++i)
            x += elem(qrow, i, dtype) * elem(k_cache, cache_index(block, g, off, i, Hkv, bs, d), dtype);
        x *= scale;
        if (x > m) m = x;
    }
    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double l = 0.0;
    for (int t = t0; t < t1; ++t) {
        int64_t block = table_row[t / bs];
        int off = t % bs;
        double x = 0.0;
        for (int i = 0; i < d; ++i)
            x += elem(qrow, i, dtype) * elem(k_cache, cache_index(block, g, off, i, Hkv, bs, d), dtype);
        x *= scale;
        double w = exp(x - m);
        l += w;
        for (int i = 0; i < d; ++i)
            acc[i] += w * elem(v_cache, cache_index(block, g, off, i, Hkv, bs, d), dtype);
    }
    *m_out = m;
    *l_out = l;
}

/*
 * Decode: out[s][h][:] = softmax_t(scale * q[s][h] . K_t) V_t over t < ctx_s,
 * K_t, V_t gathered through block_tables[s][t / bs] at offset t % bs, KV head
 * h / (Hq / Hkv).  out is double [S][Hq][d].  Returns 0, or -1 on bad shapes.
 */
int oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_tables, int max_blocks, const int32_t *context_lens, int S,
                  int Hq, int Hkv, int d, int bs, double scale, int dtype, double *out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    double m, l;
    for (int s = 0; s < S; ++s) {
        int ctx = context_lens[s];
        const int32_t *row = block_tables + (int64_t)s * max_blocks;
        for (int h = 0; h < Hq; ++h) {
            double *o = out + ((int64_t)s * Hq + h) * d;
            const uint16_t *qrow = q + ((int64_t)s * Hq + h) * d;
            attend_range(qrow, dtype, k_cache, v_cache, row, 0, ctx, h / G, Hkv, bs, d, scale, &m,
                         &l, o);
            for (int i = 0; i < d; ++i) o[i] = (ctx > 0) ? o[i] / l : 0.0;
        }
    }
    return 0;
}

/*
 * Partial attention over logical token range [t0, t1) of sequence s, all
 * query heads: m_out, l_out [Hq], acc_out [Hq][d] (unnormalised).
 */
int oracle_decode_range(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_row, int t0, int t1, int Hq, int Hkv, int d, int bs,
                        double scale, int dtype, double *m_out, double *l_out, double *acc_out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h)
        attend_range(q + (int64_t)h * d, dtype, k_cache, v_cache, block_row, t0, t1, h / G, Hkv, bs,
                     d, scale, m_out + h, l_out + h, acc_out + (int64_t)h * d);
    return 0;
}

/*
 * Log-sum-exp merge of n partials for one row: M = max m_j,
 * L = sum exp(m_j - M) l_j, out = sum exp(m_j - M) acc_j / L.
 * Partials with m = -inf (empty ranges) contribute nothing.
 */
void oracle_merge(int n, const double *m, const double *l, const double *acc, int d, double *out) {
    double M = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (m[j] > M) M = m[j];
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (M == -INFINITY) return;
    double L = 0.0;
    for (int j = 0; j < n; ++j) {
        if (m[j] == -INFINITY) continue;
        double w = exp(m[j] - M);
        L += w * l[j];
        for (int i = 0; i < d; ++i) out[i] += w * acc[(int64_t)j * d + i];
    }
    for (int i = 0; i < d; ++i) out[i] /= L;
}

/*
 * Prefill: for chunk c, query rows cu_seqlens[c] .. cu_seqlens[c+1]-1 (q_len
 * of them); row i sits at position p = ctx_c - q_len + i and attends logical
 * keys 0 .. p inclusive.  out is double [total_q][Hq][d].
 * Returns 0, or -1 if some chunk has q_len > ctx or bad shapes.
 */
int oracle_prefill(const uint16_t *q, const int32_t *cu_seqlens, int S, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *block_tables, int max_blocks,
                   const int32_t *context_lens, int Hq, int Hkv, int d, int bs, double scale,
                   int dtype, double *out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    double m, l;
    for (int c = 0; c < S; ++c) {
        int q0 = cu_seqlens[c], q_len = cu_seqlens[c + 1] - cu_seqlens[c];
        int ctx = context_lens[c];
        if (q_len < 0 || q_len > ctx) return -1;
        const int32_t *row = block_tables + (int64_t)c * max_blocks;
        for (int i = 0; i < q_len; ++i) {
            int p = ctx - q_len + i;
            for (int h = 0; h < Hq; ++h) {
                int64_t r = ((int64_t)(q0 + i) * Hq + h) * d;
                attend_range(q + r, dtype, k_cache, v_cache, row, 0, p + 1, h / G, Hkv, bs, d,
                             scale, &m, &l, out + r);
                for (int j = 0; j < d; ++j) out[r + j] /= l;
            }
        }
    }
    return 0;
}

/*
 * Dense attention for one sequence on contiguous K/V [ctx][Hkv][d] and query
 * [Hq][d]: out[h][:] = softmax_t(scale q[h] . K[t][h/G]) V[t][h/G].
 */
int oracle_dense(const uint16_t *q, const uint16_t *k, const uint16_t *v, int ctx, int Hq, int Hkv,
                 int d, double scale, int dtype, double *out) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        double *o = out + (int64_t)h * d;
        double m = -INFINITY;
        for (int t = 0; t < ctx; ++t) {
            double x = 0.0;
            for (int i = 0; i < d; ++i)
                x += elem(q, (int64_t)h * d + i, dtype) * elem(k, ((int64_t)t * Hkv + g) * d + i, dtype);
            x *= scale;
            if (x > m) m = x;
        }
        double l = 0.0;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int t = 0; t < ctx; ++t) {
            double x = 0.0;
            for (int i = 0; i < d; ++i)
                x += elem(q, (int64_t)h * d + i, dtype) * elem(k, ((int64_t)t * Hkv + g) * d + i, dtype);
            double w = exp(x * scale - m);
            l += w;
            for (int i = 0; i < d; ++i) o[i] += w * elem(v, ((int64_t)t * Hkv + g) * d + i, dtype);
        }
        for (int i = 0; i < d; ++i) o[i] = ctx > 0 ? o[i] / l : 0.0;
    }
    return 0;
}
