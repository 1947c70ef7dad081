/*
 * pa_oracle.c -- plain, slow fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no code, header, helper or constant with the
 * CUDA path.
 *
 * Sources (web pages on LLM inference; cited by short tag below):
 *   [QA]    "LLM推理与服务：面试问题与推荐回答" (LLM inference & serving interview Q&A)
 *   [SB11]  "Scaling Book 入门第 11 章：推理优化 — KV Cache / Continuous Batching / 量化"
 *   [H100]  "09-inference-optimization.md" (LLM-Code-Hot-100, "⚡ 推理优化")
 *   [ANIM]  "推理机制动态图解（进阶）：并行、投机解码、PD、FlashAttention、调度"
 *   [PANO]  "LLM 推理优化全景实战：从 PagedAttention 到投机解码"
 *
 * What is computed, in the plainest form the pages support:
 *   - slot mapping: logical block = pos / block_size, offset = pos % block_size,
 *     slot = table[logical] * block_size + offset            ([PANO] §2.3, write_kv)
 *   - append: copy the new key/value rows to their slots      ([PANO] §2.3 write_kv;
 *     [H100] "PagedAttention", PagedKVCache.append_token)
 *   - attention: gather the sequence's blocks into a logically contiguous K, V,
 *     keep only the used slots (t < context length, as used_slots does in
 *     [H100] PagedKVCache.get_kv -- the [PANO] §2.4 paged_attention listing forgets
 *     this mask), then softmax(scale * q K^T) V                ([PANO] §2.4;
 *     [H100] "KV Cache", AttentionWithKVCache.forward for the 1/sqrt(d) scale and
 *     the causal offset triu(diagonal = Lk - Lq + 1) when several queries are new)
 *   - GQA: query heads are split into contiguous groups, one KV head per group
 *     ([QA] Q7; [ANIM] §1 figure: q heads 0-15 <-> KV heads 0-3)
 *   - split-KV partials and their combine: per partition the softmax statistics
 *     (max m, sum l of exp(s - m), unnormalised accumulator), merged with the
 *     exp(m_old - m_new) rescale of online softmax ([ANIM] §5; [SB11] §11.8
 *     FlashDecoding).  This is a derived identity, not a printed formula.
 *
 * Everything is IEEE double.  Build with -ffp-contract=off so that every machine
 * evaluates the same sequence of double operations.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_FP16 0
#define ORC_BF16 1

/* ---- 16-bit float decoding, from the IEEE 754 binary16 and bfloat16 formats ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double orc_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);             /* subnormal: f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);  /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 0xf && f == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);               /* subnormal: f * 2^(1-7-3) */
    else
        v = ldexp((double)(8 + f), e - 10);     /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* float -> e4m3, rounding to the nearest representable value, ties to the even
 * code (fraction LSB 0), magnitudes beyond 448 saturating to 448, NaN -> 0x7F.
 * Written as a search over the 127 finite non-negative codes. */
uint8_t orc_e4m3_from_float(float x)
{
    if (x != x)
        return 0x7F;
    uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_err = a;                       /* code 0 is +0 */
    for (int c = 1; c <= 0x7E; c++) {
        double err = fabs(a - orc_e4m3_to_double((uint8_t)c));
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

void orc_encode_e4m3(uint8_t *out, const float *x, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_from_float(x[i]);
}

/* Every 16-bit and 8-bit pattern decoded once, by the functions above, when the
 * library is loaded.  Decoding is exact, so looking a value up gives the same
 * double as calling the decoder; it only spares the attention loops a call to
 * ldexp per element. */
static double fp16_value[65536], bf16_value[65536], e4m3_value[256];

__attribute__((constructor)) static void fill_decode_tables(void)
{
    for (int b = 0; b < 65536; b++) {
        fp16_value[b] = orc_fp16_to_double((uint16_t)b);
        bf16_value[b] = orc_bf16_to_double((uint16_t)b);
    }
    for (int b = 0; b < 256; b++)
        e4m3_value[b] = orc_e4m3_to_double((uint8_t)b);
}

static double elt(const uint16_t *base, size_t idx, int dtype)
{
    return dtype == ORC_BF16 ? bf16_value[base[idx]] : fp16_value[base[idx]];
}

void orc_decode_bits(double *out, const uint16_t *bits, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = elt(bits, (size_t)i, dtype);
}

void orc_decode_e4m3(double *out, const uint8_t *bits, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = e4m3_value[bits[i]];
}

/* ---- slot mapping ([PANO] §2.3 write_kv) ----
 * For sequence i the new tokens are its last q_len positions
 * pos = context_lens[i] - q_len + u, u = 0..q_len-1 (context lengths already count
 * them: the cache is updated before attention, as KVCache.update precedes the
 * score computation in [H100] AttentionWithKVCache.forward).
 * Output slot_mapping[i*q_len + u]; -1 where pos < 0.  Returns 0, or -1 if a
 * position needs a block-table entry beyond max_blocks_per_seq.              */
int orc_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                     const int32_t *context_lens, int num_seqs,
                     int max_blocks_per_seq, int block_size, int q_len)
{
    for (int i = 0; i < num_seqs; i++) {
        for (int u = 0; u < q_len; u++) {
            int64_t pos = (int64_t)context_lens[i] - q_len + u;
            int64_t out;
            if (pos < 0) {
                out = -1;
            } else {
                int64_t logical_block = pos / block_size;
                int64_t block_offset = pos % block_size;
                if (logical_block >= max_blocks_per_seq)
                    return -1;
                int64_t physical_block = block_tables[(int64_t)i * max_blocks_per_seq + logical_block];
                out = physical_block * block_size + block_offset;
            }
            slot_mapping[(int64_t)i * q_len + u] = out;
        }
    }
    return 0;
}

/* ---- append ([PANO] §2.3 write_kv; [H100] PagedKVCache.append_token) ----
 * Cache layout [num_blocks][num_kv_heads][block_size][head_dim]: one page holds,
 * per head, block_size consecutive token rows (the [H100] page shape
 * [layers, heads, page_size, head_dim] for a single layer).
 * New rows k_new, v_new: [n_tokens][num_kv_heads][head_dim].  Elements are copied
 * as raw 16-bit patterns; slots < 0 are skipped.                              */
void orc_append_kv(uint16_t *k_cache, uint16_t *v_cache,
                   const uint16_t *k_new, const uint16_t *v_new,
                   const int64_t *slot_mapping, int n_tokens,
                   int num_kv_heads, int head_dim, int block_size)
{
    for (int t = 0; t < n_tokens; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            for (int d = 0; d < head_dim; d++) {
                int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_dim + d;
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
        }
    }
}

/* ---- append into an FP8 (e4m3) cache with one scale per KV head ----
 * Each new element x (fp16/bf16, exact in float) is stored as e4m3(x / scale[h]):
 * the division in float, then nearest-even rounding with saturation.  The stored
 * value stands for e4m3 * scale.                                               */
void orc_append_kv_fp8(uint8_t *k_cache, uint8_t *v_cache,
                       const uint16_t *k_new, const uint16_t *v_new,
                       const int64_t *slot_mapping, int n_tokens, int num_kv_heads,
                       int head_dim, int block_size, int new_dtype,
                       const float *k_scale, const float *v_scale)
{
    for (int t = 0; t < n_tokens; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            for (int d = 0; d < head_dim; d++) {
                int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_dim + d;
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
                float kx = (float)elt(k_new, (size_t)src, new_dtype);
                float vx = (float)elt(v_new, (size_t)src, new_dtype);
                k_cache[dst] = orc_e4m3_from_float(kx / k_scale[h]);
                v_cache[dst] = orc_e4m3_from_float(vx / v_scale[h]);
            }
        }
    }
}

/* ---- copy-on-write block copy ([QA] Q2: sequences share physical pages up to the
 * point where they diverge; a writer first gives itself a private copy) ----
 * For each pair i, every head's block_size rows of block src[i] are copied to block
 * dst[i], in both caches.  Pairs with an id outside [0, num_blocks) are skipped
 * (returns the number skipped).                                                 */
int orc_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *src, const int32_t *dst,
                    int n_pairs, int num_kv_heads, int head_dim, int block_size, int num_blocks)
{
    int skipped = 0;
    const int64_t block_elems = (int64_t)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < n_pairs; i++) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
            skipped++;
            continue;
        }
        for (int64_t e = 0; e < block_elems; e++) {
            k_cache[(int64_t)dst[i] * block_elems + e] = k_cache[(int64_t)src[i] * block_elems + e];
            v_cache[(int64_t)dst[i] * block_elems + e] = v_cache[(int64_t)src[i] * block_elems + e];
        }
    }
    return skipped;
}

/* Shared description of one attention call. */
typedef struct {
    const uint16_t *q;            /* [num_seqs][q_len][num_q_heads][head_dim] */
    const void *k_cache;          /* [num_blocks][num_kv_heads][block_size][head_dim] */
    const void *v_cache;          /* 16-bit patterns, or e4m3 bytes when kv_fp8 */
    const int32_t *block_tables;  /* [num_seqs][max_blocks_per_seq] */
    const int32_t *context_lens;  /* [num_seqs] */
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    int max_blocks_per_seq, q_len, dtype;
    double scale;
    int kv_fp8;                   /* cache holds e4m3 codes */
    const float *k_scale;         /* per KV head, kv_fp8 only: value = e4m3 * scale */
    const float *v_scale;
} orc_call;

/* Element idx of a cache, in the units of q (dequantised for an FP8 cache). */
static double cache_at(const orc_call *c, const void *cache, const float *scales, size_t idx,
                       int kvh)
{
    if (c->kv_fp8)
        return e4m3_value[((const uint8_t *)cache)[idx]] * (double)scales[kvh];
    return elt((const uint16_t *)cache, idx, c->dtype);
}

/* Address of token t (logical position) of sequence i, KV head h, in a cache. */
static size_t token_row(const orc_call *c, int i, int h, int64_t t)
{
    int64_t logical_block = t / c->block_size;
    int64_t block_offset = t % c->block_size;
    int64_t physical_block = c->block_tables[(int64_t)i * c->max_blocks_per_seq + logical_block];
    return (size_t)(((physical_block * c->num_kv_heads + h) * c->block_size + block_offset) * c->head_dim);
}

/* Output row r = (i*q_len + u)*num_q_heads + h.  Query u of sequence i sees the
 * first T = L_i - q_len + u + 1 tokens: the [H100] causal mask
 * triu(ones(Lq, Lk), diagonal = Lk - Lq + 1) hides key j from query u exactly when
 * j >= Lk - Lq + u + 1.  With q_len = 1, T = L_i.                             */
static void row_coords(const orc_call *c, int64_t r, int *i, int *u, int *h, int *kvh, int64_t *T)
{
    *h = (int)(r % c->num_q_heads);
    int64_t iu = r / c->num_q_heads;
    *u = (int)(iu % c->q_len);
    *i = (int)(iu / c->q_len);
    int group = c->num_q_heads / c->num_kv_heads;   /* query heads per KV head */
    *kvh = *h / group;
    *T = (int64_t)c->context_lens[*i] - c->q_len + *u + 1;
}

/* scale * <q_row, k_token> in double. */
static double score(const orc_call *c, int64_t r, size_t krow, int kvh)
{
    const size_t qoff = (size_t)r * c->head_dim;
    double dot = 0.0;
    for (int d = 0; d < c->head_dim; d++)
        dot += elt(c->q, qoff + d, c->dtype) * cache_at(c, c->k_cache, c->k_scale, krow + d, kvh);
    return c->scale * dot;
}

/* ---- attention for a list of output rows ([PANO] §2.4 with the used-slot mask) ----
 * out: [n_rows][head_dim].  rows: output row indices (NULL = all rows in order).
 * A row that sees no token (T <= 0, e.g. context length 0) is all zeros.
 * Returns 0, or -1 on allocation failure.                                       */
static int decode_rows(const orc_call *c, double *out, const int64_t *rows, int64_t n_rows)
{
    int64_t max_len = 0;
    for (int i = 0; i < c->num_seqs; i++)
        if (c->context_lens[i] > max_len)
            max_len = c->context_lens[i];
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!s)
        return -1;
    for (int64_t n = 0; n < n_rows; n++) {
        int64_t r = rows ? rows[n] : n;
        int i, u, h, kvh;
        int64_t T;
        row_coords(c, r, &i, &u, &h, &kvh, &T);
        double *o = out + n * c->head_dim;
        for (int d = 0; d < c->head_dim; d++)
            o[d] = 0.0;
        if (T <= 0)
            continue;
        /* scores over the gathered, logically contiguous keys */
        for (int64_t t = 0; t < T; t++)
            s[t] = score(c, r, token_row(c, i, kvh, t), kvh);
        /* softmax: exp(s - max) / sum */
        double mx = s[0];
        for (int64_t t = 1; t < T; t++)
            if (s[t] > mx)
                mx = s[t];
        double den = 0.0;
        for (int64_t t = 0; t < T; t++) {
            s[t] = exp(s[t] - mx);
            den += s[t];
        }
        /* out = sum_t softmax_t * V[t] */
        for (int64_t t = 0; t < T; t++) {
            double p = s[t] / den;
            size_t vrow = token_row(c, i, kvh, t);
            for (int d = 0; d < c->head_dim; d++)
                o[d] += p * cache_at(c, c->v_cache, c->v_scale, vrow + d, kvh);
        }
    }
    free(s);
    return 0;
}

int orc_decode(double *out, const int64_t *rows, int64_t n_rows,
               const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
               const int32_t *block_tables, const int32_t *context_lens,
               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
               int block_size, float scale, int max_blocks_per_seq, int q_len, int dtype)
{
    orc_call c = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, block_size, max_blocks_per_seq, q_len, dtype,
                  (double)scale, 0, NULL, NULL};
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 || q_len <= 0)
        return -2;
    if (rows == NULL)
        n_rows = (int64_t)num_seqs * q_len * num_q_heads;
    return decode_rows(&c, out, rows, n_rows);
}

/* Attention over an FP8 (e4m3) cache: K = e4m3 * k_scale[kvh], V = e4m3 * v_scale[kvh];
 * q and the arithmetic as in orc_decode. */
int orc_decode_fp8(double *out, const int64_t *rows, int64_t n_rows,
                   const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                   const float *k_scale, const float *v_scale,
                   const int32_t *block_tables, const int32_t *context_lens,
                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                   int block_size, float scale, int max_blocks_per_seq, int q_len, int dtype)
{
    orc_call c = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, block_size, max_blocks_per_seq, q_len, dtype,
                  (double)scale, 1, k_scale, v_scale};
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 || q_len <= 0)
        return -2;
    if (rows == NULL)
        n_rows = (int64_t)num_seqs * q_len * num_q_heads;
    return decode_rows(&c, out, rows, n_rows);
}

/* ---- split-KV partition statistics ([SB11] §11.8 FlashDecoding; [ANIM] §5) ----
 * Sequence i's ceil(L_i / block_size) blocks are cut into num_splits partitions of
 * C = ceil(ceil(L_i/block_size) / num_splits) blocks; partition p holds tokens
 * [p*C*block_size, (p+1)*C*block_size), intersected with what the row may see.
 * For each (row, p): m = max score (-inf if empty), l = sum exp(s - m) (0 if empty),
 * acc = sum exp(s - m) * V[t] (0 if empty).  Natural-log domain.
 * m_out, l_out: [num_seqs][num_splits][q_len*num_q_heads];
 * acc_out: [num_seqs][num_splits][q_len*num_q_heads][head_dim].              */
int orc_decode_partitions(double *m_out, double *l_out, double *acc_out,
                          const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, float scale, int max_blocks_per_seq, int q_len,
                          int dtype, int num_splits)
{
    orc_call c = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                  num_kv_heads, head_dim, block_size, max_blocks_per_seq, q_len, dtype,
                  (double)scale, 0, NULL, NULL};
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || num_splits <= 0 || q_len <= 0)
        return -2;
    const int64_t rows_per_seq = (int64_t)q_len * num_q_heads;
    for (int64_t r = 0; r < (int64_t)num_seqs * rows_per_seq; r++) {
        int i, u, h, kvh;
        int64_t T;
        row_coords(&c, r, &i, &u, &h, &kvh, &T);
        int64_t L = context_lens[i];
        int64_t nb = (L + block_size - 1) / block_size;
        int64_t C = (nb + num_splits - 1) / num_splits;        /* blocks per partition */
        for (int p = 0; p < num_splits; p++) {
            int64_t w = ((int64_t)i * num_splits + p) * rows_per_seq + (r % rows_per_seq);
            double *acc = acc_out + w * head_dim;
            int64_t t0 = (int64_t)p * C * block_size;
            int64_t t1 = t0 + C * block_size;
            if (t1 > T)
                t1 = T;
            double m = -INFINITY, l = 0.0;
            for (int d = 0; d < head_dim; d++)
                acc[d] = 0.0;
            for (int64_t t = t0; t < t1; t++) {
                double s = score(&c, r, token_row(&c, i, kvh, t), kvh);
                if (s > m)
                    m = s;
            }
            for (int64_t t = t0; t < t1; t++) {
                size_t row = token_row(&c, i, kvh, t);
                double e = exp(score(&c, r, row, kvh) - m);
                l += e;
                for (int d = 0; d < head_dim; d++)
                    acc[d] += e * elt(v_cache, row + d, dtype);
            }
            m_out[w] = m;
            l_out[w] = l;
        }
    }
    return 0;
}

/* ---- combine of partition statistics (derived from the [ANIM] §5 rescale) ----
 * M = max over non-empty partitions of m_p; out = sum_p e^(m_p - M) acc_p /
 * sum_p e^(m_p - M) l_p.  A row with no non-empty partition is all zeros.
 * Same layouts as orc_decode_partitions; out: [num_seqs][rows_per_seq][head_dim]. */
void orc_combine(double *out, const double *m, const double *l, const double *acc,
                 int num_seqs, int num_splits, int64_t rows_per_seq, int head_dim)
{
    for (int i = 0; i < num_seqs; i++) {
        for (int64_t r = 0; r < rows_per_seq; r++) {
            double *o = out + ((int64_t)i * rows_per_seq + r) * head_dim;
            double M = -INFINITY;
            for (int p = 0; p < num_splits; p++) {
                int64_t w = ((int64_t)i * num_splits + p) * rows_per_seq + r;
                if (l[w] > 0.0 && m[w] > M)
                    M = m[w];
            }
            for (int d = 0; d < head_dim; d++)
                o[d] = 0.0;
            if (M == -INFINITY)
                continue;
            double den = 0.0;
            for (int p = 0; p < num_splits; p++) {
                int64_t w = ((int64_t)i * num_splits + p) * rows_per_seq + r;
                if (l[w] > 0.0)
                    den += exp(m[w] - M) * l[w];
            }
            for (int p = 0; p < num_splits; p++) {
                int64_t w = ((int64_t)i * num_splits + p) * rows_per_seq + r;
                if (!(l[w] > 0.0))
                    continue;
                double wt = exp(m[w] - M);
                for (int d = 0; d < head_dim; d++)
                    o[d] += wt * acc[w * head_dim + d];
            }
            for (int d = 0; d < head_dim; d++)
                o[d] /= den;
        }
    }
}
