/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for paged FP8/BF16
 * KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no source, header, table or helper with the CUDA
 * library; it is written from the method's definition, not from the kernels.
 *
 * Sources (web pages; cited by title and paragraph):
 *  [Q]  "Cloudflare quantizes Kimi and GLM caches for 41% faster inference",
 *       2nd paragraph (KV cache quantization): the cache is held as FP8 e4m3
 *       instead of BF16; decode reads the FP8 cache.
 *  [T]  same page, 4th paragraph (KV cache integrity check): every physical
 *       page carries a tag that changes on reallocation; the server knows the
 *       (page, tag) pairs each request expects; those are checked before decode
 *       reads the cache, and a request with any mismatch is aborted.
 *  [P]  "Workers AI targets the inference bottleneck", section "KV cache
 *       compression goes open source": a block table of integer indices maps a
 *       sequence's logical blocks to physical blocks, so that each attention
 *       head can keep a different number of tokens.
 *  [I]  "How we built the most efficient inference engine for Cloudflare's
 *       network", section "Batching to feed the Tensor Cores": the KV cache is
 *       split into pages allocated on demand.
 *  [M]  "Workers AI targets the inference bottleneck", section "KV cache
 *       compression goes open source", 3rd paragraph: eviction tracks the
 *       attention each KV entry has received over past steps and evicts the
 *       entries with the lowest total, like a least-frequently-used cache.
 *  [S]  "Workers AI targets the inference bottleneck", section "Speculative
 *       decoding: predicting more than one token", 1st paragraph: the model
 *       verifies all candidate tokens in a single forward pass.
 *  [E]  The OCP 8-bit floating point specification (E4M3 "FN" variant), the
 *       format that [Q] names: 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 *       no infinities, S.1111.111 is NaN, largest finite 448.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  R1 scale granularity: one fp32 scale per (physical page, kv head) unit,
 *     separately for K and V; scale = absmax / 448 in fp32 with IEEE
 *     round-to-nearest division; absmax == 0 gives scale 1.
 *  R2 quantised byte = e4m3_rne_satfinite( fl32(x / scale) ): the division is
 *     rounded to fp32 first; values beyond +-448 saturate to +-448.
 *  R3 append: the call that writes slot 0 of a unit sets that unit's scale
 *     from the tokens this call writes into the unit; later appends reuse the
 *     stored scale (and saturate).
 *  R4 GQA grouping is consecutive: query head hq reads kv head hq / G.
 *  R5 flagged requests and zero-length heads produce all-zero output.
 *  R6 only live table entries p < ceil(len/16) are read or checked.
 *  R7 attention mass [M]: the mass of token j of kv head h at one decode step
 *     is the sum, over the G query heads that read kv head h, of the softmax
 *     weight of token j (weights normalised over the head's n tokens); a call
 *     adds it to a running total kept by the caller.  Flagged requests and
 *     zero-length heads add nothing.
 *  R8 multi-query verify [S]: a request's kq candidate tokens are the last kq
 *     tokens of each of its heads (already written); query token i (0-based)
 *     attends to the first n - kq + 1 + i tokens of the head (causal among the
 *     candidates).  A query that would see no token gives zero output.
 *
 * Precision: attention is computed in fp64 (plain two-pass softmax, natural
 * exp, sequential token order); quantisation decisions are taken in fp32, the
 * precision the kernels use, so that FP8 bytes can be compared bit for bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_PAGE 16

/* request flag bits */
#define ORC_FLAG_TAG 1u     /* tag mismatch [T]                         */
#define ORC_FLAG_PAGE 2u    /* physical page id outside [0, num_pages)  */
#define ORC_FLAG_LEN 4u     /* length / position outside the table      */

/* ------------------------------------------------------------------------ */
/* e4m3 codec [E]                                                            */
/* ------------------------------------------------------------------------ */

/* Value of an e4m3 code, from the format's closed form (exact in double).
 * Normal (e > 0):    (-1)^s * 2^(e-7) * (1 + m/8)
 * Subnormal (e = 0): (-1)^s * 2^(-6)  * (m/8)
 * 0x7F / 0xFF:       NaN                                                    */
double oracle_e4m3_to_double(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* The 127 non-negative finite magnitudes, ascending: code c -> value(c). */
static double g_mag[127];
static int g_mag_ready = 0;

static void build_mag_table(void)
{
    if (g_mag_ready)
        return;
    for (int c = 0; c < 127; ++c)
        g_mag[c] = oracle_e4m3_to_double((uint8_t)c);
    g_mag_ready = 1;
}

/* fp32 -> e4m3, round to nearest, ties to the even code, saturating to
 * +-448 (R2), NaN -> 0x7F, sign kept (so -0 -> 0x80).  Found by searching the
 * ascending magnitude table for the two neighbours of |x| and comparing |x|
 * with their midpoint; every quantity compared is exact in double.          */
uint8_t oracle_e4m3_from_float(float x)
{
    build_mag_table();
    if (isnan(x))
        return 0x7F;
    uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= g_mag[126])
        return s | 126;
    /* largest c with g_mag[c] <= a */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_mag[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    int c = lo;
    if (g_mag[c] == a)
        return s | (uint8_t)c;
    double twice = 2.0 * a;
    double sum = g_mag[c] + g_mag[c + 1];
    int pick;
    if (twice < sum)
        pick = c;
    else if (twice > sum)
        pick = c + 1;
    else
        pick = (c % 2 == 0) ? c : c + 1;
    return s | (uint8_t)pick;
}

void oracle_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    build_mag_table();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_from_float(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_to_double(codes[i]);
}

/* bf16 bit pattern -> value (bf16 is the upper half of an fp32). */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* R1: scale of a unit from the absolute maximum of the values it is set from. */
float oracle_unit_scale(float absmax)
{
    if (absmax == 0.0f)
        return 1.0f;
    volatile float num = absmax; /* keep this one fp32 division as written */
    return num / 448.0f;
}

/* R2 */
uint8_t oracle_quantize(float x, float scale)
{
    volatile float q = x / scale; /* fp32 IEEE division, rounded once */
    return oracle_e4m3_from_float(q);
}

/* ------------------------------------------------------------------------ */
/* Paged cache description (host copies of the caller's arrays)              */
/* ------------------------------------------------------------------------ */
/* Pool layout: k_pages / v_pages [num_pages][num_kv_heads][16][head_dim] of
 * either e4m3 bytes (dtype 1) or bf16 bit patterns (dtype 0); scales and tags
 * [num_pages][num_kv_heads].  A table entry phys for kv head h always names
 * the unit (phys, h) [P].                                                   */
typedef struct {
    int32_t num_pages, num_kv_heads, head_dim, dtype;
    void *k_pages, *v_pages;
    float *k_scale, *v_scale;
    const uint32_t *page_tags; /* NULL: no integrity tracking [T] */
} orc_cache;

typedef struct {
    int32_t batch, max_pages;
    const int32_t *block_tables;
    int64_t bt_stride_b, bt_stride_h;
    const int32_t *seq_lens;
    int64_t len_stride_b, len_stride_h;
    const uint32_t *expected_tags; /* same indexing as block_tables */
} orc_pages;

static int64_t unit_index(const orc_cache *c, int32_t phys, int h)
{
    return (int64_t)phys * c->num_kv_heads + h;
}

/* ------------------------------------------------------------------------ */
/* kv_append [Q] + R1..R3                                                    */
/* ------------------------------------------------------------------------ */
/* For each (b, h): tokens t < n (n = new_lens[b,h] or T) of k_new/v_new
 * [B][Hkv][T][D] (bf16 bits) go to logical positions positions[b,h] + t.
 * Position pos lands in unit (block_tables[b,h,pos/16], h), slot pos%16.
 * A destination that fails a check is not written and sets a flag bit:
 *   pos/16 >= max_pages -> LEN, page id outside the pool -> PAGE,
 *   tags present and pool tag != expected tag -> TAG.
 * flags (may be NULL) are OR-ed, never cleared.                             */
void oracle_kv_append(orc_cache *c, const orc_pages *pg, const int32_t *positions,
                      int32_t T, const int32_t *new_lens, const uint16_t *k_new,
                      const uint16_t *v_new, uint8_t *flags)
{
    const int H = c->num_kv_heads, D = c->head_dim;
    for (int b = 0; b < pg->batch; ++b) {
        for (int h = 0; h < H; ++h) {
            int64_t li = (int64_t)b * pg->len_stride_b + (int64_t)h * pg->len_stride_h;
            int32_t p0 = positions[li];
            int32_t n = new_lens ? new_lens[li] : T;
            if (n > T)
                n = T;
            if (n <= 0)
                continue;
            if (p0 < 0) {
                if (flags)
                    flags[b] |= ORC_FLAG_LEN;
                continue;
            }
            const uint16_t *kb = k_new + ((int64_t)b * H + h) * T * D;
            const uint16_t *vb = v_new + ((int64_t)b * H + h) * T * D;
            int t = 0;
            while (t < n) {
                int32_t pos = p0 + t;
                int32_t lp = pos / ORC_PAGE;
                int32_t slot = pos % ORC_PAGE;
                /* tokens of this call that fall into logical page lp */
                int cnt = ORC_PAGE - slot;
                if (cnt > n - t)
                    cnt = n - t;
                if (lp >= pg->max_pages) {
                    if (flags)
                        flags[b] |= ORC_FLAG_LEN;
                    break;
                }
                int64_t bi = (int64_t)b * pg->bt_stride_b + (int64_t)h * pg->bt_stride_h + lp;
                int32_t phys = pg->block_tables[bi];
                if (phys < 0 || phys >= c->num_pages) {
                    if (flags)
                        flags[b] |= ORC_FLAG_PAGE;
                    t += cnt;
                    continue;
                }
                int64_t u = unit_index(c, phys, h);
                if (c->page_tags && pg->expected_tags &&
                    c->page_tags[u] != pg->expected_tags[bi]) {
                    if (flags)
                        flags[b] |= ORC_FLAG_TAG;
                    t += cnt;
                    continue;
                }
                if (c->dtype == 0) {
                    uint16_t *kp = (uint16_t *)c->k_pages;
                    uint16_t *vp = (uint16_t *)c->v_pages;
                    for (int j = 0; j < cnt; ++j)
                        for (int d = 0; d < D; ++d) {
                            kp[(u * ORC_PAGE + slot + j) * D + d] = kb[(int64_t)(t + j) * D + d];
                            vp[(u * ORC_PAGE + slot + j) * D + d] = vb[(int64_t)(t + j) * D + d];
                        }
                } else {
                    uint8_t *kp = (uint8_t *)c->k_pages;
                    uint8_t *vp = (uint8_t *)c->v_pages;
                    if (slot == 0) { /* R3: this call opens the unit */
                        float ka = 0.0f, va = 0.0f;
                        for (int j = 0; j < cnt; ++j)
                            for (int d = 0; d < D; ++d) {
                                float kx = fabsf(bf16_bits_to_float(kb[(int64_t)(t + j) * D + d]));
                                float vx = fabsf(bf16_bits_to_float(vb[(int64_t)(t + j) * D + d]));
                                if (kx > ka)
                                    ka = kx;
                                if (vx > va)
                                    va = vx;
                            }
                        c->k_scale[u] = oracle_unit_scale(ka);
                        c->v_scale[u] = oracle_unit_scale(va);
                    }
                    float ks = c->k_scale[u], vs = c->v_scale[u];
                    for (int j = 0; j < cnt; ++j)
                        for (int d = 0; d < D; ++d) {
                            float kx = bf16_bits_to_float(kb[(int64_t)(t + j) * D + d]);
                            float vx = bf16_bits_to_float(vb[(int64_t)(t + j) * D + d]);
                            kp[(u * ORC_PAGE + slot + j) * D + d] = oracle_quantize(kx, ks);
                            vp[(u * ORC_PAGE + slot + j) * D + d] = oracle_quantize(vx, vs);
                        }
                }
                t += cnt;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Integrity and bounds check before decode reads [T], R6                    */
/* ------------------------------------------------------------------------ */
/* flags[b] = OR over kv heads h of:
 *   LEN  if len < 0, len > 16*max_pages or len > max_seq_len (head skipped);
 *   else for each live entry p < ceil(len/16):
 *     PAGE if the page id is outside [0, num_pages),
 *     TAG  if tags are tracked and pool tag != expected tag.               */
void oracle_validate(const orc_cache *c, const orc_pages *pg, int32_t max_seq_len,
                     uint8_t *flags)
{
    const int H = c->num_kv_heads;
    for (int b = 0; b < pg->batch; ++b) {
        uint8_t f = 0;
        for (int h = 0; h < H; ++h) {
            int32_t n = pg->seq_lens[(int64_t)b * pg->len_stride_b + (int64_t)h * pg->len_stride_h];
            if (n < 0 || (int64_t)n > (int64_t)ORC_PAGE * pg->max_pages || n > max_seq_len) {
                f |= ORC_FLAG_LEN;
                continue;
            }
            int32_t np = (n + ORC_PAGE - 1) / ORC_PAGE;
            for (int p = 0; p < np; ++p) {
                int64_t bi = (int64_t)b * pg->bt_stride_b + (int64_t)h * pg->bt_stride_h + p;
                int32_t phys = pg->block_tables[bi];
                if (phys < 0 || phys >= c->num_pages) {
                    f |= ORC_FLAG_PAGE;
                    continue;
                }
                if (c->page_tags && pg->expected_tags &&
                    c->page_tags[unit_index(c, phys, h)] != pg->expected_tags[bi])
                    f |= ORC_FLAG_TAG;
            }
        }
        flags[b] = f;
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention [Q][P][I], R4, R5                                        */
/* ------------------------------------------------------------------------ */
/* Value of element d of token slot `slot` in unit u of pool `pages`,
 * dequantised (e4m3 value times the unit scale, or the exact bf16 value).   */
static double kv_value(const orc_cache *c, const void *pages, const float *scale,
                       int64_t u, int slot, int d)
{
    int64_t idx = (u * ORC_PAGE + slot) * c->head_dim + d;
    if (c->dtype == 0)
        return (double)bf16_bits_to_float(((const uint16_t *)pages)[idx]);
    return oracle_e4m3_to_double(((const uint8_t *)pages)[idx]) * (double)scale[u];
}

/* out [B][Hq][D] (fp64), q [B][Hq][D] (bf16 bits).  For each request b and
 * query head hq, with kv head h = hq / G and n = len[b,h]:
 *   zero output if flags[b] != 0 or n == 0;
 *   else s_j = sm_scale * sum_d q_d k_jd,  m = max_j s_j,
 *        out_d = sum_j exp(s_j - m) v_jd / sum_j exp(s_j - m),
 * where token j lives in unit (bt[b,h,j/16], h), slot j%16.
 * flags_out (may be NULL) receives the request flags of oracle_validate.    */
void oracle_paged_decode(const orc_cache *c, const orc_pages *pg, const uint16_t *q,
                         int32_t num_q_heads, double sm_scale, int32_t max_seq_len,
                         double *out, uint8_t *flags_out)
{
    const int H = c->num_kv_heads, D = c->head_dim, Hq = num_q_heads;
    const int G = Hq / H;
    const int B = pg->batch;
    uint8_t *flags = (uint8_t *)malloc(B > 0 ? (size_t)B : 1);
    oracle_validate(c, pg, max_seq_len, flags);
    if (flags_out)
        memcpy(flags_out, flags, (size_t)B);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bq = 0; bq < (int64_t)B * Hq; ++bq) {
        int b = (int)(bq / Hq), hq = (int)(bq % Hq);
        int h = hq / G;
        double *o = out + bq * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        int32_t n = pg->seq_lens[(int64_t)b * pg->len_stride_b + (int64_t)h * pg->len_stride_h];
        if (flags[b] != 0 || n <= 0)
            continue;
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        for (int d = 0; d < D; ++d)
            qv[d] = (double)bf16_bits_to_float(q[bq * D + d]);
        const int32_t *row = pg->block_tables + (int64_t)b * pg->bt_stride_b + (int64_t)h * pg->bt_stride_h;
        /* pass 1: scores and their maximum */
        double m = -INFINITY;
        for (int32_t j = 0; j < n; ++j) {
            int64_t u = unit_index(c, row[j / ORC_PAGE], h);
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += qv[d] * kv_value(c, c->k_pages, c->k_scale, u, j % ORC_PAGE, d);
            s[j] = sm_scale * acc;
            if (s[j] > m)
                m = s[j];
        }
        /* pass 2: normaliser and weighted sum of values */
        double l = 0.0;
        for (int32_t j = 0; j < n; ++j) {
            double p = exp(s[j] - m);
            int64_t u = unit_index(c, row[j / ORC_PAGE], h);
            l += p;
            for (int d = 0; d < D; ++d)
                o[d] += p * kv_value(c, c->v_pages, c->v_scale, u, j % ORC_PAGE, d);
        }
        for (int d = 0; d < D; ++d)
            o[d] /= l;
        free(qv);
        free(s);
    }
    free(flags);
}

/*
 * Attention mass [M], reading R7: for every (b, h) of an unflagged request with
 * n > 0 tokens, and every token j < n,
 *   mass[b*mass_sb + h*mass_sh + j] += sum over g < G of
 *       exp(s_gj) / sum_i exp(s_gi),   s_gj = sm_scale * q[b, h*G + g] . k_j
 * in fp64, each query head's softmax taken on its own (max subtracted first).
 * One (b, h) per iteration, so no two threads add to the same entry.
 */
void oracle_attention_mass(const orc_cache *c, const orc_pages *pg, const uint16_t *q,
                           int32_t num_q_heads, double sm_scale, int32_t max_seq_len,
                           double *mass, int64_t mass_sb, int64_t mass_sh)
{
    const int H = c->num_kv_heads, D = c->head_dim, Hq = num_q_heads;
    const int G = Hq / H;
    const int B = pg->batch;
    uint8_t *flags = (uint8_t *)malloc(B > 0 ? (size_t)B : 1);
    oracle_validate(c, pg, max_seq_len, flags);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H);
        int32_t n = pg->seq_lens[(int64_t)b * pg->len_stride_b + (int64_t)h * pg->len_stride_h];
        if (flags[b] != 0 || n <= 0)
            continue;
        const int32_t *row = pg->block_tables + (int64_t)b * pg->bt_stride_b + (int64_t)h * pg->bt_stride_h;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        double *mrow = mass + (int64_t)b * mass_sb + (int64_t)h * mass_sh;
        for (int g = 0; g < G; ++g) {
            const uint16_t *qg = q + ((int64_t)b * Hq + (int64_t)h * G + g) * D;
            double m = -INFINITY, l = 0.0;
            for (int32_t j = 0; j < n; ++j) {
                int64_t u = unit_index(c, row[j / ORC_PAGE], h);
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += (double)bf16_bits_to_float(qg[d]) *
                           kv_value(c, c->k_pages, c->k_scale, u, j % ORC_PAGE, d);
                s[j] = sm_scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            for (int32_t j = 0; j < n; ++j)
                l += exp(s[j] - m);
            for (int32_t j = 0; j < n; ++j)
                mrow[j] += exp(s[j] - m) / l;
        }
        free(s);
    }
    free(flags);
}

/*
 * Multi-query verify [S], reading R8: q and out are [B][kq][Hq][D]; the
 * output row of (b, i, hq) is the decode attention of q[b][i][hq] over the
 * first n - kq + 1 + i tokens of kv head hq / G, n = seq_lens(b, h).  Flags are
 * those of the request (oracle_validate over its n tokens); flagged requests
 * give zero rows for every query token.
 */
void oracle_paged_decode_multi(const orc_cache *c, const orc_pages *pg, const uint16_t *q,
                               int32_t num_q_heads, int32_t kq, double sm_scale,
                               int32_t max_seq_len, double *out, uint8_t *flags_out)
{
    const int H = c->num_kv_heads, D = c->head_dim, Hq = num_q_heads;
    const int G = Hq / H;
    const int B = pg->batch;
    uint8_t *flags = (uint8_t *)malloc(B > 0 ? (size_t)B : 1);
    oracle_validate(c, pg, max_seq_len, flags);
    if (flags_out)
        memcpy(flags_out, flags, (size_t)B);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = 0; row < (int64_t)B * kq * Hq; ++row) {
        int b = (int)(row / ((int64_t)kq * Hq));
        int i = (int)((row / Hq) % kq), hq = (int)(row % Hq);
        int h = hq / G;
        double *o = out + row * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        int32_t n = pg->seq_lens[(int64_t)b * pg->len_stride_b + (int64_t)h * pg->len_stride_h];
        int64_t seen = (int64_t)n - kq + 1 + i;   /* tokens query i attends to */
        if (flags[b] != 0 || seen <= 0)
            continue;
        const int32_t *trow = pg->block_tables + (int64_t)b * pg->bt_stride_b + (int64_t)h * pg->bt_stride_h;
        double *s = (double *)malloc(sizeof(double) * (size_t)seen);
        double m = -INFINITY, l = 0.0;
        for (int64_t j = 0; j < seen; ++j) {
            int64_t u = unit_index(c, trow[j / ORC_PAGE], h);
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)bf16_bits_to_float(q[row * D + d]) *
                       kv_value(c, c->k_pages, c->k_scale, u, (int)(j % ORC_PAGE), d);
            s[j] = sm_scale * acc;
            if (s[j] > m)
                m = s[j];
        }
        for (int64_t j = 0; j < seen; ++j) {
            double p = exp(s[j] - m);
            int64_t u = unit_index(c, trow[j / ORC_PAGE], h);
            l += p;
            for (int d = 0; d < D; ++d)
                o[d] += p * kv_value(c, c->v_pages, c->v_scale, u, (int)(j % ORC_PAGE), d);
        }
        for (int d = 0; d < D; ++d)
            o[d] /= l;
        free(s);
    }
    free(flags);
}

/* Number of threads an OpenMP region of this library uses (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) { omp_set_num_threads(n); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
