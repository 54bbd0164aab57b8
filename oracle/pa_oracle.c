/*
 * Paged-attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links or calls this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header or table with the CUDA library.
 *
 * What it computes, and where each step is defined:
 *
 *  - Address translation (Week 3 Day 4: Direct Paged Attention, "Why
 *    block_table Matters" and the "logical key position -> logical page ->
 *    physical page id -> slot in page" chain in "How This Maps to tiny-llm"):
 *    logical position j of request b lives in physical page
 *    block_table[b, j / page_size] at slot j % page_size.
 *
 *  - Write path (Reading vLLM's PagedAttention Kernel, section 3.2 "Writing
 *    into the cache"): slot_mapping holds, per new token, the flat slot
 *    physical_block * page_size + offset; the token's K/V rows are copied
 *    there, bit for bit.
 *
 *  - Attention (Reading vLLM's PagedAttention Kernel, section 4, the dense
 *    reference next to the paged one; Tutorial 13, section 5 "Reading Pages
 *    for Attention", which gathers the valid prefix of every page): for query
 *    row i of request b and query head h_q, with G = H_q / H_kv, the KV head
 *    is g = h_q / G; the row sits at absolute position p = n_b - L + i (the
 *    query rows are the last L positions of the context); the visible keys
 *    are 0..p under the causal mask, 0..n_b-1 without it; scores are
 *    scale * q . k_j, the output is the softmax-weighted sum of v_j, taken in
 *    the two-pass form: maximum, then normalised exponentials.
 *
 *  - FP8 pages (Reading vLLM's PagedAttention Kernel, section 3.2, the
 *    write path's cache dtype and per-tensor scales): e4m3 encoding and
 *    decoding from the format's definition, and the quantising append
 *    (see the block above pa_oracle_e4m3_value). Attention over FP8 pages
 *    is attention over their exact decoded values times the scales.
 *
 * Element storage: query and pages are either bf16 bit patterns (uint16) or
 * fp64. bf16 -> fp64 is exact, so all arithmetic below is fp64 on the exact
 * input values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_F64 = 1 };

/* Error codes returned by the oracle (0 = success). */
enum {
    ORACLE_OK = 0,
    ORACLE_BAD_PAGE = 1,    /* a referenced page id is outside [0, num_pages) */
    ORACLE_BAD_LENGTH = 2,  /* context_len < 0 or > max_pages * page_size     */
    ORACLE_BAD_ARG = 3,     /* shape arguments are inconsistent                */
    ORACLE_NO_MEMORY = 4
};

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int64_t index, int dtype)
{
    if (dtype == ORACLE_BF16)
        return bf16_bits_to_double(((const uint16_t *)base)[index]);
    return ((const double *)base)[index];
}

/*
 * Logical position -> (physical page, slot in page), for one request's
 * block-table row. Returns ORACLE_BAD_PAGE when the page id is outside the
 * pool.
 */
int pa_oracle_translate(const int32_t *block_table_row, int32_t page_size,
                        int32_t num_pages, int64_t pos,
                        int32_t *page, int32_t *slot)
{
    int64_t logical_page = pos / page_size;
    int32_t phys = block_table_row[logical_page];
    *page = phys;
    *slot = (int32_t)(pos % page_size);
    if (phys < 0 || phys >= num_pages)
        return ORACLE_BAD_PAGE;
    return ORACLE_OK;
}

/*
 * Dense copy of the visible K (or V) rows of every request, the "gather"
 * step of the dense baseline (Week 3 Day 4: the dense path first
 * materialises each request's cached K/V contiguously, then attends).
 * pages: [num_pages, H_kv, page_size, D] bf16 bits; block_table [B,
 * max_pages]; dense: [B, H_kv, dense_len, D]. For every request b, KV head h
 * and position t < context_lens[b]: dense[b][h][t][:] = pages[page][h][slot][:]
 * with (page, slot) = translate(block_table[b], t). Rows t >= context_lens[b]
 * are left as they are. Returns ORACLE_OK, or ORACLE_BAD_PAGE (nothing
 * more copied) when a translation leaves the pool or a context is longer
 * than dense_len or the block table.
 */
int pa_oracle_gather(const uint16_t *pages, const int32_t *block_table,
                     const int32_t *context_lens, int32_t B, int32_t H_kv, int32_t D,
                     int32_t page_size, int32_t num_pages, int32_t max_pages,
                     int32_t dense_len, uint16_t *dense)
{
    for (int32_t b = 0; b < B; ++b) {
        const int32_t n = context_lens[b];
        if (n < 0 || n > dense_len || (int64_t)n > (int64_t)max_pages * page_size)
            return ORACLE_BAD_PAGE;
        const int32_t *row = block_table + (int64_t)b * max_pages;
        for (int32_t t = 0; t < n; ++t) {
            int32_t page, slot;
            if (pa_oracle_translate(row, page_size, num_pages, t, &page, &slot))
                return ORACLE_BAD_PAGE;
            for (int32_t h = 0; h < H_kv; ++h) {
                const uint16_t *src = pages + (((int64_t)page * H_kv + h) * page_size + slot) * D;
                uint16_t *dst = dense + (((int64_t)b * H_kv + h) * dense_len + t) * D;
                for (int32_t d = 0; d < D; ++d)
                    dst[d] = src[d];
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Write path. key/value: [B, H_kv, L_new, D] bf16 bits. Pages:
 * [num_pages, H_kv, page_size, D] bf16 bits. slot_mapping: [B, L_new].
 * A negative slot means "no token here" and is skipped. A slot beyond the
 * pool is skipped and counted; the count is returned (0 = every slot valid).
 */
int64_t pa_oracle_append_kv(const uint16_t *key, const uint16_t *value,
                            uint16_t *key_pages, uint16_t *value_pages,
                            const int32_t *slot_mapping,
                            int32_t B, int32_t L_new, int32_t H_kv, int32_t D,
                            int32_t page_size, int32_t num_pages)
{
    int64_t bad = 0;
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t i = 0; i < L_new; ++i) {
            int64_t s = slot_mapping[(int64_t)b * L_new + i];
            if (s < 0)
                continue;
            int64_t page = s / page_size;
            int64_t offset = s % page_size;
            if (page >= num_pages) {
                ++bad;
                continue;
            }
            for (int32_t h = 0; h < H_kv; ++h) {
                int64_t src = (((int64_t)b * H_kv + h) * L_new + i) * D;
                int64_t dst = ((page * H_kv + h) * page_size + offset) * D;
                memcpy(key_pages + dst, key + src, (size_t)D * sizeof(uint16_t));
                memcpy(value_pages + dst, value + src, (size_t)D * sizeof(uint16_t));
            }
        }
    }
    return bad;
}

/*
 * FP8 pages (Reading vLLM's PagedAttention Kernel, section 3.2: the write
 * path takes the cache dtype and per-tensor k_scale / v_scale). The pages
 * fix no rounding; the reading taken: a page stores e4m3 codes c whose value
 * times the scale stands for the input x, c being the e4m3 value nearest to
 * x / scale (x and the quotient in fp32), ties to the code with an even
 * mantissa, magnitudes past the largest finite value saturated to it.
 *
 * e4m3 (the 8-bit floating-point format "E4M3"): a sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent 0 holds the subnormals m * 2^-9; no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.
 */
double pa_oracle_e4m3_value(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e == 0 ? m * ldexp(1.0, -9) : (8 + m) * ldexp(1.0, e - 10);
    return s ? -v : v;
}

/* Nearest e4m3 code to x: a plain search over the 127 finite magnitudes. */
static uint8_t e4m3_encode_one(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int best = 0;
    double best_d = a;                      /* code 0 has the value 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs(pa_oracle_e4m3_value((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

void pa_oracle_e4m3_encode(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = e4m3_encode_one(x[k]);
}

void pa_oracle_e4m3_decode(const uint8_t *codes, double *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k)
        out[k] = pa_oracle_e4m3_value(codes[k]);
}

static float bf16_bits_to_float(uint16_t bits)
{
    const uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * FP8 write path: as pa_oracle_append_kv, but every element is stored as the
 * e4m3 code of (its fp32 value / scale), the quotient rounded to fp32 first.
 * Pages: [num_pages, H_kv, page_size, D] bytes. Returns the count of slots
 * beyond the pool (skipped).
 */
int64_t pa_oracle_append_kv_fp8(const uint16_t *key, const uint16_t *value,
                                uint8_t *key_pages, uint8_t *value_pages,
                                const int32_t *slot_mapping,
                                int32_t B, int32_t L_new, int32_t H_kv, int32_t D,
                                int32_t page_size, int32_t num_pages,
                                float k_scale, float v_scale)
{
    int64_t bad = 0;
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t i = 0; i < L_new; ++i) {
            const int64_t s = slot_mapping[(int64_t)b * L_new + i];
            if (s < 0)
                continue;
            const int64_t page = s / page_size, offset = s % page_size;
            if (page >= num_pages) {
                ++bad;
                continue;
            }
            for (int32_t h = 0; h < H_kv; ++h) {
                const int64_t src = (((int64_t)b * H_kv + h) * L_new + i) * D;
                const int64_t dst = ((page * H_kv + h) * page_size + offset) * D;
                for (int32_t d = 0; d < D; ++d) {
                    const float qk = bf16_bits_to_float(key[src + d]) / k_scale;
                    const float qv = bf16_bits_to_float(value[src + d]) / v_scale;
                    key_pages[dst + d] = e4m3_encode_one(qk);
                    value_pages[dst + d] = e4m3_encode_one(qv);
                }
            }
        }
    }
    return bad;
}

typedef struct {
    const void *query;        /* [B, H_q, L, D]                     */
    const void *key_pages;    /* [num_pages, H_kv, page_size, D]    */
    const void *value_pages;  /* same as key_pages                  */
    const int32_t *block_table;  /* [B, max_pages]                  */
    const int32_t *context_lens; /* [B]                             */
    int32_t B, H_q, H_kv, L, D, page_size, num_pages, max_pages;
    int dtype;
    double scale;
    int causal;
} oracle_problem;

/* One output row: request b, query head hq, query row i -> o[0..D). */
static int attend_row(const oracle_problem *p, int32_t b, int32_t hq, int32_t i,
                      double *o)
{
    const int32_t D = p->D;
    const int32_t group = p->H_q / p->H_kv;
    const int32_t g = hq / group;                 /* KV head of this query head */
    const int64_t n = p->context_lens[b];
    for (int32_t d = 0; d < D; ++d)
        o[d] = 0.0;
    if (n < 0 || n > (int64_t)p->max_pages * p->page_size)
        return ORACLE_BAD_LENGTH;

    const int64_t pos = n - p->L + i;             /* absolute position of row i */
    int64_t visible = p->causal ? pos + 1 : n;    /* keys 0..visible-1          */
    if (visible > n)
        visible = n;
    if (visible <= 0)
        return ORACLE_OK;                          /* no visible key: zeros      */

    const int32_t *bt_row = p->block_table + (int64_t)b * p->max_pages;
    const int64_t q_base = (((int64_t)b * p->H_q + hq) * p->L + i) * D;
    double *scores = (double *)malloc((size_t)visible * sizeof(double));
    int64_t *rows = (int64_t *)malloc((size_t)visible * sizeof(int64_t));
    if (!scores || !rows) {
        free(scores);
        free(rows);
        return ORACLE_NO_MEMORY;
    }

    /* Pass 1: scores s_j = scale * q . k_j over the gathered valid prefix. */
    int status = ORACLE_OK;
    for (int64_t j = 0; j < visible; ++j) {
        int32_t page, slot;
        if (pa_oracle_translate(bt_row, p->page_size, p->num_pages, j, &page, &slot)) {
            status = ORACLE_BAD_PAGE;
            break;
        }
        rows[j] = (((int64_t)page * p->H_kv + g) * p->page_size + slot) * D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += load_elem(p->query, q_base + d, p->dtype) *
                   load_elem(p->key_pages, rows[j] + d, p->dtype);
        scores[j] = p->scale * dot;
    }

    if (status == ORACLE_OK) {
        /* Pass 2: softmax with the maximum subtracted, then the weighted V sum. */
        double m = scores[0];
        for (int64_t j = 1; j < visible; ++j)
            if (scores[j] > m)
                m = scores[j];
        double z = 0.0;
        for (int64_t j = 0; j < visible; ++j)
            z += exp(scores[j] - m);
        for (int64_t j = 0; j < visible; ++j) {
            double w = exp(scores[j] - m) / z;
            for (int32_t d = 0; d < D; ++d)
                o[d] += w * load_elem(p->value_pages, rows[j] + d, p->dtype);
        }
    }
    free(scores);
    free(rows);
    return status;
}

/*
 * Attention over a list of output rows. rows: n_rows triples (b, h_q, i).
 * out: [n_rows, D] fp64. n_threads > 1 spreads rows over OpenMP threads
 * when the file is built with OpenMP; the per-row arithmetic is unchanged.
 * Returns the first nonzero row status, or 0.
 */
int pa_oracle_attention_rows(const void *query, const void *key_pages,
                             const void *value_pages, const int32_t *block_table,
                             const int32_t *context_lens,
                             int32_t B, int32_t H_q, int32_t H_kv, int32_t L,
                             int32_t D, int32_t page_size, int32_t num_pages,
                             int32_t max_pages, int dtype, double scale,
                             int causal, const int32_t *rows, int64_t n_rows,
                             double *out, int n_threads)
{
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || L <= 0 || D <= 0 || page_size <= 0 ||
        num_pages <= 0 || max_pages <= 0 || H_q % H_kv != 0)
        return ORACLE_BAD_ARG;
    oracle_problem p = {query, key_pages, value_pages, block_table, context_lens,
                        B, H_q, H_kv, L, D, page_size, num_pages, max_pages,
                        dtype, scale, causal};
    int status = ORACLE_OK;
    (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
        int32_t b = rows[3 * r], hq = rows[3 * r + 1], i = rows[3 * r + 2];
        int row_status = ORACLE_BAD_ARG;
        if (b >= 0 && b < B && hq >= 0 && hq < H_q && i >= 0 && i < L)
            row_status = attend_row(&p, b, hq, i, out + r * D);
        if (row_status != ORACLE_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            if (status == ORACLE_OK)
                status = row_status;
        }
    }
    return status;
}

/* Attention over every row; out: [B, H_q, L, D] fp64. */
int pa_oracle_attention(const void *query, const void *key_pages,
                        const void *value_pages, const int32_t *block_table,
                        const int32_t *context_lens,
                        int32_t B, int32_t H_q, int32_t H_kv, int32_t L, int32_t D,
                        int32_t page_size, int32_t num_pages, int32_t max_pages,
                        int dtype, double scale, int causal, double *out,
                        int n_threads)
{
    if (B <= 0 || H_q <= 0 || L <= 0)
        return ORACLE_BAD_ARG;
    int64_t n_rows = (int64_t)B * H_q * L;
    int32_t *rows = (int32_t *)malloc((size_t)n_rows * 3 * sizeof(int32_t));
    if (!rows)
        return ORACLE_NO_MEMORY;
    int64_t r = 0;
    for (int32_t b = 0; b < B; ++b)
        for (int32_t hq = 0; hq < H_q; ++hq)
            for (int32_t i = 0; i < L; ++i, ++r) {
                rows[3 * r] = b;
                rows[3 * r + 1] = hq;
                rows[3 * r + 2] = i;
            }
    int status = pa_oracle_attention_rows(query, key_pages, value_pages,
                                          block_table, context_lens, B, H_q, H_kv,
                                          L, D, page_size, num_pages, max_pages,
                                          dtype, scale, causal, rows, n_rows, out,
                                          n_threads);
    free(rows);
    return status;
}
