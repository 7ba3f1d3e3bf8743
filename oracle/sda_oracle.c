/*
 * CPU float64 oracle for DSA sparse decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; both sides receive the same bytes from the seeded input generators.
 *
 * What it follows (vLLM API docs, page "vllm.models.step5.nvidia.ops.
 * sparse_decode_attention"):
 *   - module docstring: each row takes all query heads of one KV group over the
 *     row's selected regions, pages are read in place, FP8 is dequantised, splits
 *     are merged and inactive rows are cleared;
 *   - `sparse_decode_attention` docstring: query/output [rows, heads, 192] with
 *     rows = tokens * G; cache [pages, G, block, 384] holding K then V; regions
 *     [rows, R] with -1 unused; positions/active per row; the G * query_len rows
 *     of one request share one block_table row;
 *   - `_gate`: sigmoid computed in fp32 as 1 / (1 + exp(-g)), rounded to the
 *     gate's dtype (bf16) and read back as fp32;
 *   - `sparse_decode_splits`: the split-count policy;
 * and of the page "vllm.models.step5.nvidia.sparse_attention"
 * (`Step5SplitKVFlashAttentionImpl.forward_with_headwise_gate`, which calls
 * the fused gated sliding-window decode `swa_decode_gated` for the non-DSA
 * layers with window = sliding_window[0] + 1 over the same packed cache).
 * The attention itself is the plain definition: gather the selected regions'
 * tokens, drop tokens past the row's position, softmax(scale * q k^T) v.
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes of the repository):
 *   - region id `id` covers logical tokens [id*RT, (id+1)*RT) of its request,
 *     RT = region_tokens; a token t is visible iff t <= positions[row];
 *   - the gate of (token, group g, head h) is gate[token, g*heads + h];
 *   - an active row with no visible token outputs zeros;
 *   - FP8 values are decode(byte) * per-tensor scale (E4M3 "fn" encoding);
 *   - splits partition the row's compacted list of live regions (ids != -1
 *     whose first token is visible, in their stored order) into contiguous
 *     chunks [floor(s*n/S), floor((s+1)*n/S));
 *   - sliding window: token j of request q sits at p = seq_lens[q] -
 *     query_len + j and sees the `window` tokens [max(0, p - window + 1), p];
 *   - region selection (the adapter page "vllm.models.step5.nvidia.
 *     flashinfer_sparse", `select_regions(scores, current, topk,
 *     topk_lengths=..., sort=False)`, body not shown): candidates are the ids
 *     [0, topk_lengths[r]); the current region is always kept; the other
 *     topk - 1 slots take the highest scores; NaN ranks lowest; ties and the
 *     output order are unstated (this oracle breaks ties by lower id);
 *   - indexer decode scores (the adapter page, `decode_logits` /
 *     `decode_summary_scores`, body not shown; the pages give the shapes and
 *     dtypes and name an FP8 paged MQA-logits kernel): the score of region j
 *     for row (token, g) is sum_h w[h] * max(0, <q_h, m_j>) over the 8 index
 *     heads, with q_h the token's FP8 E4M3 index query of group g, w its fp32
 *     head weights and m_j the FP8 E4M3 mean summary of group g of the
 *     8-token region j; region j's summary sits in summary slot
 *     page * (block / 8) + (8j mod block) / 8 with page = block_table[req,
 *     8j / block]; regions [0, pos / 8] are scored (pos as for the sliding
 *     window), the rest of the row is -inf.  This formula is a reading, not
 *     printed on the pages: the CPU tests pin the oracle to it, nothing pins
 *     it to the pages' own kernel.
 *
 * Everything is float64 except the gate, whose fp32 sigmoid and bf16 rounding
 * are a quantisation the page fixes in those precisions.
 *
 * Parity status: every function here is pinned by the CPU tests in
 * tests/test_oracle_pins.py (textbook dense attention, closed forms,
 * invariants, torch's e4m3/bf16 decoders, the page's split truth table).
 * oracle_summary_scores is pinned to its reading only (parity with the pages'
 * indexer kernel unpinned: its formula is not on the pages).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DIM 192
#define ORACLE_ROW 384

/* Mutation hooks.  A normal build has ORACLE_MUTANT == 0 and every MUT(n) is
 * false.  The pin-strength test compiles extra copies with one planted
 * mistake each (-DORACLE_MUTANT=n) and checks that some pin catches it. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARGS = -1,        /* a size or pointer argument is unusable   */
    ORACLE_ERR_REGION = -2,      /* a region id below -1                      */
    ORACLE_ERR_TABLE = -3,       /* a visible token maps past the table width */
    ORACLE_ERR_PAGE = -4,        /* a table entry is not a page of the cache  */
    ORACLE_ERR_ALLOC = -5,
};

/* ---------------------------------------------------------------------------
 * Number formats.
 * ------------------------------------------------------------------------- */

/* OCP 8-bit floating point, E4M3 ("fn": finite, no infinities): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds the
 * subnormals m * 2^-9; S.1111.111 is NaN; every other code is normal,
 * (1 + m/8) * 2^(e-7), up to 448. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double mag;
    if (e == 0xF && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, MUT(16) ? -10 : -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - (MUT(1) ? 8 : 7));
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_decode(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (NaN kept quiet). */
uint16_t oracle_bf16_round(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* `_gate`: g read as fp32, sigmoid = 1 / (1 + exp(-g)) with a correctly
 * rounded fp32 division, then rounded to bf16 and read back.  Returns the
 * gate factor as a double holding that bf16 value exactly. */
double oracle_gate_factor(uint16_t gate_bits)
{
    volatile float g = (float)oracle_bf16_decode(gate_bits);
    volatile float e = expf(MUT(2) ? g : -g);
    volatile float denom = 1.0f + e;
    volatile float sig = 1.0f / denom;
    return MUT(12) ? (double)sig : oracle_bf16_decode(oracle_bf16_round(sig));
}

/* `sparse_decode_splits`: start at one split and keep doubling while fewer
 * than 32 and rows * splits * 2 still fits in 256 programs. */
int oracle_sparse_decode_splits(int rows)
{
    int splits = 1;
    while (splits < 32 && (MUT(15) ? (long long)rows * splits * 2 < 256 : (long long)rows * splits * 2 <= 256))
        splits *= 2;
    return splits;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------------------
 * Problem description shared by the entry points below.
 * ------------------------------------------------------------------------- */

typedef struct {
    /* query [rows, heads, 192] bf16 bits, element strides q_s0, q_s1 (dim 1) */
    const uint16_t *query;
    int64_t q_s0, q_s1;
    int rows, heads;
    /* cache [pages, groups, block, 384]; bf16 bits or E4M3 bytes */
    const void *cache;
    int cache_fp8;
    int64_t pages;
    int groups, block;
    int64_t c_s0, c_s1, c_s2;
    /* regions [rows, R] int32, row stride reg_s0 */
    const int32_t *regions;
    int64_t reg_s0;
    int num_regions;
    /* block_table [table_rows, table_cols] int32, row stride bt_s0 */
    const int32_t *block_table;
    int64_t bt_s0;
    int table_rows, table_cols;
    const int32_t *positions;   /* [rows] */
    const uint8_t *active;      /* [rows], nonzero = active */
    double scale;
    int query_len;
    int region_tokens;
    double k_scale, v_scale;    /* ignored for a bf16 cache */
    const uint16_t *gate;       /* [tokens, groups*heads] bf16 bits or NULL */
    int64_t g_s0, g_s1;
} oracle_problem;

static double cache_value(const oracle_problem *p, int64_t page, int g, int off, int col)
{
    int64_t idx = page * p->c_s0 + (int64_t)g * p->c_s1 + (int64_t)off * p->c_s2 + col;
    if (p->cache_fp8)
        return oracle_e4m3_decode(((const uint8_t *)p->cache)[idx]);
    return oracle_bf16_decode(((const uint16_t *)p->cache)[idx]);
}

static int check_problem(const oracle_problem *p)
{
    if (!p->query || !p->cache || !p->regions || !p->block_table || !p->positions || !p->active)
        return ORACLE_ERR_ARGS;
    if (p->rows < 0 || p->heads < 1 || p->groups < 1 || p->block < 1 || p->pages < 1)
        return ORACLE_ERR_ARGS;
    if (p->num_regions < 0 || p->query_len < 1 || p->region_tokens < 1 || p->table_cols < 0)
        return ORACLE_ERR_ARGS;
    return ORACLE_OK;
}

/* The visible tokens of one row, in the order the row lists its regions:
 * for each region slot j with id = regions[row, j] != -1, the tokens
 * t in [id*RT, id*RT + RT) with t <= pos.  Region slots [j_lo, j_hi) of the
 * compacted live list only (see split partition above); pass j_lo = 0,
 * j_hi = INT32_MAX for all of them.  Returns the count or a negative error. */
static int64_t gather_tokens(const oracle_problem *p, int row, int64_t live_lo, int64_t live_hi,
                             int64_t *tokens, int64_t cap)
{
    const int32_t *reg = p->regions + (int64_t)row * p->reg_s0;
    int64_t pos = p->positions[row];
    int64_t rt = p->region_tokens;
    int64_t n = 0, live = 0;
    for (int j = 0; j < p->num_regions; ++j) {
        int64_t id = reg[j];
        if (id == -1)
            continue;
        if (id < -1)
            return ORACLE_ERR_REGION;
        if (id * rt > pos)          /* no visible token: not a live region */
            continue;
        int64_t k = live++;
        if (k < live_lo || k >= live_hi)
            continue;
        for (int64_t t = id * rt + (MUT(4) ? 1 : 0); t < id * rt + rt; ++t) {
            if (MUT(3) ? t >= pos : t > pos)
                break;
            if (n >= cap)
                return ORACLE_ERR_ARGS;
            tokens[n++] = t;
        }
    }
    return n;
}

static int64_t count_live_regions(const oracle_problem *p, int row)
{
    const int32_t *reg = p->regions + (int64_t)row * p->reg_s0;
    int64_t pos = p->positions[row];
    int64_t n = 0;
    for (int j = 0; j < p->num_regions; ++j) {
        int64_t id = reg[j];
        if (id >= 0 && id * (int64_t)p->region_tokens <= pos)
            ++n;
    }
    return n;
}

/* softmax(scale * q k^T) v for every head of `row` over the given tokens.
 * Writes o[heads][192] (unnormalised output divided by its softmax sum, i.e.
 * the attention output) and, when lse != NULL, lse[h] = log(sum_t exp(s_t))
 * (-inf when there are no tokens, with o = 0). */
static int attend(const oracle_problem *p, int row, const int64_t *tokens, int64_t n,
                  double *o, double *lse)
{
    int g = MUT(5) ? row / p->groups % p->groups : row % p->groups;
    int64_t req = row / ((int64_t)p->groups * (MUT(6) ? 1 : p->query_len));
    double ks = p->cache_fp8 ? p->k_scale : 1.0;
    double vs = p->cache_fp8 ? p->v_scale : 1.0;
    memset(o, 0, sizeof(double) * (size_t)p->heads * ORACLE_DIM);
    if (n == 0) {
        if (lse)
            for (int h = 0; h < p->heads; ++h)
                lse[h] = -INFINITY;
        return ORACLE_OK;
    }
    if (req >= p->table_rows)
        return ORACLE_ERR_TABLE;

    /* Resolve every token to its page and dequantised K, V rows. */
    double *k = malloc(sizeof(double) * (size_t)n * ORACLE_DIM);
    double *v = malloc(sizeof(double) * (size_t)n * ORACLE_DIM);
    double *s = malloc(sizeof(double) * (size_t)n);
    if (!k || !v || !s) {
        free(k); free(v); free(s);
        return ORACLE_ERR_ALLOC;
    }
    int err = ORACLE_OK;
    for (int64_t i = 0; i < n && !err; ++i) {
        int64_t t = tokens[i];
        int64_t col = t / p->block;
        int off = (int)(MUT(10) ? (t + 1) % p->block : t % p->block);
        if (col >= p->table_cols) { err = ORACLE_ERR_TABLE; break; }
        int64_t page = p->block_table[req * p->bt_s0 + col];
        if (page < 0 || page >= p->pages) { err = ORACLE_ERR_PAGE; break; }
        for (int d = 0; d < ORACLE_DIM; ++d) {
            k[i * ORACLE_DIM + d] = cache_value(p, page, g, off, MUT(7) ? ORACLE_DIM + d : d) * ks;
            v[i * ORACLE_DIM + d] = cache_value(p, page, g, off, MUT(7) ? d : ORACLE_DIM + d) * (MUT(8) ? 1.0 : vs);
        }
    }
    for (int h = 0; h < p->heads && !err; ++h) {
        const uint16_t *q = p->query + (int64_t)row * p->q_s0 + (int64_t)h * p->q_s1;
        double smax = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            double dot = 0.0;
            for (int d = 0; d < ORACLE_DIM; ++d)
                dot += oracle_bf16_decode(q[d]) * k[i * ORACLE_DIM + d];
            s[i] = (MUT(9) ? 1.0 : p->scale) * dot;
            if (s[i] > smax)
                smax = s[i];
        }
        double sum = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            s[i] = exp(s[i] - smax);
            sum += s[i];
        }
        double *oh = o + (size_t)h * ORACLE_DIM;
        for (int64_t i = 0; i < n; ++i)
            for (int d = 0; d < ORACLE_DIM; ++d)
                oh[d] += (s[i] / sum) * v[i * ORACLE_DIM + d];
        if (lse)
            lse[h] = (MUT(14) ? 0.0 : smax) + log(sum);
    }
    free(k); free(v); free(s);
    return err;
}

static oracle_problem make_problem(
    const uint16_t *query, int64_t q_s0, int64_t q_s1, int rows, int heads,
    const void *cache, int cache_fp8, int64_t pages, int groups, int block,
    int64_t c_s0, int64_t c_s1, int64_t c_s2,
    const int32_t *regions, int64_t reg_s0, int num_regions,
    const int32_t *block_table, int64_t bt_s0, int table_rows, int table_cols,
    const int32_t *positions, const uint8_t *active,
    double scale, int query_len, int region_tokens, double k_scale, double v_scale,
    const uint16_t *gate, int64_t g_s0, int64_t g_s1)
{
    oracle_problem p;
    p.query = query; p.q_s0 = q_s0; p.q_s1 = q_s1; p.rows = rows; p.heads = heads;
    p.cache = cache; p.cache_fp8 = cache_fp8; p.pages = pages; p.groups = groups;
    p.block = block; p.c_s0 = c_s0; p.c_s1 = c_s1; p.c_s2 = c_s2;
    p.regions = regions; p.reg_s0 = reg_s0; p.num_regions = num_regions;
    p.block_table = block_table; p.bt_s0 = bt_s0; p.table_rows = table_rows;
    p.table_cols = table_cols; p.positions = positions; p.active = active;
    p.scale = scale; p.query_len = query_len; p.region_tokens = region_tokens;
    p.k_scale = k_scale; p.v_scale = v_scale;
    p.gate = gate; p.g_s0 = g_s0; p.g_s1 = g_s1;
    return p;
}

/* ---------------------------------------------------------------------------
 * Entry points.
 * ------------------------------------------------------------------------- */

/* The full op for the listed rows (row_ids == NULL: rows 0..rows-1 in order).
 * out: [n_out][heads][192] float64.  Per row:
 *   1. inactive -> +0.0 everywhere;
 *   2. gather the visible tokens of the row's selected regions;
 *   3. per head, softmax(scale * q . k_t) weighted sum of v_t (0 if no token);
 *   4. with a gate, multiply by the bf16-rounded fp32 sigmoid of
 *      gate[row / G, (row % G) * heads + h].
 * Returns 0 or the first negative error found. */
int oracle_sparse_decode_attention(
    const uint16_t *query, int64_t q_s0, int64_t q_s1, int rows, int heads,
    const void *cache, int cache_fp8, int64_t pages, int groups, int block,
    int64_t c_s0, int64_t c_s1, int64_t c_s2,
    const int32_t *regions, int64_t reg_s0, int num_regions,
    const int32_t *block_table, int64_t bt_s0, int table_rows, int table_cols,
    const int32_t *positions, const uint8_t *active,
    double scale, int query_len, int region_tokens, double k_scale, double v_scale,
    const uint16_t *gate, int64_t g_s0, int64_t g_s1,
    const int32_t *row_ids, int n_out, double *out)
{
    oracle_problem p = make_problem(query, q_s0, q_s1, rows, heads, cache, cache_fp8, pages,
                                    groups, block, c_s0, c_s1, c_s2, regions, reg_s0,
                                    num_regions, block_table, bt_s0, table_rows, table_cols,
                                    positions, active, scale, query_len, region_tokens,
                                    k_scale, v_scale, gate, g_s0, g_s1);
    int err = check_problem(&p);
    if (err)
        return err;
    if (!row_ids)
        n_out = rows;
    int64_t cap = (int64_t)num_regions * region_tokens;
    int first_err = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_out; ++i) {
        int row = row_ids ? row_ids[i] : i;
        double *o = out + (size_t)i * heads * ORACLE_DIM;
        int e = ORACLE_OK;
        if (row < 0 || row >= rows) {
            e = ORACLE_ERR_ARGS;
        } else if (!MUT(17) && !p.active[row]) {
            for (size_t j = 0; j < (size_t)heads * ORACLE_DIM; ++j)
                o[j] = 0.0;
        } else {
            int64_t *tok = malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
            if (!tok) {
                e = ORACLE_ERR_ALLOC;
            } else {
                int64_t n = gather_tokens(&p, row, 0, INT64_MAX, tok, cap);
                e = n < 0 ? (int)n : attend(&p, row, tok, n, o, NULL);
                free(tok);
            }
            if (!e && gate) {
                int64_t token = row / groups;
                int g = row % groups;
                for (int h = 0; h < heads; ++h) {
                    double f = oracle_gate_factor(gate[token * g_s0 + (int64_t)(MUT(11) ? h * groups + g : g * heads + h) * g_s1]);
                    for (int d = 0; d < ORACLE_DIM; ++d)
                        o[(size_t)h * ORACLE_DIM + d] *= f;
                }
            }
        }
        if (e) {
#pragma omp critical
            if (!first_err)
                first_err = e;
        }
    }
    return first_err;
}

/* Split-KV partials of the listed rows: for split s of S the row's live
 * regions [floor(s*n/S), floor((s+1)*n/S)) of its compacted live list.
 * partial: [n_out][S][heads][192] attention output of that chunk alone
 * (0 when it has no token); lse: [n_out][S][heads] natural-log sum of
 * exp(scale * q . k) over the chunk (-inf when empty).  No gate, and
 * inactive rows are computed like active ones (the caller ignores them). */
int oracle_split_partials(
    const uint16_t *query, int64_t q_s0, int64_t q_s1, int rows, int heads,
    const void *cache, int cache_fp8, int64_t pages, int groups, int block,
    int64_t c_s0, int64_t c_s1, int64_t c_s2,
    const int32_t *regions, int64_t reg_s0, int num_regions,
    const int32_t *block_table, int64_t bt_s0, int table_rows, int table_cols,
    const int32_t *positions, const uint8_t *active,
    double scale, int query_len, int region_tokens, double k_scale, double v_scale,
    int splits, const int32_t *row_ids, int n_out, double *partial, double *lse)
{
    oracle_problem p = make_problem(query, q_s0, q_s1, rows, heads, cache, cache_fp8, pages,
                                    groups, block, c_s0, c_s1, c_s2, regions, reg_s0,
                                    num_regions, block_table, bt_s0, table_rows, table_cols,
                                    positions, active, scale, query_len, region_tokens,
                                    k_scale, v_scale, NULL, 0, 0);
    int err = check_problem(&p);
    if (err)
        return err;
    if (splits < 1)
        return ORACLE_ERR_ARGS;
    if (!row_ids)
        n_out = rows;
    int64_t cap = (int64_t)num_regions * region_tokens;
    int first_err = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_out; ++i) {
        int row = row_ids ? row_ids[i] : i;
        int e = ORACLE_OK;
        int64_t *tok = malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
        if (!tok)
            e = ORACLE_ERR_ALLOC;
        if (!e && (row < 0 || row >= rows))
            e = ORACLE_ERR_ARGS;
        int64_t n_live = e ? 0 : count_live_regions(&p, row);
        for (int s = 0; s < splits && !e; ++s) {
            int64_t lo = MUT(13) ? ((int64_t)s * n_live + splits - 1) / splits : (int64_t)s * n_live / splits;
            int64_t hi = MUT(13) ? ((int64_t)(s + 1) * n_live + splits - 1) / splits : (int64_t)(s + 1) * n_live / splits;
            size_t base = ((size_t)i * splits + s) * heads;
            int64_t n = gather_tokens(&p, row, lo, hi, tok, cap);
            e = n < 0 ? (int)n : attend(&p, row, tok, n, partial + base * ORACLE_DIM, lse + base);
        }
        free(tok);
        if (e) {
#pragma omp critical
            if (!first_err)
                first_err = e;
        }
    }
    return first_err;
}

/* Gated sliding-window decode for the listed rows (row_ids == NULL: all).
 * Row r is group r % G of token r / G; its request is r / (G * query_len),
 * its token within the request j = (r / G) % query_len, its position
 * p = seq_lens[request] - query_len + j; it attends, per head, over the
 * tokens [max(0, p - window + 1), p] of its request (none when p < 0), then
 * the optional headwise gate applies as for the sparse path.  Every row is
 * active.  out: [n_out][heads][192] float64. */
int oracle_swa_decode(
    const uint16_t *query, int64_t q_s0, int64_t q_s1, int rows, int heads,
    const void *cache, int cache_fp8, int64_t pages, int groups, int block,
    int64_t c_s0, int64_t c_s1, int64_t c_s2,
    const int32_t *block_table, int64_t bt_s0, int table_rows, int table_cols,
    const int32_t *seq_lens, int num_requests,
    double scale, int query_len, int window, double k_scale, double v_scale,
    const uint16_t *gate, int64_t g_s0, int64_t g_s1,
    const int32_t *row_ids, int n_out, double *out)
{
    static const int32_t no_region = -1;
    static const uint8_t one = 1;
    oracle_problem p = make_problem(query, q_s0, q_s1, rows, heads, cache, cache_fp8, pages,
                                    groups, block, c_s0, c_s1, c_s2, &no_region, 0, 1,
                                    block_table, bt_s0, table_rows, table_cols, &no_region, &one,
                                    scale, query_len, 1, k_scale, v_scale, gate, g_s0, g_s1);
    int err = check_problem(&p);
    if (err)
        return err;
    if (!seq_lens || window < 1 || num_requests < 0)
        return ORACLE_ERR_ARGS;
    if (!row_ids)
        n_out = rows;
    int first_err = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_out; ++i) {
        int row = row_ids ? row_ids[i] : i;
        double *o = out + (size_t)i * heads * ORACLE_DIM;
        int e = ORACLE_OK;
        int64_t req = row / ((int64_t)groups * query_len);
        if (row < 0 || row >= rows || req >= num_requests) {
            e = ORACLE_ERR_ARGS;
        } else {
            int64_t j = (row / groups) % query_len;
            int64_t pos = (int64_t)seq_lens[req] - query_len + j + (MUT(19) ? 1 : 0);
            int64_t lo = pos - window + (MUT(18) ? 0 : 1);
            if (lo < 0)
                lo = 0;
            int64_t n = pos >= lo ? pos - lo + 1 : 0;
            int64_t *tok = malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
            if (!tok) {
                e = ORACLE_ERR_ALLOC;
            } else {
                for (int64_t k = 0; k < n; ++k)
                    tok[k] = lo + k;
                e = attend(&p, row, tok, n, o, NULL);
                free(tok);
            }
            if (!e && gate) {
                int64_t token = row / groups;
                int g = row % groups;
                for (int h = 0; h < heads; ++h) {
                    double f = oracle_gate_factor(gate[token * g_s0 + (int64_t)(g * heads + h) * g_s1]);
                    for (int d = 0; d < ORACLE_DIM; ++d)
                        o[(size_t)h * ORACLE_DIM + d] *= f;
                }
            }
        }
        if (e) {
#pragma omp critical
            if (!first_err)
                first_err = e;
        }
    }
    return first_err;
}

/* One row of region selection: writes the selected ids (current first, then
 * the others in ascending id order) to out[0..topk), padding with -1.  Plain
 * definition: rank every candidate other than the current one by (score
 * descending, id ascending) with a full sort and keep the first topk - 1. */
typedef struct {
    float score;
    int32_t id;
} oracle_cand;

static int cand_cmp(const void *a, const void *b)
{
    const oracle_cand *x = a, *y = b;
    int xn = isnan(x->score), yn = isnan(y->score);
    if (xn != yn)
        return xn - yn;                      /* NaN after everything */
    if (!xn && x->score != y->score)
        return x->score > y->score ? -1 : 1;  /* higher score first */
    return (x->id > y->id) - (x->id < y->id);
}

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int oracle_select_regions(const float *scores, int64_t s_s0, int rows, int n_cols,
                          const int32_t *current, const int32_t *topk_lengths, int topk,
                          int32_t *out)
{
    if (!scores || !current || !out || rows < 0 || n_cols < 0 || topk < 1)
        return ORACLE_ERR_ARGS;
    int first_err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < rows; ++r) {
        int32_t *o = out + (int64_t)r * topk;
        int len = topk_lengths ? topk_lengths[r] : n_cols;
        if (len > n_cols)
            len = n_cols;
        if (len < 0)
            len = 0;
        int cur = current[r];
        int forced = cur >= 0 && cur < len && !MUT(20);
        oracle_cand *c = malloc(sizeof(oracle_cand) * (size_t)(len > 0 ? len : 1));
        int32_t *ids = malloc(sizeof(int32_t) * (size_t)(topk > 0 ? topk : 1));
        if (!c || !ids) {
            free(c);
            free(ids);
#pragma omp critical
            first_err = ORACLE_ERR_ALLOC;
            continue;
        }
        int n = 0;
        for (int i = 0; i < len; ++i) {
            if (forced && i == cur)
                continue;
            c[n].score = scores[(int64_t)r * s_s0 + i];
            c[n].id = i;
            ++n;
        }
        qsort(c, (size_t)n, sizeof *c, cand_cmp);
        int keep = topk - forced;
        if (keep > n)
            keep = n;
        int k = 0;
        if (forced)
            o[k++] = cur;
        for (int i = 0; i < keep; ++i)
            ids[i] = c[MUT(21) ? n - 1 - i : i].id;
        qsort(ids, (size_t)keep, sizeof *ids, cmp_i32);
        for (int i = 0; i < keep; ++i)
            o[k++] = ids[i];
        while (k < topk)
            o[k++] = -1;
        free(ids);
        free(c);
    }
    return first_err;
}

/* Indexer decode scores for the rows (token, g) listed in row_ids (all
 * tokens * groups rows when row_ids is NULL), written densely to
 * scores[n_out, n_cols] with the -inf tail, plus the row's current region and
 * scored length.  Plain definition: for every scored region, resolve its
 * summary slot through the block table, decode the 256 summary bytes and each
 * head's 256 query bytes, take the dot product, clamp at zero, weight, sum over
 * the 8 heads. */
#define ORACLE_IDX_HEADS 8
#define ORACLE_IDX_DIM 256
#define ORACLE_IDX_REGION 8

int oracle_summary_scores(const uint8_t *query, int64_t q_s0, int64_t q_s1, int tokens, int groups,
                          const float *weights, int64_t w_s0, int64_t w_s1,
                          const uint8_t *summaries, int64_t m_s0, int64_t n_slots,
                          const int32_t *block_table, int64_t bt_s0, int n_reqs, int width,
                          const int32_t *seq_lens, int block, int query_len, int n_cols,
                          const int32_t *row_ids, int n_out, double *scores, int32_t *current,
                          int32_t *lengths)
{
    if (!query || !weights || !summaries || !block_table || !seq_lens || !scores || tokens < 0 ||
        groups < 1 || block < ORACLE_IDX_REGION || block % ORACLE_IDX_REGION || query_len < 1 ||
        n_cols < 0 || n_out < 0 || tokens % query_len || tokens / query_len > n_reqs)
        return ORACLE_ERR_ARGS;
    const int per_page = block / ORACLE_IDX_REGION;
    int first_err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n_out; ++i) {
        int64_t row = row_ids ? row_ids[i] : i;
        double *out = scores + (int64_t)i * n_cols;
        int err = ORACLE_OK;
        if (row < 0 || row >= (int64_t)tokens * groups) {
            err = ORACLE_ERR_ARGS;
        } else {
            int tok = (int)(row / groups), g = (int)(row % groups);
            if (MUT(25))
                g = 0;
            int req = tok / query_len;
            int64_t pos = (int64_t)seq_lens[req] - query_len + tok % query_len + (MUT(26) ? 1 : 0);
            int64_t n = pos >= 0 ? pos / ORACLE_IDX_REGION + (MUT(24) ? 0 : 1) : 0;
            if (n > n_cols)
                n = n_cols;
            if (current)
                current[i] = pos >= 0 ? (int32_t)(pos / ORACLE_IDX_REGION) : -1;
            if (lengths)
                lengths[i] = (int32_t)n;
            double q[ORACLE_IDX_HEADS][ORACLE_IDX_DIM], w[ORACLE_IDX_HEADS];
            for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
                const uint8_t *qh = query + (int64_t)tok * q_s0 + (int64_t)g * q_s1 +
                                    (int64_t)h * ORACLE_IDX_DIM;
                for (int d = 0; d < ORACLE_IDX_DIM; ++d)
                    q[h][d] = oracle_e4m3_decode(qh[d]);
                w[h] = weights[(int64_t)tok * w_s0 + (int64_t)g * w_s1 +
                               (MUT(23) ? (h + 1) % ORACLE_IDX_HEADS : h)];
            }
            for (int64_t j = 0; j < n_cols; ++j)
                out[j] = -INFINITY;
            for (int64_t j = 0; j < n && !err; ++j) {
                int64_t t0 = j * ORACLE_IDX_REGION;
                if (t0 / block >= width) {
                    err = ORACLE_ERR_TABLE;
                    break;
                }
                int64_t page = block_table[(int64_t)req * bt_s0 + t0 / block];
                int64_t slot = page * per_page + (t0 % block) / ORACLE_IDX_REGION;
                if (page < 0 || slot >= n_slots) {
                    err = ORACLE_ERR_PAGE;
                    break;
                }
                const uint8_t *m = summaries + slot * m_s0 + (int64_t)g * ORACLE_IDX_DIM;
                double md[ORACLE_IDX_DIM];
                for (int d = 0; d < ORACLE_IDX_DIM; ++d)
                    md[d] = oracle_e4m3_decode(m[d]);
                double sum = 0.0;
                for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
                    double dot = 0.0;
                    for (int d = 0; d < ORACLE_IDX_DIM; ++d)
                        dot += q[h][d] * md[d];
                    sum += w[h] * (MUT(22) ? dot : (dot > 0.0 ? dot : 0.0));
                }
                out[j] = sum;
            }
        }
        if (err) {
#pragma omp critical
            if (!first_err)
                first_err = err;
        }
    }
    return first_err;
}
