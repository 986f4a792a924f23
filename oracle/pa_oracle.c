/*
 * pa_oracle.c -- plain, slow, obviously-correct CPU oracle for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file.  Its only users are the test suite, the smoke check in
 * __graft_entry__.py, and the CPU-baseline leg of bench.py.  It shares no code,
 * header, table or helper with the CUDA kernels of paged_attention_decode_split_gb300.
 *
 * Everything is computed in IEEE double precision.  bf16 inputs are widened to
 * double exactly (a bf16 value is the top 16 bits of an IEEE binary32 value).
 *
 * Sources (web pages this library restates; cited by title and section):
 *   [DCU-832]  "DCU page832 attention" (luanjiahao.me, 2026-07-17):
 *              Sec.1 block-table address math; Sec.4 K/V cache shape
 *              [num_physical_pages, BLOCK_SIZE, kv_heads, head_size] after unbind;
 *              Sec.5 per-tile loop score = dot(Q,K)*scale + online softmax;
 *              Sec.7 page-contiguous decode loop ("no logical page is skipped,
 *              the causal range is unchanged").
 *   [RADEON]   "Hybrid SSM decode rate on dual Radeon under vLLM"
 *              (cadamcat.github.io, hybrid-ssm-collapse), section on the
 *              upstream fix vllm#45916: the KV range is cut across many
 *              workgroups and the pieces are reduced afterwards.
 *   [MI350P]   "Qwen3.8 on MI350P: kernels, errors and measurements"
 *              (flozi.net), Lektion 3: verify rows share K/V tiles, a causal
 *              mask is applied per row, partial softmax statistics are merged.
 *
 * Readings where the pages are silent:
 *   - query head h reads KV head h / (num_q_heads / num_kv_heads)  (contiguous GQA);
 *   - seq_lens[b] counts every cached token of sequence b, including the q_len
 *     rows just written; row r (0-based) of a q_len-row block sees keys
 *     0 .. seq_lens[b] - q_len + r inclusive;
 *   - plain softmax: no ALiBi, sinks or soft-cap (the DCU page lists those as
 *     excluded conditions, Sec.6);
 *   - sliding window (the RTX 3090 page's 2048-position window): with window
 *     W > 0 a row sees only its last W visible keys, i.e. keys
 *     (last visible key - W, last visible key]; W = 0 means no window;
 *   - a row that sees no key returns zeros;
 *   - a negative slot in reshape_and_cache is a padding slot and is skipped;
 *   - quantised KV cache (the RTX 3090 page runs a Q4_0 cache, ggml's own
 *     format): here fp8 e4m3 with one binary32 scale per KV head, code =
 *     e4m3(x / scale) with the division in binary32, rounding to nearest
 *     even and saturating to +-448; the cached value is decoded(code) * scale.
 *
 * Return codes: 0 ok, -1 bad argument, -2 an index (page, slot) out of range.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bf16 bit pattern. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp8 e4m3 (the "FN" variant): 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits, no infinities; exponent 15 with mantissa 7 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448.  Exponent 0 holds the
 * subnormals m/8 * 2^-6.  Decoding is exact in double. */
static double e4m3_to_double(uint8_t c)
{
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return (c & 0x80) ? -v : v;
}

/* Nearest e4m3 value to x, ties to the even code; magnitudes at or above 448
 * (infinities included) give +-448; NaN gives NaN with x's sign. */
static uint8_t e4m3_from_float(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x))
        return sign | 0x7F;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* representable values are spaced 2^(E-3) in the binade [2^E, 2^(E+1))
     * for E >= -6, and 2^-9 below 2^-6 */
    int E;
    frexp(a, &E); /* a = f * 2^E with f in [0.5, 1) */
    E -= 1;
    if (a == 0.0 || E < -6)
        E = -6;
    double step = ldexp(1.0, E - 3);
    double k = floor(a / step);
    double rem = a - k * step;
    if (rem > 0.5 * step || (rem == 0.5 * step && fmod(k, 2.0) != 0.0))
        k += 1.0;
    double v = k * step; /* the rounded magnitude, <= 448 */
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9));
    int e2;
    frexp(v, &e2);
    int eb = e2 - 1; /* v in [2^eb, 2^(eb+1)) */
    int mant = (int)(v / ldexp(1.0, eb - 3)) - 8;
    return sign | (uint8_t)(((eb + 7) << 3) | mant);
}

int oracle_e4m3_encode(const float *x, uint8_t *codes, int64_t n)
{
    if (n < 0 || (n > 0 && (!x || !codes)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = e4m3_from_float(x[i]);
    return 0;
}

int oracle_e4m3_decode(const uint8_t *codes, double *out, int64_t n)
{
    if (n < 0 || (n > 0 && (!codes || !out)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_to_double(codes[i]);
    return 0;
}

/* [DCU-832] Sec.1: logical_page = t // BLOCK_SIZE, page_offset = t % BLOCK_SIZE,
 * physical_page = block_table[logical_page]; then the cache strides over
 * (page, offset, kv_head, dim) of a [num_pages, BLOCK_SIZE, kv_heads, head_dim]
 * tensor (Sec.4) give the element offset of the row.  Returns -1 when the
 * table entry is outside [0, num_pages). */
static int64_t row_offset(const int32_t *block_table_row, int64_t t, int block_size,
                          int num_kv_heads, int head_dim, int kv_head, int64_t num_pages)
{
    int64_t logical_page = t / block_size;
    int64_t page_offset = t % block_size;
    int64_t physical_page = block_table_row[logical_page];
    if (physical_page < 0 || physical_page >= num_pages)
        return -1;
    return ((physical_page * block_size + page_offset) * num_kv_heads + kv_head) * (int64_t)head_dim;
}

/* ------------------------------------------------------------------------ */
/* reshape_and_cache: k_cache[s / BS, s % BS, h, :] = k_new[i, h, :] for the
 * slot s = slot_mapping[i] of every new token i (same for V).  Bit copy. */
int oracle_reshape_and_cache(const uint16_t *k_new, const uint16_t *v_new,
                             uint16_t *k_cache, uint16_t *v_cache,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int block_size,
                             int64_t num_pages)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_pages < 0)
        return -1;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue; /* padding slot */
        if (s >= num_pages * block_size)
            return -2;
        int64_t page = s / block_size;
        int64_t off = s % block_size;
        int64_t dst = (page * block_size + off) * row;
        memcpy(k_cache + dst, k_new + i * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_cache + dst, v_new + i * row, (size_t)row * sizeof(uint16_t));
    }
    return 0;
}

/* reshape_and_cache into an fp8 cache: the same scatter, each element of KV
 * head h stored as e4m3(bf16 value / scale[h]) with the division in binary32. */
int oracle_reshape_and_cache_fp8(const uint16_t *k_new, const uint16_t *v_new,
                                 uint8_t *k_cache, uint8_t *v_cache,
                                 const int64_t *slot_mapping, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int64_t num_pages, const float *k_scale, const float *v_scale)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_pages < 0 ||
        !k_scale || !v_scale)
        return -1;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= num_pages * block_size)
            return -2;
        int64_t dst = ((s / block_size) * block_size + s % block_size) * row;
        for (int h = 0; h < num_kv_heads; ++h)
            for (int d = 0; d < head_dim; ++d) {
                int64_t e = (int64_t)h * head_dim + d;
                float kq = (float)bf16_to_double(k_new[i * row + e]) / k_scale[h];
                float vq = (float)bf16_to_double(v_new[i * row + e]) / v_scale[h];
                k_cache[dst + e] = e4m3_from_float(kq);
                v_cache[dst + e] = e4m3_from_float(vq);
            }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Problem description shared by the attention entry points. */
typedef struct {
    const uint16_t *q;          /* [num_seqs*q_len, num_q_heads, head_dim] bf16 bits */
    const uint16_t *k_cache;    /* [num_pages, block_size, num_kv_heads, head_dim]  */
    const uint16_t *v_cache;
    const int32_t *block_table; /* [num_seqs, max_pages_per_seq] */
    const int32_t *seq_lens;    /* [num_seqs] */
    int num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_pages_per_seq;
    int64_t num_pages;
    double scale;
    int64_t window; /* 0: none; W > 0: each row sees only its last W visible keys */
    /* fp8 cache (k_cache/v_cache unused): e4m3 codes and one scale per KV head */
    const uint8_t *k_cache8, *v_cache8;
    const float *k_scale, *v_scale;
} problem;

/* Cached K (which = 0) or V (which = 1) element at element offset off. */
static double kv_elem(const problem *p, int which, int64_t off, int kv_head)
{
    if (p->k_cache8) {
        const uint8_t *c = which ? p->v_cache8 : p->k_cache8;
        const float *sc = which ? p->v_scale : p->k_scale;
        return e4m3_to_double(c[off]) * (double)sc[kv_head];
    }
    return bf16_to_double((which ? p->v_cache : p->k_cache)[off]);
}

/* Number of keys query row r of sequence b may attend to (causal rule). */
static int64_t visible_keys(const problem *p, int b, int r)
{
    int64_t n = (int64_t)p->seq_lens[b] - p->q_len + r + 1;
    return n < 0 ? 0 : n;
}

/* Softmax attention of one (row, query head) over keys [t_begin, t_end) of its
 * sequence, clipped to the visible range.  Returns the normalised output o
 * (head_dim doubles), the maximum logit m and the sum l of exp(s_t - m).
 * An empty range gives o = 0, m = -inf, l = 0.  Scores are summed over d in
 * index order and the softmax sums run over t in logical token order.
 * scratch holds at least (t_end - t_begin) doubles. */
static int attend_range(const problem *p, int64_t row, int h, int64_t t_begin, int64_t t_end,
                        double *o, double *m_out, double *l_out, double *scratch)
{
    int D = p->head_dim;
    int b = (int)(row / p->q_len);
    int r = (int)(row % p->q_len);
    int group = p->num_q_heads / p->num_kv_heads;
    int kv_head = h / group;
    const int32_t *bt = p->block_table + (int64_t)b * p->max_pages_per_seq;
    const uint16_t *qv = p->q + (row * p->num_q_heads + h) * (int64_t)D;

    int64_t n = visible_keys(p, b, r);
    if (t_end > n)
        t_end = n;
    if (t_begin < 0)
        t_begin = 0;
    if (p->window > 0 && t_begin < n - p->window)
        t_begin = n - p->window; /* the sliding window's first key */
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (t_begin >= t_end) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return 0;
    }

    /* scores s_t = scale * sum_d q_d k_{t,d}   ([DCU-832] Sec.5) */
    double m = -INFINITY;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t off = row_offset(bt, t, p->block_size, p->num_kv_heads, D, kv_head, p->num_pages);
        if (off < 0)
            return -2;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_to_double(qv[d]) * kv_elem(p, 0, off + d, kv_head);
        double s = p->scale * dot;
        scratch[t - t_begin] = s;
        if (s > m)
            m = s;
    }
    /* max-subtracted exponentials, their sum, and the weighted sum of V rows */
    double l = 0.0;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t off = row_offset(bt, t, p->block_size, p->num_kv_heads, D, kv_head, p->num_pages);
        double w = exp(scratch[t - t_begin] - m);
        l += w;
        for (int d = 0; d < D; ++d)
            o[d] += w * kv_elem(p, 1, off + d, kv_head);
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
    return 0;
}

static int check_problem(const problem *p)
{
    if (!p->q || !p->block_table || !p->seq_lens)
        return -1;
    if (p->k_cache8 ? (!p->v_cache8 || !p->k_scale || !p->v_scale) : (!p->k_cache || !p->v_cache))
        return -1;
    if (p->num_seqs < 0 || p->q_len <= 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->head_dim <= 0 || p->block_size <= 0 || p->max_pages_per_seq < 0 || p->num_pages < 0)
        return -1;
    if (p->num_q_heads % p->num_kv_heads != 0)
        return -1;
    for (int b = 0; b < p->num_seqs; ++b) {
        int64_t L = p->seq_lens[b];
        if (L < 0 || (L + p->block_size - 1) / p->block_size > p->max_pages_per_seq)
            return -1;
    }
    return 0;
}

typedef struct {
    const problem *p;
    double *out;
    int64_t first_item, item_stride, num_items;
    int status;
} worker_arg;

static void *attention_worker(void *varg)
{
    worker_arg *a = (worker_arg *)varg;
    const problem *p = a->p;
    int64_t max_keys = 1;
    for (int b = 0; b < p->num_seqs; ++b)
        if (p->seq_lens[b] > max_keys)
            max_keys = p->seq_lens[b];
    double *scratch = (double *)malloc((size_t)max_keys * sizeof(double));
    if (!scratch) {
        a->status = -1;
        return NULL;
    }
    a->status = 0;
    for (int64_t item = a->first_item; item < a->num_items; item += a->item_stride) {
        int64_t row = item / p->num_q_heads;
        int h = (int)(item % p->num_q_heads);
        double m, l;
        double *o = a->out + item * p->head_dim; /* out[row, h, :] */
        int rc = attend_range(p, row, h, 0, INT64_MAX, o, &m, &l, scratch);
        if (rc != 0) {
            a->status = rc;
            break;
        }
    }
    free(scratch);
    return NULL;
}

/* ------------------------------------------------------------------------ */
/* Full paged attention: out[row, h, :] = sum_t softmax_t(scale q.K_t) V_t over
 * the keys the row may see.  Rows are ordered (sequence, new-row), i.e. row =
 * b * q_len + r.  q_len == 1 is plain decode; q_len > 1 is the verify variant.
 * Work is spread over num_threads POSIX threads by (row, head) item. */
int oracle_paged_attention_window(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int max_pages_per_seq,
                                  int64_t num_pages, double scale, int64_t window, double *out,
                                  int num_threads);

static int run_attention(const problem *p, double *out, int num_threads);

int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, int max_pages_per_seq,
                           int64_t num_pages, double scale, double *out, int num_threads)
{
    return oracle_paged_attention_window(q, k_cache, v_cache, block_table, seq_lens, num_seqs, q_len,
                                         num_q_heads, num_kv_heads, head_dim, block_size, max_pages_per_seq,
                                         num_pages, scale, 0, out, num_threads);
}

/* The same with a sliding window of W keys per row (W = 0: none). */
int oracle_paged_attention_window(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int max_pages_per_seq,
                                  int64_t num_pages, double scale, int64_t window, double *out,
                                  int num_threads)
{
    problem p = {q, k_cache, v_cache, block_table, seq_lens, num_seqs, q_len, num_q_heads,
                 num_kv_heads, head_dim, block_size, max_pages_per_seq, num_pages, scale, window,
                 NULL, NULL, NULL, NULL};
    return run_attention(&p, out, num_threads);
}

/* The same over an fp8 cache: e4m3 codes [num_pages, block_size,
 * num_kv_heads, head_dim] and one scale per KV head for K and for V. */
int oracle_paged_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_table, const int32_t *seq_lens,
                               int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int max_pages_per_seq,
                               int64_t num_pages, double scale, int64_t window, double *out,
                               int num_threads)
{
    problem p = {q, NULL, NULL, block_table, seq_lens, num_seqs, q_len, num_q_heads,
                 num_kv_heads, head_dim, block_size, max_pages_per_seq, num_pages, scale, window,
                 k_cache, v_cache, k_scale, v_scale};
    return run_attention(&p, out, num_threads);
}

static int run_attention(const problem *pp, double *out, int num_threads)
{
    const problem p = *pp;
    const int num_seqs = p.num_seqs, q_len = p.q_len, num_q_heads = p.num_q_heads;
    if (!out || check_problem(&p) != 0 || p.window < 0)
        return -1;
    if (num_threads < 1)
        num_threads = 1;
    int64_t num_items = (int64_t)num_seqs * q_len * num_q_heads;
    if (num_threads > num_items)
        num_threads = num_items > 0 ? (int)num_items : 1;

    pthread_t *tids = (pthread_t *)calloc((size_t)num_threads, sizeof(pthread_t));
    worker_arg *args = (worker_arg *)calloc((size_t)num_threads, sizeof(worker_arg));
    if (!tids || !args) {
        free(tids);
        free(args);
        return -1;
    }
    int rc = 0;
    for (int i = 0; i < num_threads; ++i) {
        args[i] = (worker_arg){&p, out, i, num_threads, num_items, 0};
        if (num_threads == 1)
            attention_worker(&args[i]);
        else if (pthread_create(&tids[i], NULL, attention_worker, &args[i]) != 0)
            rc = -1;
    }
    if (num_threads > 1)
        for (int i = 0; i < num_threads; ++i)
            pthread_join(tids[i], NULL);
    for (int i = 0; i < num_threads && rc == 0; ++i)
        rc = args[i].status;
    free(tids);
    free(args);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* One split of the method ([RADEON], split-KV fix): attention of one (row, head)
 * restricted to keys [t_begin, t_end).  Gives the split's normalised output
 * o (head_dim doubles), its max logit m and its exponential sum l. */
int oracle_attention_partial(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *block_table, const int32_t *seq_lens,
                             int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                             int head_dim, int block_size, int max_pages_per_seq,
                             int64_t num_pages, double scale, int64_t row, int head,
                             int64_t t_begin, int64_t t_end, double *o, double *m, double *l)
{
    problem p = {q, k_cache, v_cache, block_table, seq_lens, num_seqs, q_len, num_q_heads,
                 num_kv_heads, head_dim, block_size, max_pages_per_seq, num_pages, scale, 0,
                 NULL, NULL, NULL, NULL};
    if (!o || !m || !l || check_problem(&p) != 0)
        return -1;
    if (row < 0 || row >= (int64_t)num_seqs * q_len || head < 0 || head >= num_q_heads)
        return -1;
    int64_t span = t_end - t_begin;
    double *scratch = (double *)malloc((size_t)(span > 1 ? span : 1) * sizeof(double));
    if (!scratch)
        return -1;
    int rc = attend_range(&p, row, head, t_begin, t_end, o, m, l, scratch);
    free(scratch);
    return rc;
}

/* The reduce step of the split method: given n split results (o_i, m_i, l_i),
 * M = max_i m_i, w_i = l_i exp(m_i - M), out = sum_i w_i o_i / sum_i w_i.
 * Splits with l_i == 0 (no keys) carry no weight; if every split is empty the
 * output is zero. */
int oracle_lse_combine(const double *o_parts, const double *m_parts, const double *l_parts,
                       int n, int head_dim, double *out)
{
    if (n < 0 || head_dim <= 0 || !out)
        return -1;
    double M = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (l_parts[i] > 0.0 && m_parts[i] > M)
            M = m_parts[i];
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (M == -INFINITY)
        return 0;
    double wsum = 0.0;
    for (int i = 0; i < n; ++i) {
        if (l_parts[i] <= 0.0)
            continue;
        double w = l_parts[i] * exp(m_parts[i] - M);
        wsum += w;
        for (int d = 0; d < head_dim; ++d)
            out[d] += w * o_parts[(int64_t)i * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d)
        out[d] /= wsum;
    return 0;
}

/* Page length (tokens) for a hybrid model whose attention KV cache and
 * recurrent-state cache share one page granularity, as the "Why Qwen3.5's
 * Hybrid Cache Makes This Problem More Complex" section of the DCU page-832
 * article states it for the path without prefix caching: the state page,
 * measured in attention tokens, rounded up to a whole number of
 * alignment-token groups,
 *     page = ceil(state_page_bytes / (alignment * attn_bytes_per_token)) * alignment.
 * Returns -1 for non-positive arguments. */
int64_t oracle_hybrid_page_tokens(int64_t state_page_bytes, int64_t attn_bytes_per_token, int64_t alignment)
{
    if (state_page_bytes <= 0 || attn_bytes_per_token <= 0 || alignment <= 0)
        return -1;
    const int64_t group_bytes = alignment * attn_bytes_per_token;
    const int64_t groups = (state_page_bytes + group_bytes - 1) / group_bytes;
    return groups * alignment;
}
