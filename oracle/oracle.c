/*
 * Oracle for load-balanced paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant table with the CUDA
 * library: every number here is recomputed from the definitions below.
 *
 * What it computes (plain definitions, fp64, no blocking, no fusion):
 *
 *  - oracle_attention: decode attention of one new query token per request
 *    against the request's whole live KV cache.  "Decode attention over a
 *    request's full KV cache" is stated in the vLLM integration post
 *    ("The challenge: mixed-length decode in every batch") and in the SGLang
 *    post (section on load balancing for variable-length decode).  For request
 *    r and query head hq, with kv head h = floor(hq / G), G = Hq / Hkv:
 *        s_j   = sm_scale * sum_d q[r,hq,d] * k[r,j,h,d]      for j < L_r
 *        p     = softmax(s)   (max subtracted first)
 *        out_d = sum_j p_j * v[r,j,h,d]
 *    where k[r,j,h,:] = k_cache[block_table[r, j / page], j % page, h, :]
 *    (paged KV consumed in place, SGLang post, "From HPC-Ops kernel to
 *    SGLang"; page size 64 from its launch flags).  A request with L_r = 0
 *    yields a zero row.
 *  - oracle_partial: the same over a sub-range [j0, j1) of the live tokens,
 *    returning the normalised partial output and its natural-log
 *    log-sum-exp, as the persistent kernel's per-descriptor result is
 *    described in the vLLM post ("Compute and combine").
 *  - oracle_combine: merge of partials under the global softmax
 *    normalisation (SGLang post, execution paragraph of the live-KV
 *    scheduling section; vLLM post, "Compute and combine").
 *  - oracle_attention_mq: decode with q_len new query tokens per request
 *    (the speculative / MTP layer of Hy3, vLLM post "A Quick Word on
 *    Hy3-series models"): the request's last q_len live tokens are the
 *    queries, q is [B, q_len, Hq, D], and query token i sees the live tokens
 *    j < L_r - q_len + 1 + i (everything before it and itself), the plain
 *    causal reading.  Query rows with no visible token yield zero rows.
 *
 * Inputs are raw storage words: bf16 as uint16 bit patterns, FP8-E4M3 as
 * bytes.  Both are decoded here from their bit-level format definitions
 * (bf16 = upper half of an IEEE binary32; E4M3 = 1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits, subnormals m/8 * 2^-6, no infinities,
 * S.1111.111 = NaN, largest finite 448).  FP8 values are dequantised before
 * use: k = e4m3(k8) * k_scale, v = e4m3(v8) * v_scale,
 * q = e4m3(q8) * q_scale[r, hq].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes for the storage words this file reads */
#define ORACLE_BF16 0
#define ORACLE_E4M3 1

double oracle_bf16_to_double(uint16_t bits) {
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exponent = (code >> 3) & 0xF;
    int mantissa = code & 0x7;
    double mag;
    if (exponent == 0xF && mantissa == 0x7) return NAN;
    if (exponent == 0)
        mag = ldexp((double)mantissa / 8.0, 1 - 7); /* subnormal */
    else
        mag = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
    return sign ? -mag : mag;
}

/* Element (index i) of a storage array of the given dtype, as a double. */
static double load_elem(const void *base, int dtype, size_t i) {
    if (dtype == ORACLE_E4M3) return oracle_e4m3_to_double(((const uint8_t *)base)[i]);
    return oracle_bf16_to_double(((const uint16_t *)base)[i]);
}

typedef struct {
    const void *q;
    int q_dtype;
    const float *q_scale; /* [B, Hq], used when q_dtype is E4M3 */
    const void *k_cache;  /* [num_pages, page, Hkv, D] */
    const void *v_cache;
    int kv_dtype;
    double k_scale, v_scale;
    const int32_t *block_table; /* [B, max_pages] */
    int max_pages;
    const int32_t *seqlens; /* [B] */
    int B, Hq, Hkv, D, page;
    double sm_scale;
    int q_len; /* query tokens per request (1: plain decode) */
} oracle_problem;

/* Dequantised query qi = i * Hq + hq of request r (q is [B, q_len, Hq, D]) into qv[D]. */
static void load_query(const oracle_problem *p, int r, int qi, double *qv) {
    size_t row = (size_t)r * p->q_len * p->Hq + qi;
    double scale = 1.0;
    if (p->q_dtype == ORACLE_E4M3) scale = (double)p->q_scale[row];
    for (int d = 0; d < p->D; ++d) qv[d] = load_elem(p->q, p->q_dtype, row * p->D + d) * scale;
}

/* Offset of k[r, j, h, 0] inside a cache, through the block table. */
static size_t kv_offset(const oracle_problem *p, int r, int j, int h) {
    int page_id = p->block_table[(size_t)r * p->max_pages + j / p->page];
    int slot = j % p->page;
    return (((size_t)page_id * p->page + slot) * p->Hkv + h) * p->D;
}

/*
 * Attention of query qi = i * Hq + hq of request r over live tokens
 * [j0, j1).  Writes the normalised output o[D] and returns the natural-log
 * log-sum-exp of the scaled scores; an empty range gives o = 0 and returns
 * -INFINITY.  s and qv are caller scratch of sizes (j1 - j0) and D.
 */
static double attend_range(const oracle_problem *p, int r, int qi, int j0, int j1, double *o,
                           double *s, double *qv) {
    int G = p->Hq / p->Hkv;
    int h = (qi % p->Hq) / G;
    for (int d = 0; d < p->D; ++d) o[d] = 0.0;
    if (j1 <= j0) return -INFINITY;
    load_query(p, r, qi, qv);
    double kscale = p->kv_dtype == ORACLE_E4M3 ? p->k_scale : 1.0;
    double vscale = p->kv_dtype == ORACLE_E4M3 ? p->v_scale : 1.0;
    double smax = -INFINITY;
    for (int j = j0; j < j1; ++j) {
        size_t off = kv_offset(p, r, j, h);
        double dot = 0.0;
        for (int d = 0; d < p->D; ++d) dot += qv[d] * (load_elem(p->k_cache, p->kv_dtype, off + d) * kscale);
        s[j - j0] = p->sm_scale * dot;
        if (s[j - j0] > smax) smax = s[j - j0];
    }
    double denom = 0.0;
    for (int j = j0; j < j1; ++j) {
        double w = exp(s[j - j0] - smax);
        size_t off = kv_offset(p, r, j, h);
        for (int d = 0; d < p->D; ++d) o[d] += w * (load_elem(p->v_cache, p->kv_dtype, off + d) * vscale);
        denom += w;
    }
    for (int d = 0; d < p->D; ++d) o[d] /= denom;
    return smax + log(denom);
}

static int max_seqlen(const oracle_problem *p) {
    int m = 0;
    for (int r = 0; r < p->B; ++r)
        if (p->seqlens[r] > m) m = p->seqlens[r];
    return m;
}

/*
 * Unsplit decode attention for the listed query rows (row = r * Hq + hq;
 * rows == NULL means every row in order).  out is [n_rows, D] fp64.
 * Returns 0, or -1 when a scratch allocation fails.
 */
int oracle_attention(const void *q, int q_dtype, const float *q_scale, const void *k_cache,
                     const void *v_cache, int kv_dtype, double k_scale, double v_scale,
                     const int32_t *block_table, int max_pages, const int32_t *seqlens, int B, int Hq,
                     int Hkv, int D, int page, double sm_scale, const int64_t *rows, int64_t n_rows,
                     double *out, int num_threads) {
    oracle_problem p = {q, q_dtype, q_scale, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                        block_table, max_pages, seqlens, B, Hq, Hkv, D, page, sm_scale, 1};
    int64_t total = rows ? n_rows : (int64_t)B * Hq;
    int lmax = max_seqlen(&p);
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qv) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < total; ++i) {
                int64_t row = rows ? rows[i] : i;
                int r = (int)(row / Hq), hq = (int)(row % Hq);
                attend_range(&p, r, hq, 0, seqlens[r], out + i * D, s, qv);
            }
        }
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

/*
 * Partial attention of query (r, hq) over live tokens [j0, j1): normalised
 * partial output o[D] and natural-log LSE (returned through *lse).
 */
int oracle_partial(const void *q, int q_dtype, const float *q_scale, const void *k_cache,
                   const void *v_cache, int kv_dtype, double k_scale, double v_scale,
                   const int32_t *block_table, int max_pages, const int32_t *seqlens, int B, int Hq,
                   int Hkv, int D, int page, double sm_scale, int r, int hq, int j0, int j1, double *o,
                   double *lse) {
    oracle_problem p = {q, q_dtype, q_scale, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                        block_table, max_pages, seqlens, B, Hq, Hkv, D, page, sm_scale, 1};
    int n = j1 > j0 ? j1 - j0 : 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !qv) {
        free(s);
        free(qv);
        return -1;
    }
    *lse = attend_range(&p, r, hq, j0, j1, o, s, qv);
    free(s);
    free(qv);
    return 0;
}

/*
 * Multi-query decode attention for the listed rows (row = (r * q_len + i) *
 * Hq + hq; rows == NULL means every row in order).  Query token i of
 * request r attends live tokens [0, L_r - q_len + 1 + i).  out is
 * [n_rows, D] fp64.  Returns 0, or -1 when a scratch allocation fails.
 */
int oracle_attention_mq(const void *q, int q_dtype, const float *q_scale, const void *k_cache,
                        const void *v_cache, int kv_dtype, double k_scale, double v_scale,
                        const int32_t *block_table, int max_pages, const int32_t *seqlens, int B,
                        int Hq, int Hkv, int D, int page, double sm_scale, int q_len,
                        const int64_t *rows, int64_t n_rows, double *out, int num_threads) {
    oracle_problem p = {q, q_dtype, q_scale, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                        block_table, max_pages, seqlens, B, Hq, Hkv, D, page, sm_scale, q_len};
    int64_t per_req = (int64_t)q_len * Hq;
    int64_t total = rows ? n_rows : (int64_t)B * per_req;
    int lmax = max_seqlen(&p);
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qv) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t n = 0; n < total; ++n) {
                int64_t row = rows ? rows[n] : n;
                int r = (int)(row / per_req), qi = (int)(row % per_req);
                int i = qi / Hq;
                int visible = seqlens[r] - q_len + 1 + i;
                attend_range(&p, r, qi, 0, visible, out + n * D, s, qv);
            }
        }
        free(s);
        free(qv);
    }
    return failed ? -1 : 0;
}

/*
 * Merge n partials (o_i normalised over their own ranges, lse_i natural
 * log) into the output over the union of the ranges:
 *     M = max_i lse_i,  w_i = exp(lse_i - M),  out = sum_i w_i o_i / sum_i w_i.
 * Partials with lse = -inf carry no tokens and get weight 0; with none
 * left the output is zero.
 */
void oracle_combine(const double *parts, const double *lses, int n, int D, double *out) {
    double m = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (lses[i] > m) m = lses[i];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (m == -INFINITY) return;
    double wsum = 0.0;
    for (int i = 0; i < n; ++i) {
        if (lses[i] == -INFINITY) continue;
        double w = exp(lses[i] - m);
        wsum += w;
        for (int d = 0; d < D; ++d) out[d] += w * parts[(size_t)i * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= wsum;
}
