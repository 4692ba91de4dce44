/*
 * ua_oracle.c -- plain fp64 CPU oracle for the forward pass of unified paged,
 * variable-length attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker that the CUDA
 * path is compared against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  It shares no code, header, table
 * or helper with the CUDA library and includes nothing from it.
 *
 * What it computes (gfx950 "Unified paged attention on gfx950, from the math
 * up", section 1 "What unified attention computes"): for one query row i of one
 * (sequence, query head h) and the key positions j = 0 .. S_k-1 of that
 * sequence,
 *
 *   x_j   = tau * <Q_i, K_j>                                   (step 1, scale)
 *   x_j   = c * tanh(x_j / c)              if SOFTCAP          (step 2)
 *   x_j  += slope_h * (j - ctx)            if ALIBI            (step 3)
 *   x_j  += bias[i][j - ctx]  for j >= ctx  if QQ-BIAS          (step 4)
 *   j visible iff (not CAUSAL or j <= i + ctx)                 (step 5)
 *             and (not WINDOW or j >= i + ctx - W + 1)         (step 6)
 *   den   = sum_{j visible} e^{x_j}  (+ e^{sink_h} if SINKS)   (step 7)
 *   O_i   = sum_{j visible} e^{x_j} V_j / den
 *
 * with ctx = S_k - S_q (the query chunk is the last S_q of the S_k keys), the
 * GQA head map h_k = floor(h / g), g = H_q / H_k, and the paged lookup
 * K_j = k_cache[block_table[s][j / b]][j mod b][h_k][:] (section 0, notation,
 * and the serving layout described below it).  The window keeps the W keys
 * i+ctx-W+1 .. i+ctx, the convention the dense prefill kernel's spec states
 * (attention_dense.py, AttentionDenseSpec.sliding_window docstring).  An empty
 * denominator gives O_i = 0 (gfx1151 ALGORITHM.md section 6, the l = 0 guard).
 *
 * The exponentials are taken after subtracting the largest visible logit
 * (gfx1151 ALGORITHM.md section 2: softmax is invariant to a common shift);
 * this changes no value, it only keeps e^x finite in fp64.  There is no
 * tiling, no online recurrence, no base-2 domain and no lazy rescale here:
 * every row is the definition evaluated directly over all of its keys.
 *
 * bf16 inputs are widened exactly (a bf16 value is the upper half of an
 * IEEE-754 binary32), and every product and sum is fp64.
 *
 * The QQ-bias (step 4, "inside the query section") is one fp64 matrix shared by
 * every sequence and head, indexed by the local query index i and the key's
 * offset j - ctx inside the chunk; keys before the chunk (j < ctx) get none.
 *
 * Sparse top-k mode ("[Triton/Gluon] [GFX950] Sparse paged attention and
 * Sparse MLA", the token-granular top-k gather of its sparse decode): each
 * query token t carries its own list of key positions topk_idx[t][0 .. n_t-1]
 * (n_t = topk_len[t]) into its sequence's paged cache, and the row attends to
 * the listed keys instead of to all S_k of them: the sum above runs over the
 * list entries e with j = topk_idx[t][e], every entry with the same score
 * chain and masks as key j.  Entries outside [0, S_k) are padding (not keys).
 * An entry listed twice counts twice (a plain sum over the list).
 *
 * fp8 KV cache (gfx950 page, section 7.3 "fp8 KV cache (bf16-Q + fp8-KV)"):
 * the cache holds e4m3 codes with one scale per tensor, K_j = e4m3(k) * k_scale
 * and V_j = e4m3(v) * v_scale, decoded exactly (OCP 8-bit float e4m3: 1 sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent 0, the
 * all-ones code NaN, no infinities); Q stays bf16.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1       /* malformed arguments */
#define ORACLE_ERR_CTX -2       /* seqused_k < S_q for some sequence */
#define ORACLE_ERR_BLOCK -3     /* block id outside [0, num_blocks) */
#define ORACLE_ERR_CU -4        /* cu_seqlens_q not non-decreasing */
#define ORACLE_ERR_NOMEM -5

typedef struct {
    int32_t num_seqs, hq, hk, d, b;
    int64_t num_blocks;
    const uint16_t *q;              /* bf16 bit patterns */
    const void *k, *v;              /* bf16 bit patterns, or e4m3 codes when kv_fp8 */
    int32_t kv_fp8;
    double k_scale, v_scale;        /* applied to decoded e4m3 values */
    const int32_t *block_table;     /* [num_seqs, bt_stride] */
    int32_t bt_stride;
    const int32_t *cu_seqlens_q;    /* [num_seqs + 1] */
    const int32_t *seqused_k;       /* [num_seqs] */
    double scale;
    int32_t causal;
    double softcap;                 /* 0 = off */
    int32_t window;                 /* 0 = off */
    const double *alibi_slopes;     /* [hq] or NULL */
    const double *sinks;            /* [hq] or NULL */
    const double *qq_bias;          /* [>= S_q][qq_stride] or NULL */
    int64_t qq_stride;
    const int32_t *topk_idx;        /* [total_q][topk_stride] key positions, or NULL */
    const int32_t *topk_len;        /* [total_q] list lengths (with topk_idx) */
    int64_t topk_stride;
} oracle_problem;

static double widen_bf16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Value of an OCP e4m3 code: (-1)^s (1 + m/8) 2^(e-7), or m/8 2^-6 when e = 0;
 * exponent 15 with mantissa 7 is NaN. */
static double decode_e4m3(uint8_t x)
{
    const int s = x >> 7, e = (x >> 3) & 15, m = x & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* Element `idx` of a K or V cache, widened exactly (fp8: times its scale). */
static double kv_elem(const oracle_problem *P, const void *base, int64_t idx, double scale)
{
    if (P->kv_fp8) return decode_e4m3(((const uint8_t *)base)[idx]) * scale;
    return widen_bf16(((const uint16_t *)base)[idx]);
}

/* Sequence that owns packed query row `token` (cu_seqlens_q is non-decreasing). */
static int32_t owner_seq(const oracle_problem *P, int64_t token)
{
    int32_t lo = 0, hi = P->num_seqs - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if ((int64_t)P->cu_seqlens_q[mid] <= token) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static int validate(const oracle_problem *P)
{
    if (P->num_seqs < 0 || P->hq <= 0 || P->hk <= 0 || P->d <= 0 || P->b <= 0)
        return ORACLE_ERR_ARG;
    if (P->hq % P->hk != 0) return ORACLE_ERR_ARG;
    if (P->window < 0 || P->softcap < 0.0) return ORACLE_ERR_ARG;
    if (P->window > 0 && !P->causal) return ORACLE_ERR_ARG;
    if (P->cu_seqlens_q[0] != 0) return ORACLE_ERR_CU;
    if (P->topk_idx) {
        if (!P->topk_len || P->topk_stride < 1) return ORACLE_ERR_ARG;
        const int64_t total_q = P->num_seqs > 0 ? P->cu_seqlens_q[P->num_seqs] : 0;
        for (int64_t t = 0; t < total_q; ++t)
            if (P->topk_len[t] < 0 || P->topk_len[t] > P->topk_stride) return ORACLE_ERR_ARG;
    }
    for (int32_t s = 0; s < P->num_seqs; ++s) {
        int32_t sq = P->cu_seqlens_q[s + 1] - P->cu_seqlens_q[s];
        int32_t sk = P->seqused_k[s];
        if (sq < 0) return ORACLE_ERR_CU;
        if (sk < sq) return ORACLE_ERR_CTX;
        int32_t nblk = (sk + P->b - 1) / P->b;
        if (nblk > P->bt_stride) return ORACLE_ERR_ARG;
        for (int32_t n = 0; n < nblk; ++n) {
            int32_t id = P->block_table[(int64_t)s * P->bt_stride + n];
            if (id < 0 || (int64_t)id >= P->num_blocks) return ORACLE_ERR_BLOCK;
        }
    }
    return ORACLE_OK;
}

/* Number of keys row `token` ranges over: S_k, or its list length. */
static int64_t row_keys(const oracle_problem *P, int64_t token, int32_t sk)
{
    return P->topk_idx ? P->topk_len[token] : sk;
}

/* Key position of the row's e-th key: e itself, or the e-th list entry. */
static int64_t key_at(const oracle_problem *P, int64_t token, int64_t e)
{
    return P->topk_idx ? P->topk_idx[token * P->topk_stride + e] : e;
}

/*
 * One output row.  `x` and `vis` are caller scratch of length >= the row's
 * key count n (S_k, or its top-k list length).  If `weights` is non-NULL it
 * receives the n softmax weights followed by the sink's weight (0 when SINKS
 * is off); masked keys get weight 0.
 */
static void one_row(const oracle_problem *P, int64_t token, int32_t h, double *out,
                    double *weights, double *x, unsigned char *vis)
{
    const int32_t s = owner_seq(P, token);
    const int32_t sq = P->cu_seqlens_q[s + 1] - P->cu_seqlens_q[s];
    const int32_t sk = P->seqused_k[s];
    const int64_t ctx = (int64_t)sk - sq;
    const int64_t i = token - P->cu_seqlens_q[s];
    const int32_t g = P->hq / P->hk;
    const int32_t hkv = h / g;
    const int32_t d = P->d;
    const uint16_t *qrow = P->q + (token * P->hq + h) * (int64_t)d;

    const int64_t n = row_keys(P, token, sk);
    double m = -INFINITY;
    for (int64_t e = 0; e < n; ++e) {
        const int64_t j = key_at(P, token, e);
        int visible = j >= 0 && j < sk;
        if (P->causal && j > i + ctx) visible = 0;
        if (P->window > 0 && j < i + ctx - P->window + 1) visible = 0;
        vis[e] = (unsigned char)visible;
        if (!visible) { x[e] = -INFINITY; continue; }
        int64_t blk = P->block_table[(int64_t)s * P->bt_stride + j / P->b];
        const int64_t krow = ((blk * P->b + j % P->b) * P->hk + hkv) * (int64_t)d;
        double dot = 0.0;
        for (int32_t t = 0; t < d; ++t) dot += widen_bf16(qrow[t]) * kv_elem(P, P->k, krow + t, P->k_scale);
        double xj = P->scale * dot;
        if (P->softcap > 0.0) xj = P->softcap * tanh(xj / P->softcap);
        if (P->alibi_slopes) xj += P->alibi_slopes[h] * (double)(j - ctx);
        if (P->qq_bias && j >= ctx) xj += P->qq_bias[i * P->qq_stride + (j - ctx)];
        x[e] = xj;
        if (xj > m) m = xj;
    }
    const int have_sink = P->sinks != NULL;
    const double sink = have_sink ? P->sinks[h] : -INFINITY;
    if (have_sink && sink > m) m = sink;

    for (int32_t t = 0; t < d; ++t) out[t] = 0.0;
    if (weights)
        for (int64_t e = 0; e <= n; ++e) weights[e] = 0.0;

    if (m == INFINITY) {
        /* A +inf sink takes all of the probability mass and has no value row. */
        if (weights) weights[n] = 1.0;
        return;
    }
    if (m == -INFINITY) return; /* nothing visible, no sink: den = 0, O = 0 */

    double den = 0.0;
    for (int64_t e = 0; e < n; ++e) {
        if (!vis[e]) continue;
        x[e] = exp(x[e] - m);
        den += x[e];
    }
    double e_sink = have_sink ? exp(sink - m) : 0.0;
    den += e_sink;
    if (!(den > 0.0)) return;

    for (int64_t e = 0; e < n; ++e) {
        if (!vis[e]) continue;
        const int64_t j = key_at(P, token, e);
        int64_t blk = P->block_table[(int64_t)s * P->bt_stride + j / P->b];
        const int64_t vrow = ((blk * P->b + j % P->b) * P->hk + hkv) * (int64_t)d;
        double wgt = x[e];
        for (int32_t t = 0; t < d; ++t) out[t] += wgt * kv_elem(P, P->v, vrow + t, P->v_scale);
        if (weights) weights[e] = x[e] / den;
    }
    for (int32_t t = 0; t < d; ++t) out[t] /= den;
    if (weights) weights[n] = e_sink / den;
}

typedef struct {
    const oracle_problem *P;
    const int64_t *rows;   /* row id = token * hq + head, or NULL for all rows */
    int64_t n_rows;
    double *out;           /* [n_rows, d] */
    int32_t max_sk;
    int64_t next;          /* shared work counter */
    pthread_mutex_t lock;
    int failed;
} job_t;

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *x = (double *)malloc(sizeof(double) * (size_t)(J->max_sk + 1));
    unsigned char *vis = (unsigned char *)malloc((size_t)J->max_sk + 1);
    if (!x || !vis) {
        pthread_mutex_lock(&J->lock); J->failed = 1; pthread_mutex_unlock(&J->lock);
        free(x); free(vis);
        return NULL;
    }
    const int64_t chunk = 16;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t begin = J->next;
        J->next += chunk;
        pthread_mutex_unlock(&J->lock);
        if (begin >= J->n_rows) break;
        int64_t end = begin + chunk < J->n_rows ? begin + chunk : J->n_rows;
        for (int64_t r = begin; r < end; ++r) {
            int64_t id = J->rows ? J->rows[r] : r;
            one_row(J->P, id / J->P->hq, (int32_t)(id % J->P->hq),
                    J->out + r * (int64_t)J->P->d, NULL, x, vis);
        }
    }
    free(x); free(vis);
    return NULL;
}

static int run_rows(const oracle_problem *P, const int64_t *rows, int64_t n_rows,
                    double *out, int32_t nthreads)
{
    int rc = validate(P);
    if (rc != ORACLE_OK) return rc;
    int64_t total_q = P->cu_seqlens_q[P->num_seqs];
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_q * P->hq) return ORACLE_ERR_ARG;
    }
    int32_t max_sk = 0;
    for (int32_t s = 0; s < P->num_seqs; ++s)
        if (P->seqused_k[s] > max_sk) max_sk = P->seqused_k[s];
    if (P->topk_idx && P->topk_stride > max_sk) {
        if (P->topk_stride > INT32_MAX - 1) return ORACLE_ERR_ARG;
        max_sk = (int32_t)P->topk_stride;
    }

    job_t J;
    J.P = P; J.rows = rows; J.n_rows = n_rows; J.out = out; J.max_sk = max_sk;
    J.next = 0; J.failed = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) { pthread_mutex_destroy(&J.lock); return ORACLE_ERR_NOMEM; }
    int32_t started = 0;
    for (int32_t t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int32_t t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Exported entry points.  Argument meaning mirrors the library's forward call:
 * q [total_q, hq, d], k_cache / v_cache [num_blocks, b, hk, d] (bf16 bits),
 * block_table [num_seqs, bt_stride], cu_seqlens_q [num_seqs + 1],
 * seqused_k [num_seqs]; softcap <= 0 and window <= 0 switch those terms off;
 * alibi_slopes / sinks may be NULL; kv_fp8 != 0 reads the caches as e4m3
 * codes scaled by k_scale / v_scale; qq_bias (or NULL) is the query-section
 * bias, row i at qq_bias + i * qq_stride; topk_idx (or NULL) switches to the
 * sparse top-k mode: token t's list at topk_idx + t * topk_stride, of
 * topk_len[t] <= topk_stride entries.  Output is fp64.
 * ------------------------------------------------------------------------- */

#define FILL_PROBLEM()                                                        \
    oracle_problem P;                                                         \
    P.num_seqs = num_seqs; P.hq = hq; P.hk = hk; P.d = d; P.b = b;            \
    P.num_blocks = num_blocks; P.q = q; P.k = k_cache; P.v = v_cache;         \
    P.block_table = block_table; P.bt_stride = bt_stride;                     \
    P.cu_seqlens_q = cu_seqlens_q; P.seqused_k = seqused_k;                   \
    P.scale = scale; P.causal = causal;                                       \
    P.softcap = softcap > 0.0 ? softcap : 0.0;                                \
    P.window = window > 0 ? window : 0;                                       \
    P.alibi_slopes = alibi_slopes; P.sinks = sinks;                           \
    P.kv_fp8 = kv_fp8 ? 1 : 0; P.k_scale = k_scale; P.v_scale = v_scale;      \
    P.qq_bias = qq_bias; P.qq_stride = qq_stride;                             \
    P.topk_idx = topk_idx; P.topk_len = topk_len; P.topk_stride = topk_stride;

#define PROBLEM_ARGS                                                          \
    int32_t num_seqs, int32_t hq, int32_t hk, int32_t d, int32_t b,          \
    int64_t num_blocks, const uint16_t *q, const void *k_cache,              \
    const void *v_cache, const int32_t *block_table, int32_t bt_stride,      \
    const int32_t *cu_seqlens_q, const int32_t *seqused_k, double scale,     \
    int32_t causal, double softcap, int32_t window,                          \
    const double *alibi_slopes, const double *sinks, int32_t kv_fp8,         \
    double k_scale, double v_scale, const double *qq_bias, int64_t qq_stride,   \
    const int32_t *topk_idx, const int32_t *topk_len, int64_t topk_stride

/* Every output row: out [total_q, hq, d]. */
int ua_oracle_forward(PROBLEM_ARGS, double *out, int32_t nthreads)
{
    FILL_PROBLEM();
    if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out)
        return ORACLE_ERR_ARG;
    int64_t total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
    return run_rows(&P, NULL, total_q * hq, out, nthreads);
}

/* Selected rows only: row id = token * hq + head; out [n_rows, d]. */
int ua_oracle_rows(PROBLEM_ARGS, const int64_t *rows, int64_t n_rows, double *out,
                   int32_t nthreads)
{
    FILL_PROBLEM();
    if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seqused_k || !out || !rows)
        return ORACLE_ERR_ARG;
    return run_rows(&P, rows, n_rows, out, nthreads);
}

/*
 * Softmax weights of one row: weights [n + 1] for its n keys (S_k, or its
 * top-k list length), the last entry being the sink's share (0 when SINKS is
 * off).  out_row [d] receives O_i.
 */
int ua_oracle_row_weights(PROBLEM_ARGS, int64_t token, int32_t head, double *weights,
                          double *out_row)
{
    FILL_PROBLEM();
    int rc = validate(&P);
    if (rc != ORACLE_OK) return rc;
    if (!weights || !out_row) return ORACLE_ERR_ARG;
    int64_t total_q = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
    if (token < 0 || token >= total_q || head < 0 || head >= hq) return ORACLE_ERR_ARG;
    int32_t sk = seqused_k[owner_seq(&P, token)];
    const int64_t n = row_keys(&P, token, sk);
    double *x = (double *)malloc(sizeof(double) * (size_t)(n + 1));
    unsigned char *vis = (unsigned char *)malloc((size_t)n + 1);
    if (!x || !vis) { free(x); free(vis); return ORACLE_ERR_NOMEM; }
    one_row(&P, token, head, out_row, weights, x, vis);
    free(x); free(vis);
    return ORACLE_OK;
}

/* The value of one e4m3 code (exposed for the tests that pin the decoder). */
double ua_oracle_e4m3(uint32_t code)
{
    return decode_e4m3((uint8_t)(code & 0xffu));
}
