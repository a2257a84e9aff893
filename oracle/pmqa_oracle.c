/*
 * pmqa_oracle.c -- plain CPU oracle for the FP8 paged MQA-logits indexer and
 * its per-row top-k.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. It shares no code, header, table or
 * helper with the CUDA library: every step below is written out again here
 * from the definitions it cites.
 *
 * Sources (page titles and sections):
 *   [P1] "[Bug] aiter ops triton attention pa" (stepcodex.com issue mirror),
 *        section "Minimal reproduction": the reference function `torch_ref`
 *        (the definition of the logits) and the `test` driver (input layout,
 *        the -inf clean-up and the top-k with k = min(2048, ctx)).
 *   [P3] "[Bugfix][Hardware][AMD] Fix last_page_len calculation in AITER MLA
 *        decode" (vLLM PR 31282), sections "The Bug" / "Comparison with Other
 *        Backends": how many tokens a request's last page holds.
 *   [OFP8] the OCP 8-bit floating point specification, E4M3 format, which the
 *        pages name as torch.float8_e4m3fn.
 *
 * What is computed (for request i, draft row j, logical token t):
 *   valid(i,j,t)  <=>  t < ctx_i  and  t <= ctx_i - next_n + j          [P1]
 *   phys          =   block_tables[i][t / P] * P + t % P                [P1]
 *   k_t[d]        =   e4m3fn(kv[phys][d]),  d < 128                     [P1, OFP8]
 *   s_t           =   fp32 from kv[phys][128..131], little-endian        [P1]
 *   x_h           =   s_t * sum_d q[i][j][h][d] * k_t[d]
 *   logit         =   sum_h w[i*next_n+j][h] * relu(x_h)               [P1]
 *   logit         =   -inf where not valid, up to max_model_len          [P1]
 * The sum over d is exact in double precision (every e4m3 value is a multiple
 * of 2^-9, so a product is a multiple of 2^-18 and |sum| < 2^25 needs fewer
 * than 53 significant bits). The head sum runs in double in head order and is
 * rounded once to fp32 (round to nearest even).
 * The per-entry tolerance 1e-3 * (1 + sum_h |w_h| * |x_h|) is returned beside
 * each logit.
 *
 * Top-k [P1]: per row, the entries t < valid_len sorted by (value descending,
 * index ascending); the first min(k, valid_len) indices, the rest -1.
 *
 * The last section of this file is the oracle of the sparse MLA decode that
 * consumes the top-k positions; its sources and readings are listed there.
 *
 * Readings where the pages leave a step open: the reference function names a
 * "bf16 reference" but computes in fp32; here the arithmetic is the exact real
 * one (double). NaN inputs propagate as they do under IEEE rules (relu keeps a
 * NaN); the inputs this oracle is run on are finite.
 *
 * Build: gcc -O2 -fPIC -shared -pthread pmqa_oracle.c -o libpmqa_oracle.so -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PMQA_REF_HEAD_DIM 128
#define PMQA_REF_ROW_BYTES 132

/* ---- fp8 e4m3fn, from the OFP8 definition --------------------------------
 * bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * exponent 0: subnormal, value m * 2^-9.  S.1111.111 is NaN; no infinities. */
static double e4m3fn_from_bits(unsigned b)
{
    unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

void pmqa_ref_e4m3fn_table(double out[256])
{
    for (unsigned b = 0; b < 256u; ++b)
        out[b] = e4m3fn_from_bits(b);
}

/* fp32 whose little-endian bytes are p[0..3], independent of host byte order. */
static float f32_from_le_bytes(const uint8_t *p)
{
    uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                 ((uint32_t)p[3] << 24);
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double relu(double x)
{
    if (x != x)
        return x; /* NaN stays NaN */
    return x > 0.0 ? x : 0.0;
}

/* ---- logits ---------------------------------------------------------------- */

typedef struct {
    const uint8_t *q, *kv;
    const float *w;
    const int32_t *ctx, *bt;
    int bs, next_n, heads, P, width;
    int64_t num_blocks, mml;
    float *out;
    double *out64, *tol;
    double table[256];
    /* work split: item = (request, token chunk) */
    int64_t chunk;
    int64_t *item_req, *item_t0;
    int64_t n_items;
    int next_item;
    pthread_mutex_t lock;
    int error;
} logits_job;

static void logits_request_range(logits_job *J, int i, int64_t t0, int64_t t1,
                                 double *qd, double *kd)
{
    const int H = J->heads, nn = J->next_n;
    const int64_t c = J->ctx[i];
    /* decoded q of this request: [next_n][heads][128] */
    for (int j = 0; j < nn; ++j)
        for (int h = 0; h < H; ++h)
            for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
                qd[((int64_t)j * H + h) * PMQA_REF_HEAD_DIM + d] =
                    J->table[J->q[(((int64_t)i * nn + j) * H + h) * PMQA_REF_HEAD_DIM + d]];
    for (int64_t t = t0; t < t1; ++t) {
        int64_t blk = t / J->P, off = t % J->P;
        int32_t b = J->bt[(int64_t)i * J->width + blk];
        if (b < 0 || (int64_t)b >= J->num_blocks) {
            J->error = 1;
            return;
        }
        const uint8_t *row = J->kv + ((int64_t)b * J->P + off) * PMQA_REF_ROW_BYTES;
        for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
            kd[d] = J->table[row[d]];
        const double s = (double)f32_from_le_bytes(row + PMQA_REF_HEAD_DIM);
        for (int j = 0; j < nn; ++j) {
            if (t > c - nn + j)
                continue; /* causal mask: stays -inf */
            const int64_t r = (int64_t)i * nn + j;
            const float *w = J->w + r * H;
            double sum = 0.0, mag = 0.0;
            for (int h = 0; h < H; ++h) {
                const double *qh = qd + ((int64_t)j * H + h) * PMQA_REF_HEAD_DIM;
                double dot = 0.0;
                for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
                    dot += qh[d] * kd[d];
                const double x = dot * s;
                sum += (double)w[h] * relu(x);
                mag += fabs((double)w[h]) * fabs(x);
            }
            const int64_t o = r * J->mml + t;
            J->out[o] = (float)sum;
            if (J->out64)
                J->out64[o] = sum;
            if (J->tol)
                J->tol[o] = 1e-3 * (1.0 + mag);
        }
    }
}

static void *logits_worker(void *arg)
{
    logits_job *J = (logits_job *)arg;
    double *qd = (double *)malloc(sizeof(double) * (size_t)J->next_n * (size_t)J->heads *
                                  PMQA_REF_HEAD_DIM);
    double kd[PMQA_REF_HEAD_DIM];
    if (!qd) {
        J->error = 2;
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t it = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (it >= J->n_items || J->error)
            break;
        int i = (int)J->item_req[it];
        int64_t t0 = J->item_t0[it];
        int64_t t1 = t0 + J->chunk;
        if (t1 > J->ctx[i])
            t1 = J->ctx[i];
        logits_request_range(J, i, t0, t1, qd, kd);
    }
    free(qd);
    return NULL;
}

/*
 * q            [bs, next_n, heads, 128] e4m3fn bytes
 * kv           [num_blocks, block_size, 132] bytes
 * weights      [bs*next_n, heads] fp32
 * context_lens [bs]; block_tables [bs, width]
 * out          [bs*next_n, max_model_len] fp32 (written entirely)
 * out64, tol   same shape in double, or NULL
 * Returns 0, or -1 for bad sizes, -2 for a context longer than max_model_len
 * or than the table covers, -3 for a table entry outside the pool, -4 when out
 * of memory.
 */
int pmqa_ref_logits(const uint8_t *q, const uint8_t *kv, const float *weights,
                    const int32_t *context_lens, const int32_t *block_tables, int bs,
                    int next_n, int heads, int head_dim, int block_size, int64_t num_blocks,
                    int width, int64_t max_model_len, float *out, double *out64, double *tol,
                    int nthreads)
{
    if (bs < 0 || next_n < 1 || heads < 1 || head_dim != PMQA_REF_HEAD_DIM || block_size < 1 ||
        num_blocks < 0 || width < 0 || max_model_len < 0)
        return -1;
    const int64_t rows = (int64_t)bs * next_n, total = rows * max_model_len;
    for (int64_t e = 0; e < total; ++e) {
        out[e] = -INFINITY;
        if (out64)
            out64[e] = -INFINITY;
        if (tol)
            tol[e] = 0.0;
    }
    logits_job J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.kv = kv;
    J.w = weights;
    J.ctx = context_lens;
    J.bt = block_tables;
    J.bs = bs;
    J.next_n = next_n;
    J.heads = heads;
    J.P = block_size;
    J.width = width;
    J.num_blocks = num_blocks;
    J.mml = max_model_len;
    J.out = out;
    J.out64 = out64;
    J.tol = tol;
    pmqa_ref_e4m3fn_table(J.table);
    J.chunk = 1024;
    int64_t n_items = 0;
    for (int i = 0; i < bs; ++i) {
        int64_t c = context_lens[i];
        if (c < 0 || c > max_model_len || (c + block_size - 1) / block_size > width)
            return -2;
        n_items += (c + J.chunk - 1) / J.chunk;
    }
    J.item_req = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_items + 1));
    J.item_t0 = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_items + 1));
    if (!J.item_req || !J.item_t0) {
        free(J.item_req);
        free(J.item_t0);
        return -4;
    }
    int64_t n = 0;
    for (int i = 0; i < bs; ++i)
        for (int64_t t0 = 0; t0 < context_lens[i]; t0 += J.chunk) {
            J.item_req[n] = i;
            J.item_t0[n] = t0;
            ++n;
        }
    J.n_items = n;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int k = 0; th && k < nthreads; ++k)
        if (pthread_create(&th[k], NULL, logits_worker, &J) == 0)
            ++started;
    if (started == 0)
        logits_worker(&J);
    for (int k = 0; k < started; ++k)
        pthread_join(th[k], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    free(J.item_req);
    free(J.item_t0);
    if (J.error == 1)
        return -3;
    if (J.error)
        return -4;
    return 0;
}

/* ---- top-k ----------------------------------------------------------------- */

typedef struct {
    double v;
    int32_t t;
} ref_entry;

static int entry_order(const void *a, const void *b)
{
    const ref_entry *x = (const ref_entry *)a, *y = (const ref_entry *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->t > y->t) - (x->t < y->t);
}

typedef struct {
    const double *vals;
    const int32_t *ctx;
    int bs, next_n, k;
    int64_t width;
    int32_t *idx;
    int next_row;
    pthread_mutex_t lock;
    int error;
} topk_job;

/* Number of entries of row (i, j) that the causal window admits [P1]. */
static int64_t row_valid_len(int64_t c, int next_n, int j)
{
    int64_t v = c - next_n + j + 1;
    if (v > c)
        v = c;
    return v < 0 ? 0 : v;
}

static void *topk_worker(void *arg)
{
    topk_job *J = (topk_job *)arg;
    const int rows = J->bs * J->next_n;
    ref_entry *buf = (ref_entry *)malloc(sizeof(ref_entry) * (size_t)(J->width + 1));
    if (!buf) {
        J->error = 1;
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int r = J->next_row++;
        pthread_mutex_unlock(&J->lock);
        if (r >= rows)
            break;
        int i = r / J->next_n, j = r % J->next_n;
        int64_t n = row_valid_len(J->ctx[i], J->next_n, j);
        if (n > J->width)
            n = J->width;
        const double *v = J->vals + (int64_t)r * J->width;
        for (int64_t t = 0; t < n; ++t) {
            buf[t].v = v[t];
            buf[t].t = (int32_t)t;
        }
        qsort(buf, (size_t)n, sizeof(ref_entry), entry_order);
        int32_t *o = J->idx + (int64_t)r * J->k;
        for (int64_t s = 0; s < J->k; ++s)
            o[s] = s < n ? buf[s].t : -1;
    }
    free(buf);
    return NULL;
}

/*
 * vals [bs*next_n, width] in double; idx [bs*next_n, k] (written entirely).
 * Row (i, j) considers t < min(ctx_i, ctx_i - next_n + j + 1).
 */
int pmqa_ref_topk(const double *vals, int64_t width, const int32_t *context_lens, int bs,
                  int next_n, int k, int32_t *idx, int nthreads)
{
    if (bs < 0 || next_n < 1 || k < 1 || width < 0)
        return -1;
    topk_job J;
    memset(&J, 0, sizeof J);
    J.vals = vals;
    J.ctx = context_lens;
    J.bs = bs;
    J.next_n = next_n;
    J.k = k;
    J.width = width;
    J.idx = idx;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; th && t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, topk_worker, &J) == 0)
            ++started;
    if (started == 0)
        topk_worker(&J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.error ? -4 : 0;
}

/* ---- prefill logits: contiguous keys, a key range per query row ------------
 * Source: the page "[Bug] aiter ops triton attention pa", section "Observations
 * while narrowing it down", which names the prefill indexer `fp8_mqa_logits`
 * (heads 32, head dimension 128, up to 8192 keys; query lengths M up to 4096)
 * beside the paged decode kernel. The pages
 * give its name and shapes only; its arithmetic is read here as the decode
 * definition above with the paging removed and the causal window replaced by
 * one key range per query row:
 *   k_n[d]       = e4m3fn(k[n][d]),  s_n = k_scale[n]
 *   logits[m][n] = sum_h w[m][h] * relu(s_n * sum_d q[m][h][d] * k_n[d])
 *                  for max(ks[m], 0) <= n < min(ke[m], N), else -inf.
 * Same exact double arithmetic, rounding and tolerance as pmqa_ref_logits.
 */

typedef struct {
    const uint8_t *q, *k;
    const float *ks_scale, *w;
    const int32_t *ks, *ke;
    int64_t m, n;
    int heads;
    float *out;
    double *out64, *tol;
    double table[256];
    int64_t next_row;
    pthread_mutex_t lock;
    int error;
} mqa_job;

static void mqa_row(mqa_job *J, int64_t r, double *qd)
{
    const int H = J->heads;
    int64_t lo = J->ks[r], hi = J->ke[r];
    if (lo < 0)
        lo = 0;
    if (hi > J->n)
        hi = J->n;
    for (int h = 0; h < H; ++h)
        for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
            qd[(int64_t)h * PMQA_REF_HEAD_DIM + d] =
                J->table[J->q[((int64_t)r * H + h) * PMQA_REF_HEAD_DIM + d]];
    const float *w = J->w + r * H;
    double kd[PMQA_REF_HEAD_DIM];
    for (int64_t t = lo; t < hi; ++t) {
        const uint8_t *krow = J->k + t * PMQA_REF_HEAD_DIM;
        for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
            kd[d] = J->table[krow[d]];
        const double s = (double)J->ks_scale[t];
        double sum = 0.0, mag = 0.0;
        for (int h = 0; h < H; ++h) {
            const double *qh = qd + (int64_t)h * PMQA_REF_HEAD_DIM;
            double dot = 0.0;
            for (int d = 0; d < PMQA_REF_HEAD_DIM; ++d)
                dot += qh[d] * kd[d];
            const double x = dot * s;
            sum += (double)w[h] * relu(x);
            mag += fabs((double)w[h]) * fabs(x);
        }
        const int64_t o = r * J->n + t;
        J->out[o] = (float)sum;
        if (J->out64)
            J->out64[o] = sum;
        if (J->tol)
            J->tol[o] = 1e-3 * (1.0 + mag);
    }
}

static void *mqa_worker(void *arg)
{
    mqa_job *J = (mqa_job *)arg;
    double *qd = (double *)malloc(sizeof(double) * (size_t)J->heads * PMQA_REF_HEAD_DIM);
    if (!qd) {
        J->error = 1;
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t r = J->next_row++;
        pthread_mutex_unlock(&J->lock);
        if (r >= J->m || J->error)
            break;
        mqa_row(J, r, qd);
    }
    free(qd);
    return NULL;
}

/*
 * q        [m, heads, 128] e4m3fn bytes
 * k        [n, 128] e4m3fn bytes; k_scale [n] fp32
 * weights  [m, heads] fp32; ks, ke [m] int32 (the row's key range [ks, ke))
 * out      [m, n] fp32 (written entirely); out64, tol same shape in double, or NULL
 * Returns 0, -1 for bad sizes, -4 when out of memory.
 */
int pmqa_ref_mqa_logits(const uint8_t *q, const uint8_t *k, const float *k_scale,
                        const float *weights, const int32_t *ks, const int32_t *ke, int64_t m,
                        int64_t n, int heads, int head_dim, float *out, double *out64, double *tol,
                        int nthreads)
{
    if (m < 0 || n < 0 || heads < 1 || head_dim != PMQA_REF_HEAD_DIM)
        return -1;
    const int64_t total = m * n;
    for (int64_t e = 0; e < total; ++e) {
        out[e] = -INFINITY;
        if (out64)
            out64[e] = -INFINITY;
        if (tol)
            tol[e] = 0.0;
    }
    mqa_job J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.k = k;
    J.ks_scale = k_scale;
    J.w = weights;
    J.ks = ks;
    J.ke = ke;
    J.m = m;
    J.n = n;
    J.heads = heads;
    J.out = out;
    J.out64 = out64;
    J.tol = tol;
    pmqa_ref_e4m3fn_table(J.table);
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; th && t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, mqa_worker, &J) == 0)
            ++started;
    if (started == 0)
        mqa_worker(&J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.error ? -4 : 0;
}

/* ---- sparse MLA decode ----------------------------------------------------
 *
 * Sources (page titles and sections):
 *   [P1] "[Bug] aiter ops triton attention pa", section "Downstream impact":
 *        the indexer's top-k positions are the ones the sparse MLA attention
 *        of the same decode step attends to.
 *   [P2] "[Bug][ROCm]: ROCM_AITER_MLA can select an aiter MLA decode kernel
 *        that silently returns uncorrelated output" (chat-gpts.plus summary):
 *        the MLA decode with fp8 Q and fp8 KV, 16 query heads sharing one
 *        latent KV head (gqa_ratio 16), 1..4 query rows per request
 *        (decode_qlen), and a log-sum-exp output used by decode context
 *        parallelism.
 *   [P3] "[Bugfix][Hardware][AMD] Fix last_page_len calculation in AITER MLA
 *        decode", section "The Bug": the MLA KV cache uses pages of one token
 *        (the paged form with larger pages is the same lookup).
 *
 * Readings where the pages are silent: a cached token is one latent row of
 * 576 fp8 values whose first 512 are also its value vector (the MLA layout of
 * a 512-wide compressed KV plus a 64-wide rotary key); q and the cache carry
 * one fp32 scale each (per tensor); the score of position t for head h is
 * sm_scale * q_h . k_t on the dequantised values; every listed position counts
 * once per listing (a repeated position twice), -1 entries are skipped.
 *
 * For row r (request i = row_req[r]) and head h, over its listed positions t:
 *   s_t      = sm_scale * sum_d (q_scale * q[r][h][d]) * (kv_scale * k_t[d]),  d < 576
 *   out[d]   = sum_t exp(s_t - m) * kv_scale * k_t[d] / sum_t exp(s_t - m),    d < 512
 *   lse      = m + log(sum_t exp(s_t - m)),   m = max_t s_t
 * (the softmax-weighted mean of the value rows; the shift by m changes
 * nothing mathematically and keeps exp finite). A row with no listed
 * position gives out = 0 and lse = -inf.
 * Beside them, for the parity tolerance: a_abs[d] = sum_t p_t |v_t[d]|,
 * d_abs[d] = sum_t p_t |v_t[d] - out[d]| and s_abs = max_t sm_scale *
 * sum_d |q_d k_t[d]| (dequantised), with p_t the normalised weights.
 */
#define PMQA_REF_MLA_DIM 576
#define PMQA_REF_MLA_VDIM 512

typedef struct {
    const uint8_t *q, *kv;
    const int32_t *idx, *row_req, *bt;
    double q_scale, kv_scale, sm_scale;
    int R, H, topk, P, W;
    int64_t num_blocks;
    double *out, *lse, *a_abs, *d_abs, *s_abs;
    double table[256];
    int next_row;
    pthread_mutex_t lock;
    int error;
} mla_job;

/* Slot of position t of request i, or -1 when the table does not cover it. */
static int64_t mla_slot(const mla_job *J, int i, int64_t t)
{
    if (t < 0 || t >= (int64_t)J->W * J->P)
        return -1;
    const int64_t page = J->bt[(int64_t)i * J->W + t / J->P];
    if (page < 0 || page >= J->num_blocks)
        return -1;
    return page * J->P + t % J->P;
}

static int mla_row(mla_job *J, int r, double *kd, double *s, int64_t *slot)
{
    const int H = J->H, D = PMQA_REF_MLA_DIM, V = PMQA_REF_MLA_VDIM;
    const int i = J->row_req[r];
    int n = 0;
    for (int e = 0; e < J->topk; ++e) {
        const int32_t t = J->idx[(int64_t)r * J->topk + e];
        if (t < 0)
            continue;
        const int64_t sl = mla_slot(J, i, t);
        if (sl < 0)
            return -2;
        slot[n++] = sl;
    }
    for (int h = 0; h < H; ++h) {
        const uint8_t *qrow = J->q + ((int64_t)r * H + h) * D;
        double *o = J->out + ((int64_t)r * H + h) * V;
        double qd[PMQA_REF_MLA_DIM];
        for (int d = 0; d < D; ++d)
            qd[d] = J->q_scale * J->table[qrow[d]];
        double m = -INFINITY, smag = 0.0;
        for (int e = 0; e < n; ++e) {
            const uint8_t *krow = J->kv + slot[e] * D;
            double dot = 0.0, mag = 0.0;
            for (int d = 0; d < D; ++d) {
                const double kv = J->kv_scale * J->table[krow[d]];
                dot += qd[d] * kv;
                mag += fabs(qd[d] * kv);
            }
            s[e] = J->sm_scale * dot;
            if (s[e] > m)
                m = s[e];
            if (J->sm_scale * mag > smag)
                smag = J->sm_scale * mag;
        }
        for (int d = 0; d < V; ++d)
            o[d] = 0.0;
        if (J->s_abs)
            J->s_abs[(int64_t)r * H + h] = smag;
        if (n == 0) {
            J->lse[(int64_t)r * H + h] = -INFINITY;
            if (J->a_abs)
                for (int d = 0; d < V; ++d)
                    J->a_abs[((int64_t)r * H + h) * V + d] = 0.0;
            if (J->d_abs)
                for (int d = 0; d < V; ++d)
                    J->d_abs[((int64_t)r * H + h) * V + d] = 0.0;
            continue;
        }
        double l = 0.0;
        for (int e = 0; e < n; ++e) {
            s[e] = exp(s[e] - m); /* s now holds the unnormalised weight */
            l += s[e];
        }
        for (int e = 0; e < n; ++e) {
            const uint8_t *krow = J->kv + slot[e] * D;
            const double p = s[e] / l;
            for (int d = 0; d < V; ++d)
                o[d] += p * (J->kv_scale * J->table[krow[d]]);
        }
        J->lse[(int64_t)r * H + h] = m + log(l);
        if (J->a_abs || J->d_abs) {
            double *aa = J->a_abs ? J->a_abs + ((int64_t)r * H + h) * V : NULL;
            double *da = J->d_abs ? J->d_abs + ((int64_t)r * H + h) * V : NULL;
            for (int d = 0; d < V; ++d) {
                if (aa)
                    aa[d] = 0.0;
                if (da)
                    da[d] = 0.0;
            }
            for (int e = 0; e < n; ++e) {
                const uint8_t *krow = J->kv + slot[e] * D;
                const double p = s[e] / l;
                for (int d = 0; d < V; ++d) {
                    kd[d] = J->kv_scale * J->table[krow[d]];
                    if (aa)
                        aa[d] += p * fabs(kd[d]);
                    if (da)
                        da[d] += p * fabs(kd[d] - o[d]);
                }
            }
        }
    }
    return 0;
}

static void *mla_worker(void *arg)
{
    mla_job *J = (mla_job *)arg;
    double *kd = (double *)malloc(sizeof(double) * PMQA_REF_MLA_VDIM);
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->topk > 0 ? J->topk : 1));
    int64_t *slot = (int64_t *)malloc(sizeof(int64_t) * (size_t)(J->topk > 0 ? J->topk : 1));
    if (!kd || !s || !slot) {
        J->error = -4;
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            int r = J->next_row++;
            pthread_mutex_unlock(&J->lock);
            if (r >= J->R || J->error)
                break;
            int rc = mla_row(J, r, kd, s, slot);
            if (rc) {
                pthread_mutex_lock(&J->lock);
                J->error = rc;
                pthread_mutex_unlock(&J->lock);
            }
        }
    }
    free(kd);
    free(s);
    free(slot);
    return NULL;
}

/*
 * q        [R, heads, 576] e4m3fn bytes (row r's query heads)
 * kv       [num_blocks, P, 576] e4m3fn bytes (one latent row per slot)
 * indices  [R, topk] int32 positions in the row's request, -1 = no entry
 * row_req  [R] int32: the request (block-table row) of each query row
 * block_tables [bs, W] int32
 * out      [R, heads, 512] double; lse [R, heads] double
 * a_abs, d_abs [R, heads, 512] and s_abs [R, heads] double, or NULL
 * Returns 0, -1 for bad sizes, -2 for a listed position that the table does
 * not map into the pool, -4 when out of memory.
 */
int pmqa_ref_sparse_mla(const uint8_t *q, double q_scale, const uint8_t *kv, double kv_scale,
                        const int32_t *indices, const int32_t *row_req,
                        const int32_t *block_tables, int R, int heads, int topk, int P, int W,
                        int64_t num_blocks, double sm_scale, double *out, double *lse,
                        double *a_abs, double *d_abs, double *s_abs, int nthreads)
{
    if (R < 0 || heads < 1 || topk < 0 || P < 1 || W < 0 || num_blocks < 0)
        return -1;
    mla_job J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.kv = kv;
    J.idx = indices;
    J.row_req = row_req;
    J.bt = block_tables;
    J.q_scale = q_scale;
    J.kv_scale = kv_scale;
    J.sm_scale = sm_scale;
    J.R = R;
    J.H = heads;
    J.topk = topk;
    J.P = P;
    J.W = W;
    J.num_blocks = num_blocks;
    J.out = out;
    J.lse = lse;
    J.a_abs = a_abs;
    J.d_abs = d_abs;
    J.s_abs = s_abs;
    pmqa_ref_e4m3fn_table(J.table);
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; th && t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, mla_worker, &J) == 0)
            ++started;
    if (started == 0)
        mla_worker(&J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return J.error;
}
