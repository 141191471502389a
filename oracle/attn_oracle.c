/*
 * attn_oracle.c -- plain fp64 CPU oracle of standard (materialised) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA kernels are checked against.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it; the product library
 * never links, calls or falls back to it.  It shares no code, header, table
 * or helper with the CUDA path.
 *
 * What it computes -- the definition of exact attention, written out:
 *
 *   "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *    IO-Awareness" (abstract) and the apxml.com chapter "高效注意力算法实现
 *   (FlashAttention)", section "FlashAttention：融合算子与分块处理": the tiled
 *   method changes how attention is executed, not what it computes, so the
 *   oracle is the standard computation with S = QK^T and P = softmax(S)
 *   materialised (the same chapter's introduction, and the study notes
 *   "FlashAttention学习笔记", sections "标准attention计算" and "标准Safe
 *   softmax").
 *
 *   For one (batch b, head h), with rows q_i, k_j, v_j of Q, K, V (d wide):
 *     s_ij = scale * sum_c q_ic k_jc
 *     M(i) = { j : j < len_b  and (not causal or j <= i)
 *                 and (w < 0 or i - w <= j <= i)
 *                 and (no block mask or bm[i / bs][j / bs] != 0) }   (visible keys)
 *     m_i  = max_{j in M(i)} s_ij
 *     p_ij = exp(s_ij - m_i) / sum_{j' in M(i)} exp(s_ij' - m_i),  j in M(i)
 *     p_ij = 0                                                   otherwise
 *     o_i  = sum_j p_ij v_j
 *     L_i  = m_i + ln sum_{j in M(i)} exp(s_ij - m_i)     (natural log)
 *   An empty M(i) gives o_i = 0 and L_i = -inf.
 *
 *   Backward (the gradient of the above; the pages only say that the
 *   backward pass recomputes the attention matrix from the stored softmax
 *   statistics -- fmread.com summary, section 三.2 "反向传播优化"):
 *     dV   = P^T dO
 *     dP   = dO V^T
 *     D_i  = sum_j p_ij dP_ij            (from P and dP, not from O)
 *     dS   = P o (dP - D)                (o = elementwise)
 *     dQ   = scale * dS K
 *     dK   = scale * dS^T Q
 *
 * The two optional mask terms are the pages' extensions: a sliding (local)
 * window, named as a feature in the bxzpzcl.cn article (section "高级功能配置"),
 * read as the causal band of the w keys before each query plus the query's
 * own position; and block-sparse attention (the paper's abstract; fmread.com
 * summary, section 六 item 3), read as a 0/1 mask over (query block, key
 * block) pairs of bs x bs positions: pairs with 0 are left out, every other
 * mask still applies inside the pairs kept.
 *
 * Dropout on the attention weights (the study notes list dropout among the
 * steps fused into the kernel -- section "Kernel融合" -- without defining it),
 * read as the usual inverted dropout on P after the softmax normalisation:
 *     Pd_ij = P_ij * Z_ij / q,   o_i = sum_j Pd_ij v_j,   L unchanged,
 * Z_ij in {0, 1} kept with probability q = 1 - p.  Z comes from the
 * counter-based generator Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11), written below from
 * its definition: counter (j / 8, i, h, b), key (seed low, seed high word);
 * the call's 128 bits are eight 16-bit values u, value j % 8 (low half of
 * word (j % 8) / 2 first) deciding key j; Z_ij = [u >= t] with the integer
 * threshold t = floor(p * 65536), so q = (65536 - t) / 65536 exactly.
 * Backward with dropout: dPd = dO V^T, dP = dPd o Z / q, D_i = sum_j P_ij dP_ij,
 * dS = P o (dP - D), dV = Pd^T dO (dQ, dK as above).
 *
 * Memory: S and P are materialised for a panel of complete rows (all keys of
 * each row), so every softmax is a plain two-pass safe softmax: no online
 * rescaling appears here.  Tensors are contiguous [B, H, N, d] fp64; L and
 * kv_len are [B, H, N] and [B].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11): ten rounds of two 32x32->64 multiplications whose  */
/* high halves are XORed into the other counter words with the round key;   */
/* the key is bumped by two Weyl constants after every round.               */

static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t m0 = (uint64_t)0xD2511F53u * x0;
        uint64_t m1 = (uint64_t)0xCD9E8D57u * x2;
        uint32_t y0 = (uint32_t)(m1 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)m1;
        uint32_t y2 = (uint32_t)(m0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)m0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

int oracle_philox4x32_10(const unsigned *ctr, const unsigned *key, unsigned *out)
{
    if (!ctr || !key || !out) return 1;
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]}, k[2] = {key[0], key[1]}, o[4];
    philox4x32_10(c, k, o);
    for (int t = 0; t < 4; ++t) out[t] = o[t];
    return 0;
}

/* Dropout of one (batch, head): thr = 0 means none. */
typedef struct {
    uint32_t thr;          /* floor(p * 65536) */
    uint32_t key[2];       /* seed */
    uint32_t b, h;
    double inv_q;          /* 65536 / (65536 - thr) */
} drop_t;

static drop_t make_drop(double p, unsigned long long seed, int64_t b, int64_t h)
{
    drop_t z;
    double t = floor(p * 65536.0);
    if (t < 0) t = 0;
    if (t > 65535) t = 65535;
    z.thr = (uint32_t)t;
    z.key[0] = (uint32_t)(seed & 0xffffffffu);
    z.key[1] = (uint32_t)(seed >> 32);
    z.b = (uint32_t)b;
    z.h = (uint32_t)h;
    z.inv_q = 65536.0 / (65536.0 - (double)z.thr);
    return z;
}

/* The dropout multiplier Z_ij / q of element (i, j): 0 or 1/q. */
static double drop_mult(const drop_t *z, int64_t i, int64_t j)
{
    if (z->thr == 0) return 1.0;
    uint32_t ctr[4] = {(uint32_t)(j / 8), (uint32_t)i, z->h, z->b}, out[4];
    philox4x32_10(ctr, z->key, out);
    int t = (int)(j % 8);
    uint32_t w = out[t / 2];
    uint32_t u = (t % 2) ? (w >> 16) : (w & 0xffffu);
    return u >= z->thr ? z->inv_q : 0.0;
}

/* The mask terms of one (batch, head). */
typedef struct {
    int causal;
    int64_t len;                 /* len_b */
    int64_t window;              /* w; < 0: no window */
    const unsigned char *bmask;  /* [ceil(N/bs)][ceil(N/bs)] or NULL */
    int64_t bs, nkb;             /* block size, key blocks per mask row */
} mask_t;

/* Is key j visible from query i? (the mask set M(i) above) */
static int visible(int64_t i, int64_t j, const mask_t *m)
{
    if (j >= m->len) return 0;
    if (m->causal && j > i) return 0;
    if (m->window >= 0 && (j > i || j < i - m->window)) return 0;
    if (m->bmask && !m->bmask[(i / m->bs) * m->nkb + j / m->bs]) return 0;
    return 1;
}

static mask_t make_mask(int causal, int64_t len, int window, const unsigned char *bmask,
                        int bs, int64_t N)
{
    mask_t m;
    m.causal = causal;
    m.len = len;
    m.window = window;
    m.bmask = bmask;
    m.bs = bs > 0 ? bs : 1;
    m.nkb = (N + m.bs - 1) / m.bs;
    return m;
}

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/* ------------------------------------------------------------------------ */
/* A tiny task pool: tasks 0..ntasks-1 are handed out to nthreads threads.  */

typedef void (*task_fn)(void *ctx, int64_t task, int worker);

typedef struct {
    task_fn fn;
    void *ctx;
    int64_t ntasks;
    int64_t next;
    pthread_mutex_t lock;
} pool_t;

typedef struct {
    pool_t *pool;
    int worker;
} worker_arg_t;

static void *pool_worker(void *arg)
{
    worker_arg_t *wa = (worker_arg_t *)arg;
    pool_t *p = wa->pool;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        int64_t t = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (t >= p->ntasks) break;
        p->fn(p->ctx, t, wa->worker);
    }
    return NULL;
}

static void run_pool(task_fn fn, void *ctx, int64_t ntasks, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.ntasks = ntasks;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg_t *wa = (worker_arg_t *)malloc(sizeof(worker_arg_t) * (size_t)nthreads);
    for (int w = 0; w < nthreads; ++w) {
        wa[w].pool = &p;
        wa[w].worker = w;
    }
    for (int w = 1; w < nthreads; ++w) pthread_create(&th[w], NULL, pool_worker, &wa[w]);
    pool_worker(&wa[0]);
    for (int w = 1; w < nthreads; ++w) pthread_join(th[w], NULL);
    pthread_mutex_destroy(&p.lock);
    free(th);
    free(wa);
}

/* ------------------------------------------------------------------------ */
/* Row panel of one head: S and P for rows [r0, r0+R) against all N keys.   */

/* Fills s[r*N + j] = scale * q_i . k_j and p[r*N + j] = softmax over M(i);
 * lse[r] = the row's logsumexp.  Entries outside M(i) get p = 0 (s is left at
 * 0 there and never read). */
static void panel_probs(const double *q, const double *k, int64_t N, int d,
                        double scale, const mask_t *msk, int64_t r0,
                        int64_t R, double *s, double *p, double *lse)
{
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = r0 + r;
        double *srow = s + r * N;
        double *prow = p + r * N;
        double mx = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            if (visible(i, j, msk)) {
                srow[j] = scale * dot(q + i * d, k + j * d, d);
                if (srow[j] > mx) mx = srow[j];
            } else {
                srow[j] = 0.0;
            }
        }
        if (mx == -INFINITY) { /* empty M(i) */
            for (int64_t j = 0; j < N; ++j) prow[j] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (visible(i, j, msk)) {
                prow[j] = exp(srow[j] - mx);
                sum += prow[j];
            } else {
                prow[j] = 0.0;
            }
        }
        for (int64_t j = 0; j < N; ++j) prow[j] /= sum;
        lse[r] = mx + log(sum);
    }
}

/* Panel height so that one fp64 N-wide panel matrix stays under ~32 MB. */
static int64_t panel_rows(int64_t N)
{
    int64_t R = (int64_t)(32 << 20) / (8 * (N > 0 ? N : 1));
    if (R < 1) R = 1;
    if (R > N) R = N;
    return R;
}

/* ------------------------------------------------------------------------ */
/* Forward over whole tensors.                                               */

typedef struct {
    const double *q, *k, *v;
    int64_t H, N;
    int d;
    double scale;
    int causal;
    const int *kv_len;
    int window;
    const unsigned char *bmask;
    int bs;
    double drop_p;
    unsigned long long seed;
    double *o, *L;
    int err;
} fwd_ctx_t;

/* Rows of the panels first, first + stride, ... of head bh. */
static void fwd_panels(fwd_ctx_t *c, int64_t bh, int64_t first, int64_t stride)
{
    int64_t N = c->N;
    int d = c->d;
    int64_t b = bh / c->H;
    int64_t len = c->kv_len ? c->kv_len[b] : N;
    mask_t msk = make_mask(c->causal, len, c->window, c->bmask, c->bs, N);
    drop_t z = make_drop(c->drop_p, c->seed, b, bh % c->H);
    const double *q = c->q + bh * N * d, *k = c->k + bh * N * d, *v = c->v + bh * N * d;
    double *o = c->o + bh * N * d, *L = c->L + bh * N;
    int64_t R = panel_rows(N);
    double *s = (double *)malloc(sizeof(double) * (size_t)(R * N));
    double *p = (double *)malloc(sizeof(double) * (size_t)(R * N));
    double *lse = (double *)malloc(sizeof(double) * (size_t)R);
    if (!s || !p || !lse) {
        c->err = ORACLE_ERR_NOMEM;
        free(s); free(p); free(lse);
        return;
    }
    for (int64_t r0 = first * R; r0 < N; r0 += stride * R) {
        int64_t rr = (r0 + R <= N) ? R : N - r0;
        panel_probs(q, k, N, d, c->scale, &msk, r0, rr, s, p, lse);
        for (int64_t r = 0; r < rr; ++r) {
            int64_t i = r0 + r;
            double *oi = o + i * d;
            for (int c2 = 0; c2 < d; ++c2) oi[c2] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double pij = p[r * N + j];
                if (pij == 0.0) continue;
                pij *= drop_mult(&z, i, j);
                const double *vj = v + j * d;
                for (int c2 = 0; c2 < d; ++c2) oi[c2] += pij * vj[c2];
            }
            L[i] = lse[r];
        }
    }
    free(s); free(p); free(lse);
}

/* Split of the host threads: heads run in parallel; when there are fewer
 * heads than threads, the row panels of one head are dealt out to a team of
 * `inner` threads (panel t to team member t mod inner). */
typedef struct {
    void *ctx;
    int64_t bh;
    int64_t member, inner;
    double *dk, *dv; /* backward: this member's partial dK, dV of the head */
} team_arg_t;

static void *fwd_member(void *arg)
{
    team_arg_t *t = (team_arg_t *)arg;
    fwd_panels((fwd_ctx_t *)t->ctx, t->bh, t->member, t->inner);
    return NULL;
}

/* Runs fn(args[0..n)) on n threads (member 0 on the calling thread). */
static void run_team(void *(*fn)(void *), team_arg_t *args, int64_t n)
{
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
    int64_t started = 1;
    if (th) {
        for (; started < n; ++started)
            if (pthread_create(&th[started], NULL, fn, &args[started]) != 0) break;
    }
    fn(&args[0]);
    for (int64_t w = 1; w < started; ++w) pthread_join(th[w], NULL);
    /* members whose thread could not be started run here, in order */
    for (int64_t w = started; w < n; ++w) fn(&args[w]);
    free(th);
}

typedef struct {
    void *ctx;
    int64_t inner;
} outer_ctx_t;

static void fwd_task(void *vctx, int64_t bh, int worker)
{
    (void)worker;
    outer_ctx_t *oc = (outer_ctx_t *)vctx;
    if (oc->inner <= 1) {
        fwd_panels((fwd_ctx_t *)oc->ctx, bh, 0, 1);
        return;
    }
    team_arg_t *ta = (team_arg_t *)calloc((size_t)oc->inner, sizeof(team_arg_t));
    if (!ta) { ((fwd_ctx_t *)oc->ctx)->err = ORACLE_ERR_NOMEM; return; }
    for (int64_t w = 0; w < oc->inner; ++w) {
        ta[w].ctx = oc->ctx;
        ta[w].bh = bh;
        ta[w].member = w;
        ta[w].inner = oc->inner;
    }
    run_team(fwd_member, ta, oc->inner);
    free(ta);
}

/* Threads per head when there are fewer heads than threads. */
static int64_t inner_threads(int64_t heads, int nthreads)
{
    if (heads < 1 || nthreads <= heads) return 1;
    return nthreads / heads;
}

int oracle_attn_fwd(const double *q, const double *k, const double *v, int B, int H,
                    int N, int d, double scale, int causal, const int *kv_len, int window,
                    const unsigned char *block_mask, int block, double drop_p,
                    unsigned long long seed, double *o, double *L, int nthreads)
{
    if (!q || !k || !v || !o || !L || B < 0 || H < 0 || N < 0 || d < 1) return ORACLE_ERR_ARG;
    if (block_mask && block < 1) return ORACLE_ERR_ARG;
    if (!(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    fwd_ctx_t c = {q, k, v, H, N, d, scale, causal, kv_len, window, block_mask, block,
                   drop_p, seed, o, L, ORACLE_OK};
    outer_ctx_t oc = {&c, inner_threads((int64_t)B * H, nthreads)};
    run_pool(fwd_task, &oc, (int64_t)B * H, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* Backward over whole tensors (one task per (b, h); a head split across a   */
/* team of threads sums the members' dK, dV partials in member order).       */

typedef struct {
    const double *q, *k, *v, *dout;
    int64_t H, N;
    int d;
    double scale;
    int causal;
    const int *kv_len;
    int window;
    const unsigned char *bmask;
    int bs;
    double drop_p;
    unsigned long long seed;
    double *dq, *dk, *dv;
    int err;
} bwd_ctx_t;

/* dQ rows of the panels first, first + stride, ... of head bh; their dK and
 * dV contributions are added to dk_acc, dv_acc ([N, d] of that head). */
static void bwd_panels(bwd_ctx_t *c, int64_t bh, int64_t first, int64_t stride,
                       double *dk_acc, double *dv_acc)
{
    int64_t N = c->N;
    int d = c->d;
    int64_t b = bh / c->H;
    int64_t len = c->kv_len ? c->kv_len[b] : N;
    mask_t msk = make_mask(c->causal, len, c->window, c->bmask, c->bs, N);
    drop_t z = make_drop(c->drop_p, c->seed, b, bh % c->H);
    int64_t off = bh * N * d;
    const double *q = c->q + off, *k = c->k + off, *v = c->v + off, *dout = c->dout + off;
    double *dq = c->dq + off;
    int64_t R = panel_rows(N);
    double *s = (double *)malloc(sizeof(double) * (size_t)(R * N));
    double *p = (double *)malloc(sizeof(double) * (size_t)(R * N));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(R * N));
    double *lse = (double *)malloc(sizeof(double) * (size_t)R);
    if (!s || !p || !dp || !lse) {
        c->err = ORACLE_ERR_NOMEM;
        free(s); free(p); free(dp); free(lse);
        return;
    }
    for (int64_t r0 = first * R; r0 < N; r0 += stride * R) {
        int64_t rr = (r0 + R <= N) ? R : N - r0;
        panel_probs(q, k, N, d, c->scale, &msk, r0, rr, s, p, lse);
        for (int64_t r = 0; r < rr; ++r) {
            int64_t i = r0 + r;
            const double *doi = dout + i * d;
            double *prow = p + r * N, *dprow = dp + r * N;
            /* dP_ij = (dO_i . v_j) Z_ij / q and D_i = sum_j p_ij dP_ij */
            double Di = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                dprow[j] = visible(i, j, &msk) ? dot(doi, v + j * d, d) * drop_mult(&z, i, j) : 0.0;
                Di += prow[j] * dprow[j];
            }
            double *dqi = dq + i * d;
            for (int c2 = 0; c2 < d; ++c2) dqi[c2] = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double pij = prow[j];
                if (pij == 0.0) continue;
                double dsij = pij * (dprow[j] - Di);
                double pdij = pij * drop_mult(&z, i, j);
                const double *kj = k + j * d;
                const double *qi = q + i * d;
                double *dkj = dk_acc + j * d, *dvj = dv_acc + j * d;
                for (int c2 = 0; c2 < d; ++c2) {
                    dqi[c2] += c->scale * dsij * kj[c2];
                    dkj[c2] += c->scale * dsij * qi[c2];
                    dvj[c2] += pdij * doi[c2];
                }
            }
        }
    }
    free(s); free(p); free(dp); free(lse);
}

static void *bwd_member(void *arg)
{
    team_arg_t *t = (team_arg_t *)arg;
    bwd_panels((bwd_ctx_t *)t->ctx, t->bh, t->member, t->inner, t->dk, t->dv);
    return NULL;
}

static void bwd_task(void *vctx, int64_t bh, int worker)
{
    (void)worker;
    outer_ctx_t *oc = (outer_ctx_t *)vctx;
    bwd_ctx_t *c = (bwd_ctx_t *)oc->ctx;
    int64_t N = c->N;
    int d = c->d;
    int64_t off = bh * N * d;
    double *dk = c->dk + off, *dv = c->dv + off;
    memset(dk, 0, sizeof(double) * (size_t)(N * d));
    memset(dv, 0, sizeof(double) * (size_t)(N * d));
    if (oc->inner <= 1) {
        bwd_panels(c, bh, 0, 1, dk, dv);
        return;
    }
    /* Member 0 adds into dk, dv; the others into partials that are then
     * added in member order (a fixed order: the result does not depend on
     * thread timing). */
    int64_t W = oc->inner;
    team_arg_t *ta = (team_arg_t *)calloc((size_t)W, sizeof(team_arg_t));
    double *part = (double *)calloc((size_t)(2 * (W - 1) * N * d), sizeof(double));
    if (!ta || !part) {
        free(ta); free(part);
        c->err = ORACLE_ERR_NOMEM;
        return;
    }
    for (int64_t w = 0; w < W; ++w) {
        ta[w].ctx = c;
        ta[w].bh = bh;
        ta[w].member = w;
        ta[w].inner = W;
        ta[w].dk = w == 0 ? dk : part + (2 * (w - 1)) * N * d;
        ta[w].dv = w == 0 ? dv : part + (2 * (w - 1) + 1) * N * d;
    }
    run_team(bwd_member, ta, W);
    for (int64_t w = 1; w < W; ++w)
        for (int64_t e = 0; e < N * d; ++e) {
            dk[e] += ta[w].dk[e];
            dv[e] += ta[w].dv[e];
        }
    free(ta); free(part);
}

int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int B, int H, int N, int d, double scale, int causal, const int *kv_len,
                    int window, const unsigned char *block_mask, int block, double drop_p,
                    unsigned long long seed, double *dq, double *dk, double *dv, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || B < 0 || H < 0 || N < 0 || d < 1)
        return ORACLE_ERR_ARG;
    if (block_mask && block < 1) return ORACLE_ERR_ARG;
    if (!(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    bwd_ctx_t c = {q, k, v, dout, H, N, d, scale, causal, kv_len, window, block_mask, block,
                   drop_p, seed, dq, dk, dv, ORACLE_OK};
    outer_ctx_t oc = {&c, inner_threads((int64_t)B * H, nthreads)};
    run_pool(bwd_task, &oc, (int64_t)B * H, nthreads);
    return c.err;
}

/* ------------------------------------------------------------------------ */
/* Sampled outputs of ONE head (q, k, v, dout are [N, d] of that head).      */
/* They follow the same definitions row by row; used where the whole result */
/* would take the CPU too long.                                              */

/* o_out[r*d..], L_out[r] for the listed query rows. */
int oracle_fwd_rows(const double *q, const double *k, const double *v, int N, int d,
                    double scale, int causal, int len, int window,
                    const unsigned char *block_mask, int block, double drop_p,
                    unsigned long long seed, int b, int h, int nrows, const int *rows,
                    double *o_out, double *L_out)
{
    if (!q || !k || !v || !rows || !o_out || !L_out || N < 1 || d < 1) return ORACLE_ERR_ARG;
    if (block_mask && block < 1) return ORACLE_ERR_ARG;
    if (!(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    mask_t msk = make_mask(causal, len, window, block_mask, block, N);
    drop_t z = make_drop(drop_p, seed, b, h);
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s || !p) { free(s); free(p); return ORACLE_ERR_NOMEM; }
    for (int r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        if (i < 0 || i >= N) { free(s); free(p); return ORACLE_ERR_ARG; }
        double lse;
        panel_probs(q, k, N, d, scale, &msk, i, 1, s, p, &lse);
        for (int c = 0; c < d; ++c) o_out[(int64_t)r * d + c] = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            double pd = p[j] * drop_mult(&z, i, j);
            for (int c = 0; c < d; ++c) o_out[(int64_t)r * d + c] += pd * v[j * d + c];
        }
        L_out[r] = lse;
    }
    free(s); free(p);
    return ORACLE_OK;
}

/* dq_out[r*d..] for the listed query rows (each dQ row needs only its own
 * row of P and dP). */
int oracle_bwd_dq_rows(const double *q, const double *k, const double *v, const double *dout,
                       int N, int d, double scale, int causal, int len, int window,
                       const unsigned char *block_mask, int block, double drop_p,
                       unsigned long long seed, int b, int h, int nrows,
                       const int *rows, double *dq_out)
{
    if (!q || !k || !v || !dout || !rows || !dq_out || N < 1 || d < 1) return ORACLE_ERR_ARG;
    if (block_mask && block < 1) return ORACLE_ERR_ARG;
    if (!(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    mask_t msk = make_mask(causal, len, window, block_mask, block, N);
    drop_t z = make_drop(drop_p, seed, b, h);
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    double *dp = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s || !p || !dp) { free(s); free(p); free(dp); return ORACLE_ERR_NOMEM; }
    for (int r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        if (i < 0 || i >= N) { free(s); free(p); free(dp); return ORACLE_ERR_ARG; }
        double lse;
        panel_probs(q, k, N, d, scale, &msk, i, 1, s, p, &lse);
        const double *doi = dout + i * d;
        double Di = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            dp[j] = visible(i, j, &msk) ? dot(doi, v + j * d, d) * drop_mult(&z, i, j) : 0.0;
            Di += p[j] * dp[j];
        }
        double *dqi = dq_out + (int64_t)r * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            double ds = p[j] * (dp[j] - Di);
            for (int c = 0; c < d; ++c) dqi[c] += scale * ds * k[j * d + c];
        }
    }
    free(s); free(p); free(dp);
    return ORACLE_OK;
}

/* dK and dV rows (keys) for the listed key indices.  Every query row's
 * logsumexp and D_i are needed first; they are computed for all N rows. */
typedef struct {
    const double *q, *k, *v, *dout;
    int64_t N;
    int d;
    double scale;
    const mask_t *msk;
    const drop_t *drop;
    double *lse, *D;
} rowstat_ctx_t;

static void rowstat_task(void *vctx, int64_t i, int worker)
{
    (void)worker;
    rowstat_ctx_t *c = (rowstat_ctx_t *)vctx;
    int64_t N = c->N;
    int d = c->d;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s || !p) { free(s); free(p); c->lse[i] = NAN; return; }
    double lse;
    panel_probs(c->q, c->k, N, d, c->scale, c->msk, i, 1, s, p, &lse);
    double Di = 0.0;
    for (int64_t j = 0; j < N; ++j)
        if (p[j] != 0.0)
            Di += p[j] * dot(c->dout + i * d, c->v + j * d, d) * drop_mult(c->drop, i, j);
    c->lse[i] = lse;
    c->D[i] = Di;
    free(s); free(p);
}

int oracle_bwd_dkdv_cols(const double *q, const double *k, const double *v,
                         const double *dout, int N, int d, double scale, int causal,
                         int len, int window, const unsigned char *block_mask, int block,
                         double drop_p, unsigned long long seed, int b, int h,
                         int ncols, const int *cols, double *dk_out,
                         double *dv_out, int nthreads)
{
    if (!q || !k || !v || !dout || !cols || !dk_out || !dv_out || N < 1 || d < 1)
        return ORACLE_ERR_ARG;
    if (block_mask && block < 1) return ORACLE_ERR_ARG;
    if (!(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    mask_t msk = make_mask(causal, len, window, block_mask, block, N);
    drop_t z = make_drop(drop_p, seed, b, h);
    double *lse = (double *)malloc(sizeof(double) * (size_t)N);
    double *D = (double *)malloc(sizeof(double) * (size_t)N);
    if (!lse || !D) { free(lse); free(D); return ORACLE_ERR_NOMEM; }
    rowstat_ctx_t rc = {q, k, v, dout, N, d, scale, &msk, &z, lse, D};
    run_pool(rowstat_task, &rc, N, nthreads);
    for (int64_t i = 0; i < N; ++i)
        if (isnan(lse[i])) { free(lse); free(D); return ORACLE_ERR_NOMEM; }
    for (int r = 0; r < ncols; ++r) {
        int64_t j = cols[r];
        if (j < 0 || j >= N) { free(lse); free(D); return ORACLE_ERR_ARG; }
        double *dkj = dk_out + (int64_t)r * d, *dvj = dv_out + (int64_t)r * d;
        for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
        for (int64_t i = 0; i < N; ++i) {
            if (!visible(i, j, &msk)) continue;
            double pij = exp(scale * dot(q + i * d, k + j * d, d) - lse[i]);
            double mij = drop_mult(&z, i, j);
            double dpij = dot(dout + i * d, v + j * d, d) * mij;
            double ds = pij * (dpij - D[i]);
            for (int c = 0; c < d; ++c) {
                dkj[c] += scale * ds * q[i * d + c];
                dvj[c] += pij * mij * dout[i * d + c];
            }
        }
    }
    free(lse); free(D);
    return ORACLE_OK;
}

/* The dropout multipliers Z_ij / q of one (batch, head), [N, N] row-major
 * (test access to the same definition the computations above use). */
int oracle_dropout_mult(int b, int h, int N, double drop_p, unsigned long long seed,
                        double *out)
{
    if (!out || N < 0 || !(drop_p >= 0.0 && drop_p < 1.0)) return ORACLE_ERR_ARG;
    drop_t z = make_drop(drop_p, seed, b, h);
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < N; ++j) out[i * N + j] = drop_mult(&z, i, j);
    return ORACLE_OK;
}
