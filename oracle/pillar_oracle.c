/*
 * pillar_oracle.c -- fp64 CPU oracle for the PillarAttn unified step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the GPU path computes.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark may load it.  It shares no code,
 * header, table or helper with the CUDA library, and it never calls it.
 *
 * Sources (page title, then section):
 *   [MLSys26-PA]  "SparseSpec-MLSys26", section "核心方法 / PillarAttn：verify
 *                 分数驱动的动态稀疏 attention" (Core method / PillarAttn).
 *                 Draft steps attend only the current Top-K critical set
 *                 (s = 0.05); the full verify step dumps attention logits and
 *                 log-sum-exp, from which exact scores are rematerialised,
 *                 averaged over the k draft tokens and the GQA group's query
 *                 heads, and Top-K'd into the next critical set.
 *   [MLSys26-UB]  same page, section "Unified batch scheduler + fused
 *                 attention kernel": page size 1 puts sparse and full
 *                 attention on one pipeline, so draft and verify requests mix
 *                 in one batch.
 *   [Blog-4.1]    "推理模型做 decode，GPU 只有 3% 在干活——SparseSpec 把稀疏
 *                 Attention 变成了 2.1× 加速", section 4.1 PillarAttn.
 *
 * Everything is computed in double precision from the exact fp64 upcast of
 * the bf16 inputs.  Softmax is the direct two-pass form (max, then the sum of
 * exponentials) taken in the order the positions are listed.  The draft
 * (listed positions) and verify (contiguous causal prefix) paths are written
 * as separate loops on purpose, so that "draft over the full list equals
 * verify" is a real check and not an identity.
 *
 * Readings of points the pages leave open (all parameters where possible):
 *   - softmax scale: caller-given; the tests use 1/sqrt(D);
 *   - LSE: natural log of the sum of exp(logit), logits already scaled;
 *   - verify row j (0..k) of a request of length L sits at position
 *     L-(k+1)+j and attends positions [0, L-(k+1)+j];
 *   - the k averaged rows are [row_lo, row_hi) (default [1, k+1));
 *   - one critical list per (request, KV head); query head h uses KV head
 *     h / (Hq/Hkv);
 *   - positions a row may not see contribute 0 to the averaged score;
 *   - Top-K ties go to the lower position; the output list is ascending;
 *   - an empty draft list yields out = 0 and lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_INDEX -4
#define ORACLE_NO_MEMORY -5

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_f64(uint16_t bits) { return bf16_to_f64(bits); }

/* ------------------------------------------------------------------------ */
/* A tiny work-sharing pool: units [0, n) are handed out one at a time.      */

typedef void (*unit_fn)(void *ctx, long unit);

typedef struct {
    unit_fn fn;
    void *ctx;
    long n;
    long next; /* shared counter */
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    for (;;) {
        long u = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (u >= p->n)
            break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static void run_units(unit_fn fn, void *ctx, long n, int nthreads)
{
    pool_t p = {fn, ctx, n, 0};
    if (nthreads <= 1 || n <= 1) {
        pool_worker(&p);
        return;
    }
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, pool_worker, &p) == 0)
            ++started;
    if (started == 0)
        pool_worker(&p);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* Attention of one query row, two ways.                                     */

typedef struct {
    const uint16_t *k_pool, *v_pool; /* [num_slots, Hkv, D] */
    long long num_slots;
    int Hkv, D;
    double scale;
} kv_view;

/* logit of query row qh (D bf16 values) against the key in slot `slot`,
 * KV head hk: scale * sum_d q[d] * k[d]. */
static double logit_of(const kv_view *kv, const uint16_t *qh, long long slot, int hk)
{
    const uint16_t *kr = kv->k_pool + (slot * kv->Hkv + hk) * (long long)kv->D;
    double acc = 0.0;
    for (int d = 0; d < kv->D; ++d)
        acc += bf16_to_f64(qh[d]) * bf16_to_f64(kr[d]);
    return kv->scale * acc;
}

/* Sparse (draft) attention [MLSys26-PA]: the query attends exactly the n
 * listed logical positions pos[0..n), each translated to a pool slot through
 * the request's slot row (page size 1, [MLSys26-UB]).  Returns the LSE and
 * writes out[D].  logit_buf must hold n doubles.  *bad is set when a listed
 * position or its slot is out of range; such an entry is skipped. */
static double attend_listed(const kv_view *kv, const uint16_t *qh, int hk, const int32_t *slots,
                            int L, const int32_t *pos, int n, double *out, double *logit_buf, int *bad)
{
    for (int d = 0; d < kv->D; ++d)
        out[d] = 0.0;
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
        int t = pos[i];
        if (t < 0 || t >= L || slots[t] < 0 || slots[t] >= kv->num_slots) {
            *bad = 1;
            logit_buf[i] = -INFINITY;
            continue;
        }
        logit_buf[i] = logit_of(kv, qh, slots[t], hk);
        if (logit_buf[i] > m)
            m = logit_buf[i];
    }
    if (m == -INFINITY)
        return -INFINITY; /* empty (or fully invalid) list */
    double z = 0.0;
    for (int i = 0; i < n; ++i)
        if (logit_buf[i] != -INFINITY)
            z += exp(logit_buf[i] - m);
    for (int i = 0; i < n; ++i) {
        if (logit_buf[i] == -INFINITY)
            continue;
        double p = exp(logit_buf[i] - m) / z;
        const uint16_t *vr = kv->v_pool + ((long long)slots[pos[i]] * kv->Hkv + hk) * (long long)kv->D;
        for (int d = 0; d < kv->D; ++d)
            out[d] += p * bf16_to_f64(vr[d]);
    }
    return m + log(z);
}

/* Full causal (verify) attention [MLSys26-PA]: the query attends every
 * position t in [0, upto).  Written as its own loop over t.  logits[0..L) is
 * filled with the scaled logits for t < upto and -inf beyond. */
static double attend_prefix(const kv_view *kv, const uint16_t *qh, int hk, const int32_t *slots,
                            int L, int upto, double *out, double *logits, int *bad)
{
    for (int d = 0; d < kv->D; ++d)
        out[d] = 0.0;
    double m = -INFINITY;
    for (int t = 0; t < L; ++t) {
        if (t >= upto) {
            logits[t] = -INFINITY;
            continue;
        }
        if (slots[t] < 0 || slots[t] >= kv->num_slots) {
            *bad = 1;
            logits[t] = -INFINITY;
            continue;
        }
        logits[t] = logit_of(kv, qh, slots[t], hk);
        if (logits[t] > m)
            m = logits[t];
    }
    if (m == -INFINITY)
        return -INFINITY;
    double z = 0.0;
    for (int t = 0; t < upto; ++t)
        if (logits[t] != -INFINITY)
            z += exp(logits[t] - m);
    for (int t = 0; t < upto; ++t) {
        if (logits[t] == -INFINITY)
            continue;
        double p = exp(logits[t] - m) / z;
        const uint16_t *vr = kv->v_pool + ((long long)slots[t] * kv->Hkv + hk) * (long long)kv->D;
        for (int d = 0; d < kv->D; ++d)
            out[d] += p * bf16_to_f64(vr[d]);
    }
    return m + log(z);
}

/* ------------------------------------------------------------------------ */
/* The unified step: every request of the batch, draft or verify.            */

typedef struct {
    kv_view kv;
    int B, Hq, Hkv, D, k, max_sparse;
    const uint16_t *q;
    const int32_t *slot_table, *req_mode, *req_len, *sparse_idx, *sparse_cnt;
    const uint8_t *select;
    const long long *q_off, *kv_off, *logit_off; /* per request */
    double *out, *lse, *logits;
    int bad; /* any out-of-range index or slot seen */
} unified_ctx;

static void unified_unit(void *vctx, long unit)
{
    unified_ctx *c = (unified_ctx *)vctx;
    int b = (int)(unit / c->Hq), h = (int)(unit % c->Hq);
    if (c->select && !c->select[b])
        return;
    int G = c->Hq / c->Hkv, hk = h / G, L = c->req_len[b], D = c->D;
    const int32_t *slots = c->slot_table + c->kv_off[b];
    int bad = 0;
    if (c->req_mode[b] == 0) {
        /* draft: one query row, attends its critical list */
        int n = c->sparse_cnt[(long long)b * c->Hkv + hk];
        if (n < 0)
            n = 0, bad = 1;
        if (n > c->max_sparse)
            n = c->max_sparse, bad = 1;
        const int32_t *pos = c->sparse_idx + ((long long)b * c->Hkv + hk) * c->max_sparse;
        double *buf = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!buf) {
            __atomic_store_n(&c->bad, ORACLE_NO_MEMORY, __ATOMIC_RELAXED);
            return;
        }
        long long row = c->q_off[b];
        const uint16_t *qh = c->q + (row * c->Hq + h) * (long long)D;
        c->lse[row * c->Hq + h] = attend_listed(&c->kv, qh, hk, slots, L, pos, n,
                                                c->out + (row * c->Hq + h) * (long long)D, buf, &bad);
        free(buf);
    } else {
        /* verify: k+1 causal rows, each attends [0, L-(k+1)+j] */
        double *buf = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (!buf) {
            __atomic_store_n(&c->bad, ORACLE_NO_MEMORY, __ATOMIC_RELAXED);
            return;
        }
        for (int j = 0; j <= c->k; ++j) {
            long long row = c->q_off[b] + j;
            const uint16_t *qh = c->q + (row * c->Hq + h) * (long long)D;
            int upto = L - (c->k + 1) + j + 1;
            double *lg = c->logits ? c->logits + c->logit_off[b] + ((long long)h * (c->k + 1) + j) * L : buf;
            c->lse[row * c->Hq + h] = attend_prefix(&c->kv, qh, hk, slots, L, upto,
                                                    c->out + (row * c->Hq + h) * (long long)D, lg, &bad);
        }
        free(buf);
    }
    if (bad)
        __atomic_store_n(&c->bad, ORACLE_BAD_INDEX, __ATOMIC_RELAXED);
}

/*
 * oracle_attn_unified -- the whole unified draft/verify step.
 *
 *   q           [T_q, Hq, D] bf16 bits; requests packed in batch order, one row
 *               for a draft request, k+1 rows for a verify request
 *   k_pool/v_pool [num_slots, Hkv, D] bf16 bits
 *   slot_table  request b's L_b slots start at sum_{b'<b} L_b'
 *   req_mode    [B] 0 draft, 1 verify;  req_len [B] context length L_b
 *   sparse_idx  [B, Hkv, max_sparse] logical positions; sparse_cnt [B, Hkv]
 *   select      [B] or NULL: when given, only requests with select[b] != 0
 *               are computed (the others' outputs are left untouched) and the
 *               logits buffer is packed over the selected verify requests only
 *   out         [T_q, Hq, D] fp64;  lse [T_q, Hq] fp64 (draft rows too)
 *   logits      NULL or packed [sum over (selected) verify v][Hq][k+1][L_v]
 *
 * Returns 0, -1 for bad dimensions, -4 if an out-of-range position or slot
 * was skipped, -5 if memory ran out.
 */
int oracle_attn_unified(int B, int Hq, int Hkv, int D, int k, long long num_slots, double scale,
                        int max_sparse, const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        const int32_t *slot_table, const int32_t *req_mode, const int32_t *req_len,
                        const int32_t *sparse_idx, const int32_t *sparse_cnt, const uint8_t *select,
                        double *out, double *lse, double *logits, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || k < 0 || max_sparse < 0)
        return ORACLE_BAD_ARG;
    if (B == 0)
        return ORACLE_OK;
    long long *offs = (long long *)malloc(sizeof(long long) * 3 * (size_t)B);
    if (!offs)
        return ORACLE_NO_MEMORY;
    long long *q_off = offs, *kv_off = offs + B, *logit_off = offs + 2 * B;
    long long qa = 0, ka = 0, la = 0;
    for (int b = 0; b < B; ++b) {
        if (req_mode[b] != 0 && req_mode[b] != 1) {
            free(offs);
            return ORACLE_BAD_ARG;
        }
        if (req_mode[b] == 1 && req_len[b] < k + 1) {
            free(offs);
            return ORACLE_BAD_ARG;
        }
        q_off[b] = qa;
        kv_off[b] = ka;
        logit_off[b] = la;
        qa += req_mode[b] ? k + 1 : 1;
        ka += req_len[b];
        if (req_mode[b] && (!select || select[b]))
            la += (long long)Hq * (k + 1) * req_len[b];
    }
    unified_ctx c = {{k_pool, v_pool, num_slots, Hkv, D, scale},
                     B, Hq, Hkv, D, k, max_sparse, q, slot_table, req_mode, req_len, sparse_idx, sparse_cnt,
                     select, q_off, kv_off, logit_off, out, lse, logits, 0};
    run_units(unified_unit, &c, (long)B * Hq, nthreads);
    free(offs);
    return c.bad;
}

/* ------------------------------------------------------------------------ */
/* Verify-score rematerialisation, averaging and Top-K [MLSys26-PA].         */

typedef struct {
    double score;
    int t;
} scored_pos;

/* Larger score first; equal scores: lower position first. */
static int by_score_then_pos(const void *a, const void *b)
{
    const scored_pos *x = (const scored_pos *)a, *y = (const scored_pos *)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->t > y->t) - (x->t < y->t);
}

static int by_pos(const void *a, const void *b)
{
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

typedef struct {
    int V, Hq, Hkv, k, row_lo, row_hi, max_topk;
    const double *logits, *lse;
    const int32_t *L, *K;
    const long long *logit_off, *score_off;
    int32_t *next_idx, *next_cnt;
    double *scores;
    int err;
} topk_ctx;

static void topk_unit(void *vctx, long unit)
{
    topk_ctx *c = (topk_ctx *)vctx;
    int v = (int)(unit / c->Hkv), g = (int)(unit % c->Hkv);
    int G = c->Hq / c->Hkv, L = c->L[v], R = c->row_hi - c->row_lo;
    scored_pos *sp = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(L > 0 ? L : 1));
    int *sel = (int *)malloc(sizeof(int) * (size_t)(L > 0 ? L : 1));
    if (!sp || !sel) {
        free(sp);
        free(sel);
        __atomic_store_n(&c->err, ORACLE_NO_MEMORY, __ATOMIC_RELAXED);
        return;
    }
    /* score[t] = (1 / (R*G)) * sum over averaged rows r and the group's heads
     * h of the exact softmax probability exp(logit[h][r][t] - lse[h][r]). */
    for (int t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int r = c->row_lo; r < c->row_hi; ++r)
            for (int h = g * G; h < (g + 1) * G; ++h) {
                double lg = c->logits[c->logit_off[v] + ((long long)h * (c->k + 1) + r) * L + t];
                double ls = c->lse[((long long)v * c->Hq + h) * (c->k + 1) + r];
                if (lg != -INFINITY)
                    acc += exp(lg - ls);
            }
        sp[t].score = acc / ((double)R * G);
        sp[t].t = t;
        if (c->scores)
            c->scores[c->score_off[v] + (long long)g * L + t] = sp[t].score;
    }
    int K = c->K[v];
    if (K > L)
        K = L;
    if (K < 0)
        K = 0;
    if (K > c->max_topk) {
        K = c->max_topk;
        __atomic_store_n(&c->err, ORACLE_BAD_ARG, __ATOMIC_RELAXED);
    }
    qsort(sp, (size_t)L, sizeof(scored_pos), by_score_then_pos);
    for (int i = 0; i < K; ++i)
        sel[i] = sp[i].t;
    qsort(sel, (size_t)K, sizeof(int), by_pos);
    int32_t *dst = c->next_idx + ((long long)v * c->Hkv + g) * c->max_topk;
    for (int i = 0; i < K; ++i)
        dst[i] = sel[i];
    c->next_cnt[(long long)v * c->Hkv + g] = K;
    free(sp);
    free(sel);
}

/*
 * oracle_topk_select -- next critical lists from one verify pass.
 *
 *   logits    packed [V][Hq][k+1][L_v] (fp64; -inf where a row may not look)
 *   lse       [V][Hq][k+1]
 *   L         [V] context length of each verify request
 *   K         [V] number of positions to keep (clamped to [0, L_v])
 *   next_idx  [V, Hkv, max_topk] ascending positions; next_cnt [V, Hkv]
 *   scores    NULL or packed [V][Hkv][L_v]: the averaged scores
 */
int oracle_topk_select(int V, int Hq, int Hkv, int k, int row_lo, int row_hi, int max_topk,
                       const double *logits, const double *lse, const int32_t *L, const int32_t *K,
                       int32_t *next_idx, int32_t *next_cnt, double *scores, int nthreads)
{
    if (V < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || k < 0 || row_lo < 0 || row_hi > k + 1 ||
        row_lo >= row_hi || max_topk < 0)
        return ORACLE_BAD_ARG;
    if (V == 0)
        return ORACLE_OK;
    long long *offs = (long long *)malloc(sizeof(long long) * 2 * (size_t)V);
    if (!offs)
        return ORACLE_NO_MEMORY;
    long long la = 0, sa = 0;
    for (int v = 0; v < V; ++v) {
        if (L[v] < 0) {
            free(offs);
            return ORACLE_BAD_ARG;
        }
        offs[v] = la;
        offs[V + v] = sa;
        la += (long long)Hq * (k + 1) * L[v];
        sa += (long long)Hkv * L[v];
    }
    topk_ctx c = {V, Hq, Hkv, k, row_lo, row_hi, max_topk, logits, lse, L, K, offs, offs + V,
                  next_idx, next_cnt, scores, 0};
    run_units(topk_unit, &c, (long)V * Hkv, nthreads);
    free(offs);
    return c.err;
}
