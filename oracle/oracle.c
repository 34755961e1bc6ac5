/*
 * oracle.c -- plain, slow, fp64 CPU statement of what the sequence-parallel
 * attention path computes.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * library includes, links or calls this file; only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load it.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Sources (pages, cited by title and section):
 *  - "adv07: Sequence Parallel" tutorial (mini-vllm), section 3, Q4:
 *        out[i] = softmax(q[i] . K^T / sqrt(d)) . V, the causal mask hides
 *        only future positions j > i, and a Q shard masks by the GLOBAL row
 *        position (shard 1 of seq 1024 holds rows 512..1023 and its row 768
 *        sees keys 0..768).
 *  - same tutorial, section 4 (sp_attention): every Q row depends only on
 *        q[i] and the full K/V, so Q may be split into shards and the results
 *        concatenated.
 *  - "Parallel multi-head attention" (mlwithme), section 3.2: scores =
 *        q k^T / sqrt(head_dim), an additive mask, softmax in float.
 *  - "Support deepspeed sequence parallel" (huggingface/transformers PR 31525),
 *        data-collator example: sub-sequence r holds rows
 *        [r*seq/N, (r+1)*seq/N) and the key mask is (input_ids != pad).
 *  - long-context-attention issue "关于数据分割和合并": inputs are sequence
 *        shards [b, s/N, h, d]; the all-to-all regroups them so that every
 *        rank holds the full sequence for a subset of heads.
 *
 * Readings taken where the pages are silent:
 *  - key padding is right padding: key j of batch b is valid iff
 *    j < key_len[b];
 *  - a general key mask (the transformers PR 31525 collator's
 *    attention_mask = input_ids != pad_token_id, pads anywhere) removes key j
 *    of batch b where key_mask[b][j] == 0; it combines with the causal rule
 *    and key_len (a key must pass all three);
 *  - a row with no valid key has out = 0, lse = -inf and no gradient;
 *  - lse is the natural-log log-sum-exp of the scaled scores;
 *  - the backward pass is the textbook derivative of the forward definition
 *    (the pages give none):
 *        D_i   = sum_c dO_ic * out_ic
 *        dP_ij = dO_i . v_j
 *        dS_ij = P_ij * (dP_ij - D_i)
 *        dQ_i  = scale * sum_j dS_ij k_j
 *        dK_j  = scale * sum_i dS_ij q_i
 *        dV_j  = sum_i P_ij dO_i
 *
 * Layouts (all row-major, fp64): q, out, dout, dq: [B][sq][H][d];
 * k, v, dk, dv: [B][sk][H][d]; lse: [B][H][sq].
 *
 * Threads: plain pthreads over independent (batch, head, row-block) tasks.
 * Each output element is written by exactly one task, in a fixed order, so
 * results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int B, H, sq, sk, d;
    int causal;            /* 1: key j visible from row i iff j <= q_offset + i */
    int q_offset;          /* global sequence position of query row 0 */
    const int32_t* key_len;/* NULL, or [B]: keys j >= key_len[b] are padding */
    const uint8_t* key_mask;/* NULL, or [B][sk]: key j of batch b takes part iff nonzero */
    double scale;          /* multiplies q.k; the pages use 1/sqrt(head_dim) */
} oracle_problem;

/* ------------------------------------------------------------------ */
/* indexing and the visible key set J(b, i)                           */
/* ------------------------------------------------------------------ */

static size_t q_at(const oracle_problem* p, int b, int i, int h)
{
    return (((size_t)b * p->sq + i) * p->H + h) * p->d;
}

static size_t k_at(const oracle_problem* p, int b, int j, int h)
{
    return (((size_t)b * p->sk + j) * p->H + h) * p->d;
}

static int visible(const oracle_problem* p, int b, int i, int j)
{
    if (p->causal && j > p->q_offset + i) return 0;
    if (p->key_len != NULL && j >= p->key_len[b]) return 0;
    if (p->key_mask != NULL && p->key_mask[(size_t)b * p->sk + j] == 0) return 0;
    return 1;
}

static double dot(const double* a, const double* b, int n)
{
    double acc = 0.0;
    for (int c = 0; c < n; ++c) acc += a[c] * b[c];
    return acc;
}

/* ------------------------------------------------------------------ */
/* forward of one query row: out_i = sum_J P_ij v_j, lse_i = m + ln l  */
/* ------------------------------------------------------------------ */

static void row_forward(const oracle_problem* p, const double* q, const double* k,
                        const double* v, int b, int h, int i, double* srow,
                        double* out_i, double* lse_i)
{
    const int d = p->d;
    const double* qi = q + q_at(p, b, i, h);
    double m = -INFINITY;
    for (int j = 0; j < p->sk; ++j) {
        if (!visible(p, b, i, j)) continue;
        srow[j] = p->scale * dot(qi, k + k_at(p, b, j, h), d);
        if (srow[j] > m) m = srow[j];
    }
    for (int c = 0; c < d; ++c) out_i[c] = 0.0;
    if (m == -INFINITY) {           /* empty key set */
        *lse_i = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < p->sk; ++j)
        if (visible(p, b, i, j)) l += exp(srow[j] - m);
    for (int j = 0; j < p->sk; ++j) {
        if (!visible(p, b, i, j)) continue;
        const double w = exp(srow[j] - m) / l;
        const double* vj = v + k_at(p, b, j, h);
        for (int c = 0; c < d; ++c) out_i[c] += w * vj[c];
    }
    *lse_i = m + log(l);
}

/* P_ij recomputed from the row's lse: exp(s_ij - lse_i). */
static double prob(const oracle_problem* p, const double* q, const double* k, int b,
                   int h, int i, int j, double lse_i)
{
    const double s = p->scale * dot(q + q_at(p, b, i, h), k + k_at(p, b, j, h), p->d);
    return exp(s - lse_i);
}

/* ------------------------------------------------------------------ */
/* a tiny task pool                                                    */
/* ------------------------------------------------------------------ */

typedef void (*task_fn)(void* ctx, long t);

typedef struct {
    task_fn fn;
    void* ctx;
    long ntasks;
    long next;
    pthread_mutex_t mu;
} pool;

static void* pool_worker(void* arg)
{
    pool* pl = (pool*)arg;
    for (;;) {
        pthread_mutex_lock(&pl->mu);
        long t = pl->next++;
        pthread_mutex_unlock(&pl->mu);
        if (t >= pl->ntasks) break;
        pl->fn(pl->ctx, t);
    }
    return NULL;
}

static int g_threads = 0;

int oracle_set_threads(int n)
{
    g_threads = n;
    return n;
}

int oracle_get_threads(void)
{
    if (g_threads > 0) return g_threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_tasks(task_fn fn, void* ctx, long ntasks)
{
    pool pl;
    pl.fn = fn;
    pl.ctx = ctx;
    pl.ntasks = ntasks;
    pl.next = 0;
    pthread_mutex_init(&pl.mu, NULL);
    int nt = oracle_get_threads();
    if (nt > ntasks) nt = (int)ntasks;
    if (nt <= 1) {
        pool_worker(&pl);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
        for (int t = 0; t < nt; ++t) pthread_create(&th[t], NULL, pool_worker, &pl);
        for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
        free(th);
    }
    pthread_mutex_destroy(&pl.mu);
}

/* ------------------------------------------------------------------ */
/* row-range requests                                                  */
/*                                                                     */
/* Every entry point works on one head (b, h) and a half-open range of */
/* rows, so a test can evaluate sampled rows of a very long sequence.  */
/* Full tensors are the union of all heads and the full ranges.        */
/* ------------------------------------------------------------------ */

typedef struct {
    const oracle_problem* p;
    const double *q, *k, *v, *dout;
    int b, h;
    int i0, i1;          /* query rows */
    int j0, j1;          /* key rows (dK/dV) */
    double* out;         /* [i1-i0][d] */
    double* lse;         /* [i1-i0] */
    double* D;           /* [i1-i0] */
    double* dq;          /* [i1-i0][d] */
    double* dk;          /* [j1-j0][d] */
    double* dv;          /* [j1-j0][d] */
} head_job;

enum { ROWS_PER_TASK = 16 };

static void fwd_task(void* vctx, long t)
{
    head_job* J = (head_job*)vctx;
    const oracle_problem* p = J->p;
    double* srow = (double*)malloc(sizeof(double) * (size_t)(p->sk > 0 ? p->sk : 1));
    const int r0 = J->i0 + (int)t * ROWS_PER_TASK;
    const int r1 = r0 + ROWS_PER_TASK < J->i1 ? r0 + ROWS_PER_TASK : J->i1;
    for (int i = r0; i < r1; ++i) {
        double* o = J->out + (size_t)(i - J->i0) * p->d;
        row_forward(p, J->q, J->k, J->v, J->b, J->h, i, srow, o, &J->lse[i - J->i0]);
        if (J->D != NULL) {
            const double* doi = J->dout + q_at(p, J->b, i, J->h);
            J->D[i - J->i0] = dot(doi, o, p->d);
        }
    }
    free(srow);
}

static long ntasks_for(int n)
{
    return (n + ROWS_PER_TASK - 1) / ROWS_PER_TASK;
}

/* dQ_i = scale * sum_J dS_ij k_j for rows i in [i0, i1); needs lse and D of those rows. */
static void dq_task(void* vctx, long t)
{
    head_job* J = (head_job*)vctx;
    const oracle_problem* p = J->p;
    const int d = p->d;
    const int r0 = J->i0 + (int)t * ROWS_PER_TASK;
    const int r1 = r0 + ROWS_PER_TASK < J->i1 ? r0 + ROWS_PER_TASK : J->i1;
    for (int i = r0; i < r1; ++i) {
        double* dqi = J->dq + (size_t)(i - J->i0) * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        const double lse_i = J->lse[i - J->i0];
        if (lse_i == -INFINITY) continue;
        const double* doi = J->dout + q_at(p, J->b, i, J->h);
        for (int j = 0; j < p->sk; ++j) {
            if (!visible(p, J->b, i, j)) continue;
            const double P = prob(p, J->q, J->k, J->b, J->h, i, j, lse_i);
            const double dP = dot(doi, J->v + k_at(p, J->b, j, J->h), d);
            const double dS = P * (dP - J->D[i - J->i0]);
            const double* kj = J->k + k_at(p, J->b, j, J->h);
            for (int c = 0; c < d; ++c) dqi[c] += p->scale * dS * kj[c];
        }
    }
}

/*
 * dK_j, dV_j for key rows j in [j0, j1).  The job's query range [i0, i1)
 * must cover every query row that can see one of these keys, and its lse/D
 * must already hold those rows' statistics.
 */
static void dkv_task(void* vctx, long t)
{
    head_job* J = (head_job*)vctx;
    const oracle_problem* p = J->p;
    const int d = p->d;
    const int r0 = J->j0 + (int)t * ROWS_PER_TASK;
    const int r1 = r0 + ROWS_PER_TASK < J->j1 ? r0 + ROWS_PER_TASK : J->j1;
    for (int j = r0; j < r1; ++j) {
        double* dkj = J->dk + (size_t)(j - J->j0) * d;
        double* dvj = J->dv + (size_t)(j - J->j0) * d;
        for (int c = 0; c < d; ++c) dkj[c] = dvj[c] = 0.0;
        const double* vj = J->v + k_at(p, J->b, j, J->h);
        for (int i = J->i0; i < J->i1; ++i) {
            if (!visible(p, J->b, i, j)) continue;
            const double lse_i = J->lse[i - J->i0];
            if (lse_i == -INFINITY) continue;
            const double* doi = J->dout + q_at(p, J->b, i, J->h);
            const double* qi = J->q + q_at(p, J->b, i, J->h);
            const double P = prob(p, J->q, J->k, J->b, J->h, i, j, lse_i);
            const double dP = dot(doi, vj, d);
            const double dS = P * (dP - J->D[i - J->i0]);
            for (int c = 0; c < d; ++c) {
                dvj[c] += P * doi[c];
                dkj[c] += p->scale * dS * qi[c];
            }
        }
    }
}

static int check(const oracle_problem* p)
{
    if (p == NULL || p->B < 0 || p->H < 0 || p->sq < 0 || p->sk < 0 || p->d <= 0) return 1;
    if (p->key_len != NULL)
        for (int b = 0; b < p->B; ++b)
            if (p->key_len[b] < 0 || p->key_len[b] > p->sk) return 1;
    return 0;
}

/*
 * Forward on query rows [i0, i1) of head (b, h).
 * out: [i1-i0][d] (row-major), lse: [i1-i0].
 */
int oracle_attn_fwd_rows(const oracle_problem* p, const double* q, const double* k,
                         const double* v, int b, int h, int i0, int i1, double* out,
                         double* lse)
{
    if (check(p) || i0 < 0 || i1 > p->sq || i0 > i1) return 1;
    head_job J;
    memset(&J, 0, sizeof J);
    J.p = p; J.q = q; J.k = k; J.v = v; J.b = b; J.h = h;
    J.i0 = i0; J.i1 = i1; J.out = out; J.lse = lse;
    run_tasks(fwd_task, &J, ntasks_for(i1 - i0));
    return 0;
}

/*
 * Backward on one head (b, h): dQ for query rows [i0, i1) and dK/dV for
 * key rows [j0, j1).  Statistics are recomputed here, in fp64, for every
 * query row the requested outputs depend on.
 * dq: [i1-i0][d], dk/dv: [j1-j0][d]; any of them may be NULL with an empty range.
 */
int oracle_attn_bwd_rows(const oracle_problem* p, const double* q, const double* k,
                         const double* v, const double* dout, int b, int h, int i0,
                         int i1, double* dq, int j0, int j1, double* dk, double* dv)
{
    if (check(p) || i0 < 0 || i1 > p->sq || i0 > i1 || j0 < 0 || j1 > p->sk || j0 > j1)
        return 1;
    const int d = p->d;
    /* query rows needed: the dQ rows, plus every row that can see a key in [j0, j1). */
    int lo = p->sq, hi = 0;
    if (i1 > i0) { lo = i0; hi = i1; }
    if (j1 > j0) {
        int first = 0;
        if (p->causal) {
            first = j0 - p->q_offset;
            if (first < 0) first = 0;
        }
        if (first < lo) lo = first;
        hi = p->sq;
    }
    if (lo > hi) lo = hi;
    const int n = hi - lo;
    double* out = (double*)malloc(sizeof(double) * ((size_t)n * d + 1));
    double* lse = (double*)malloc(sizeof(double) * ((size_t)n + 1));
    double* D = (double*)malloc(sizeof(double) * ((size_t)n + 1));
    head_job S;
    memset(&S, 0, sizeof S);
    S.p = p; S.q = q; S.k = k; S.v = v; S.dout = dout; S.b = b; S.h = h;
    S.i0 = lo; S.i1 = hi; S.out = out; S.lse = lse; S.D = D;
    run_tasks(fwd_task, &S, ntasks_for(n));

    if (i1 > i0) {
        head_job Q = S;
        Q.i0 = i0; Q.i1 = i1;
        Q.lse = lse + (i0 - lo);
        Q.D = D + (i0 - lo);
        Q.dq = dq;
        run_tasks(dq_task, &Q, ntasks_for(i1 - i0));
    }
    if (j1 > j0) {
        head_job K = S;
        K.j0 = j0; K.j1 = j1; K.dk = dk; K.dv = dv;
        run_tasks(dkv_task, &K, ntasks_for(j1 - j0));
    }
    free(out);
    free(lse);
    free(D);
    return 0;
}

/* Full forward: out [B][sq][H][d], lse [B][H][sq]. */
int oracle_attn_fwd(const oracle_problem* p, const double* q, const double* k,
                    const double* v, double* out, double* lse)
{
    if (check(p)) return 1;
    const int d = p->d;
    double* o = (double*)malloc(sizeof(double) * ((size_t)p->sq * d + 1));
    for (int b = 0; b < p->B; ++b)
        for (int h = 0; h < p->H; ++h) {
            oracle_attn_fwd_rows(p, q, k, v, b, h, 0, p->sq, o, lse + ((size_t)b * p->H + h) * p->sq);
            for (int i = 0; i < p->sq; ++i)
                memcpy(out + q_at(p, b, i, h), o + (size_t)i * d, sizeof(double) * d);
        }
    free(o);
    return 0;
}

/* Full backward: dq [B][sq][H][d], dk/dv [B][sk][H][d]. */
int oracle_attn_bwd(const oracle_problem* p, const double* q, const double* k,
                    const double* v, const double* dout, double* dq, double* dk, double* dv)
{
    if (check(p)) return 1;
    const int d = p->d;
    double* a = (double*)malloc(sizeof(double) * ((size_t)p->sq * d + 1));
    double* bk = (double*)malloc(sizeof(double) * ((size_t)p->sk * d + 1));
    double* bv = (double*)malloc(sizeof(double) * ((size_t)p->sk * d + 1));
    for (int b = 0; b < p->B; ++b)
        for (int h = 0; h < p->H; ++h) {
            oracle_attn_bwd_rows(p, q, k, v, dout, b, h, 0, p->sq, a, 0, p->sk, bk, bv);
            for (int i = 0; i < p->sq; ++i)
                memcpy(dq + q_at(p, b, i, h), a + (size_t)i * d, sizeof(double) * d);
            for (int j = 0; j < p->sk; ++j) {
                memcpy(dk + k_at(p, b, j, h), bk + (size_t)j * d, sizeof(double) * d);
                memcpy(dv + k_at(p, b, j, h), bv + (size_t)j * d, sizeof(double) * d);
            }
        }
    free(a);
    free(bk);
    free(bv);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Ulysses regrouping as a scalar copy loop                            */
/*                                                                     */
/* Shard r holds sequence rows [r*s/N, (r+1)*s/N) of all h heads       */
/* (transformers PR 31525 data collator); group g holds heads          */
/* [g*h/N, (g+1)*h/N) of the full sequence ("Parallel multi-head       */
/* attention" section 2.2: contiguous head blocks per device).         */
/* seq-shard buffer:  [N][b][s/N][h][d]                                */
/* head-group buffer: [N][b][s][h/N][d]                                */
/* Elements are opaque 16-bit words: the copy is exact.                */
/* ------------------------------------------------------------------ */

int oracle_seq2head(const uint16_t* in, uint16_t* out, int N, int b, int s, int h, int d)
{
    if (N <= 0 || s % N != 0 || h % N != 0) return 1;
    const int sl = s / N, hl = h / N;
    for (int g = 0; g < N; ++g)
        for (int bb = 0; bb < b; ++bb)
            for (int t = 0; t < s; ++t)
                for (int j = 0; j < hl; ++j)
                    for (int c = 0; c < d; ++c) {
                        const int r = t / sl, u = t % sl, head = g * hl + j;
                        const size_t src = ((((size_t)r * b + bb) * sl + u) * h + head) * d + c;
                        const size_t dst = ((((size_t)g * b + bb) * s + t) * hl + j) * d + c;
                        out[dst] = in[src];
                    }
    return 0;
}

int oracle_head2seq(const uint16_t* in, uint16_t* out, int N, int b, int s, int h, int d)
{
    if (N <= 0 || s % N != 0 || h % N != 0) return 1;
    const int sl = s / N, hl = h / N;
    for (int r = 0; r < N; ++r)
        for (int bb = 0; bb < b; ++bb)
            for (int u = 0; u < sl; ++u)
                for (int head = 0; head < h; ++head)
                    for (int c = 0; c < d; ++c) {
                        const int g = head / hl, j = head % hl, t = r * sl + u;
                        const size_t src = ((((size_t)g * b + bb) * s + t) * hl + j) * d + c;
                        const size_t dst = ((((size_t)r * b + bb) * sl + u) * h + head) * d + c;
                        out[dst] = in[src];
                    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Ring / blockwise attention: combine per-key-chunk results.          */
/* "adv07: Sequence Parallel", sections 5 and 7: K/V blocks travel a   */
/* ring and each device attends to one block at a time.  The pages     */
/* give no combination formula; the softmax over a union of disjoint   */
/* key sets is, row by row, with m = max_k lse_k:                      */
/*     lse = m + log(sum_k exp(lse_k - m))                             */
/*     out = sum_k exp(lse_k - lse) * out_k                            */
/* A chunk with lse_k = -inf contributes nothing; all -inf gives       */
/* out = 0, lse = -inf.                                                */
/* outs: [nparts][B][sq][H][d], lses: [nparts][B][H][sq]; results in   */
/* out [B][sq][H][d] and lse [B][H][sq].                               */
/* ------------------------------------------------------------------ */

int oracle_attn_merge(int B, int H, int sq, int d, int nparts, const double* outs,
                      const double* lses, double* out, double* lse)
{
    if (B < 0 || H < 0 || sq < 0 || d <= 0 || nparts < 1) return 1;
    const size_t out_part = (size_t)B * sq * H * d, lse_part = (size_t)B * H * sq;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < sq; ++i) {
                const size_t li = ((size_t)b * H + h) * sq + i;
                const size_t oi = (((size_t)b * sq + i) * H + h) * d;
                double m = -INFINITY;
                for (int k = 0; k < nparts; ++k)
                    if (lses[k * lse_part + li] > m) m = lses[k * lse_part + li];
                for (int c = 0; c < d; ++c) out[oi + c] = 0.0;
                if (m == -INFINITY) {
                    lse[li] = -INFINITY;
                    continue;
                }
                double s = 0.0;
                for (int k = 0; k < nparts; ++k) s += exp(lses[k * lse_part + li] - m);
                const double total = m + log(s);
                lse[li] = total;
                for (int k = 0; k < nparts; ++k) {
                    const double w = exp(lses[k * lse_part + li] - total);
                    for (int c = 0; c < d; ++c) out[oi + c] += w * outs[k * out_part + oi + c];
                }
            }
    return 0;
}
