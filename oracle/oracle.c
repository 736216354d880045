/*
 * oracle.c -- slow, plain fp64 CPU oracle for exact softmax attention and row softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file:
 * only the tests, the smoke check and the bench's CPU-baseline leg use it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * What it computes (the plain definitions, written out without blocking or fusion):
 *
 *   softmax of a row x:  m = max_j x_j,  l = sum_j exp(x_j - m),  y_j = exp(x_j - m) / l,
 *                        lse = m + ln l.
 *     "How FlashAttention avoids storing the giant score table" (spicyshark.co, Online softmax
 *     lesson), sections "The fix: subtract the maximum" and "The cost: three passes": the safe
 *     softmax needs one pass for the max, one for the sum and one to write the shares.
 *
 *   attention of query row i of head (b,h):
 *        s_j  = scale * sum_k Q[b,h,i,k] * K[b,h,j,k]      for every allowed key j
 *        m    = max_j s_j
 *        l    = sum_j exp(s_j - m)
 *        O_i  = sum_j exp(s_j - m) * V[b,h,j,:] / l
 *        LSE_i = m + ln l
 *     Allowed keys: all j < N, or j <= i when causal, and, with per-sequence key lengths,
 *     only j < kv_len[b] (padding keys carry score -inf like any masked key).  With grouped
 *     heads (H_kv key/value heads shared by H query heads) query head h reads key/value head
 *     h / (H / H_kv).  Same lesson, section "From softmax to
 *     attention" (score = q.k scaled, output = softmax-weighted sum of the values, written in the
 *     max-subtracted form); the masked keys carry score -inf ("The implementation": masked
 *     positions such as the tokens after a token get score -inf).  FlashAttention computes this
 *     exact quantity, only in another order ("kbwen.com FlashAttention" page, section "More than
 *     two blocks": it is the same attention, not an approximation).
 *
 *   softmax with top-k selection: the k entries of a row with the largest x (ties: the smaller
 *     column first), their columns and their shares y_j, and lse.  Same lesson, section "Where
 *     this is used in practice" (the online normaliser serves softmax fused with top-k
 *     selection, keeping only the k largest scores); the shares are the three-pass softmax above
 *     and the selection is a plain sort of the row.
 *
 *   the gradients of the attention (the backward pass): with P the softmax shares above, O the
 *     output and dO the gradient of a loss with respect to O,
 *        dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . V_j,   D_i = dO_i . O_i,
 *        dS_ij = P_ij (dP_ij - D_i),   dQ_i = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
 *     -- the chain rule through O = P V and the softmax (the derivative of a softmax share is
 *     P_ij (delta - P_ik), which summed against dP gives P_ij (dP_ij - sum_k P_ik dP_ik) and
 *     sum_k P_ik dP_ik = dO_i . O_i).  The pages say only that training recomputes the scores in
 *     the backward pass instead of storing them ("FlashAttention" (paweldubiel.com notes),
 *     "Mechanism and details"; the lesson's "Where this is used in practice"); the formulas are
 *     the derivative of the definition, and the tests pin them by finite differences.
 *
 *   the streaming state (m, l, acc) of one score row read in blocks, and the merge of two such
 *   states: same lesson, sections "The idea", "From softmax to attention" (the block recipe)
 *   and the two-worker merge at the end of "From softmax to attention"; "kbwen.com
 *   FlashAttention" page, sections "Two blocks" and "More than two blocks".  These are the
 *   pages' algorithm restated step by step in the pages' order and notation; the oracle uses
 *   them only to reproduce the pages' worked tables and laws, never to produce the reference
 *   outputs of the attention or softmax (those come from the three-pass definitions above).
 *
 * Readings where the pages are silent (each listed in the design notes of the repository):
 *   - LSE is the natural-log log-sum-exp of the SCALED scores, m + ln l.
 *   - a row with no allowed key (all -inf) has y = 0 / O = 0 and lse = -inf: the -inf guard of
 *     the lesson's "The implementation" section says such a block "adds nothing", and the merge
 *     of an empty state keeps the other state.
 *   - bf16 inputs are widened exactly (bits << 16) to fp32, then to fp64.
 *
 * Mutants: building with -DORACLE_MUTANT=k plants one deliberate mistake (k = 1..18) so the
 * tests can show that the pins catch it.  The default build (no define) has none.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_ABI_VERSION 1

int oracle_abi_version(void) { return ORACLE_ABI_VERSION; }
int oracle_mutant(void) { return ORACLE_MUTANT; }

/* bf16 bit pattern -> exact double. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1) n = 1;
    if (n > 256) n = 256;
    return (int)n;
}

/* ------------------------------------------------------------------------------------------ */
/* Row softmax, three passes per row.                                                          */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const float* x;
    double* y;
    double* lse;
    int64_t cols;
    int64_t r0, r1;
} softmax_job;

static void softmax_one_row(const float* x, double* y, double* lse, int64_t cols) {
    /* pass 1: the maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < cols; ++j) {
        double v = (double)x[j];
        if (v > m || isnan(v)) m = v;
    }
    if (cols == 0 || m == -INFINITY) {
        /* no finite entry: nothing is allowed, every share is 0 and the log-sum-exp is -inf */
        for (int64_t j = 0; j < cols; ++j) y[j] = 0.0;
        if (lse) *lse = -INFINITY;
        return;
    }
    /* pass 2: the sum of exp(x - m) */
    double l = 0.0;
    for (int64_t j = 0; j < cols; ++j) {
#if ORACLE_MUTANT == 1
        l += exp((double)x[j]); /* mutant: forgets the max in the sum */
#else
        l += exp((double)x[j] - m);
#endif
    }
    /* pass 3: the shares */
    for (int64_t j = 0; j < cols; ++j) y[j] = exp((double)x[j] - m) / l;
    if (lse) *lse = m + log(l);
}

static void* softmax_worker(void* arg) {
    softmax_job* jb = (softmax_job*)arg;
    for (int64_t r = jb->r0; r < jb->r1; ++r)
        softmax_one_row(jb->x + r * jb->cols, jb->y + r * jb->cols, jb->lse ? jb->lse + r : NULL,
                        jb->cols);
    return NULL;
}

/* y[rows*cols], lse[rows] (lse may be NULL). Returns 0, or -1 on bad arguments. */
int oracle_softmax_rows(const float* x, int64_t rows, int64_t cols, double* y, double* lse,
                        int nthreads) {
    if (rows < 0 || cols < 0) return -1;
    if (rows == 0) return 0;
    if (!x || !y) return -1;
    int nt = resolve_threads(nthreads);
    if (nt > rows) nt = (int)rows;
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    softmax_job* jobs = (softmax_job*)calloc((size_t)nt, sizeof(softmax_job));
    if (!th || !jobs) { free(th); free(jobs); return -1; }
    for (int t = 0; t < nt; ++t) {
        jobs[t].x = x; jobs[t].y = y; jobs[t].lse = lse; jobs[t].cols = cols;
        jobs[t].r0 = rows * t / nt;
        jobs[t].r1 = rows * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, softmax_worker, &jobs[t]);
    softmax_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    free(th); free(jobs);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Softmax with top-k selection.                                                               */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    float x;
    int64_t j;
} ranked;

/* x descending, then column ascending */
static int rank_cmp(const void* a, const void* b) {
    const ranked* p = (const ranked*)a;
    const ranked* q = (const ranked*)b;
    if (p->x > q->x) return -1;
    if (p->x < q->x) return 1;
#if ORACLE_MUTANT == 14
    return (p->j > q->j) ? -1 : (p->j < q->j); /* mutant: ties go to the larger column */
#else
    return (p->j < q->j) ? -1 : (p->j > q->j);
#endif
}

typedef struct {
    const float* x;
    int64_t cols, k;
    double* values;
    int64_t* indices;
    double* lse;
    int64_t r0, r1;
    int err;
} topk_job;

static void* topk_worker(void* arg) {
    topk_job* jb = (topk_job*)arg;
    double* y = (double*)malloc(sizeof(double) * (size_t)jb->cols);
    ranked* order = (ranked*)malloc(sizeof(ranked) * (size_t)jb->cols);
    if (!y || !order) { jb->err = 1; free(y); free(order); return NULL; }
    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        const float* xr = jb->x + r * jb->cols;
        double lse;
        softmax_one_row(xr, y, &lse, jb->cols);
        if (jb->lse) jb->lse[r] = lse;
        for (int64_t j = 0; j < jb->cols; ++j) { order[j].x = xr[j]; order[j].j = j; }
        qsort(order, (size_t)jb->cols, sizeof(ranked), rank_cmp);
        for (int64_t t = 0; t < jb->k; ++t) {
#if ORACLE_MUTANT == 15
            const int64_t pick = (t + 1 < jb->cols) ? t + 1 : t; /* mutant: skips the largest */
#else
            const int64_t pick = t;
#endif
            jb->indices[r * jb->k + t] = order[pick].j;
            jb->values[r * jb->k + t] = y[order[pick].j];
        }
    }
    free(y); free(order);
    return NULL;
}

/* x [rows, cols] fp32 (no NaN); values [rows, k] fp64, indices [rows, k] int64, lse [rows] or
   NULL.  1 <= k <= cols.  Returns 0, or -1 on bad arguments. */
int oracle_softmax_topk(const float* x, int64_t rows, int64_t cols, int64_t k, double* values,
                        int64_t* indices, double* lse, int nthreads) {
    if (rows < 0 || cols < 1 || k < 1 || k > cols) return -1;
    if (rows == 0) return 0;
    if (!x || !values || !indices) return -1;
    int nt = resolve_threads(nthreads);
    if (nt > rows) nt = (int)rows;
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    topk_job* jobs = (topk_job*)calloc((size_t)nt, sizeof(topk_job));
    if (!th || !jobs) { free(th); free(jobs); return -1; }
    for (int t = 0; t < nt; ++t) {
        jobs[t].x = x; jobs[t].cols = cols; jobs[t].k = k; jobs[t].values = values;
        jobs[t].indices = indices; jobs[t].lse = lse;
        jobs[t].r0 = rows * t / nt;
        jobs[t].r1 = rows * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, topk_worker, &jobs[t]);
    topk_worker(&jobs[0]);
    int err = 0;
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nt; ++t) err |= jobs[t].err;
    free(th); free(jobs);
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Attention, three passes per query row.                                                      */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *Q, *K, *V;
    int64_t H, H_kv, N, Nk, d; /* N = queries per head, Nk = keys per head */
    double scale;
    int causal;
    const int32_t* kv_lens; /* NULL, or [B] valid keys per sequence */
    const uint8_t* mask;    /* NULL, or 1 = key allowed, [b*mask_bs + h*mask_hs + i*Nk + j] */
    int64_t mask_bs, mask_hs;
    const int64_t* rows; /* NULL: rows [r0, r1) of the flat (b*H+h)*N+i index */
    double *O, *LSE;
    int64_t r0, r1;
    int err;
} attn_job;

/* One query row.  `flat` = (b*H + h)*N + i.  s and q are scratch of Nk and d doubles. */
static void attn_one_row(const attn_job* jb, int64_t flat, double* o, double* lse_out,
                         double* s, double* q) {
    const int64_t N = jb->N, Nk = jb->Nk, d = jb->d;
    const int64_t bh = flat / N;
    const int64_t i = flat % N;
    const int64_t b = bh / jb->H, h = bh % jb->H;
#if ORACLE_MUTANT == 12
    const int64_t hk = h % jb->H_kv; /* mutant: query heads dealt round-robin to K/V heads */
#else
    const int64_t hk = h / (jb->H / jb->H_kv); /* the K/V head this query head shares */
#endif
    const int64_t bhk = b * jb->H_kv + hk;
    const uint16_t* Qh = jb->Q + bh * N * d;
    const uint16_t* Kh = jb->K + bhk * Nk * d;
    const uint16_t* Vh = jb->V + bhk * Nk * d;

    for (int64_t k = 0; k < d; ++k) q[k] = bf16_to_double(Qh[i * d + k]);

    /* number of allowed keys: all Nk, or, causal, the keys up to the query's own position when
       the N queries are the last N of the Nk positions (query i sits at position i + Nk - N) */
    int64_t nk = Nk;
    if (jb->causal) {
#if ORACLE_MUTANT == 2
        nk = i + (Nk - N);     /* mutant: strict causal mask (j < position) */
#else
        nk = i + (Nk - N) + 1; /* key j <= position of query i */
#endif
        if (nk < 0) nk = 0;
        if (nk > Nk) nk = Nk;
    }
#if ORACLE_MUTANT == 3
    if (nk > 1) nk -= 1; /* mutant: drops the last allowed key */
#endif
    /* keys past the sequence's own length are padding */
#if ORACLE_MUTANT != 13 /* mutant 13: ignores the key lengths */
    if (jb->kv_lens && nk > jb->kv_lens[b]) nk = jb->kv_lens[b] > 0 ? jb->kv_lens[b] : 0;
#endif

    /* an explicit mask: keys whose entry is 0 take no part (score -inf) */
    const uint8_t* mrow = jb->mask ? jb->mask + b * jb->mask_bs + h * jb->mask_hs + i * Nk : NULL;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
#if ORACLE_MUTANT == 19 /* mutant 19: ignores the explicit mask */
        (void)mrow;
#elif ORACLE_MUTANT == 20 /* mutant 20: reads the mask transposed (entry j, i) */
        if (mrow && j < N && i < Nk &&
            !jb->mask[b * jb->mask_bs + h * jb->mask_hs + j * Nk + i]) {
            s[j] = -INFINITY;
            continue;
        }
#else
        if (mrow && !mrow[j]) {
            s[j] = -INFINITY;
            continue;
        }
#endif
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k) {
#if ORACLE_MUTANT == 4
            /* mutant: reads K transposed (column j of a d x Nk view) */
            double kv = bf16_to_double(Kh[(k * Nk + j) % (Nk * d)]);
#else
            double kv = bf16_to_double(Kh[j * d + k]);
#endif
            acc += q[k] * kv;
        }
#if ORACLE_MUTANT == 5
        s[j] = acc; /* mutant: forgets the scale */
#else
        s[j] = jb->scale * acc;
#endif
        if (s[j] > m || isnan(s[j])) m = s[j];
    }
    if (nk == 0 || m == -INFINITY) {
        for (int64_t k = 0; k < d; ++k) o[k] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* pass 2: the normaliser l = sum_j exp(s_j - m) */
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j) l += exp(s[j] - m);
    /* pass 3: the weighted sum of the values, divided by l */
    for (int64_t k = 0; k < d; ++k) o[k] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
#if ORACLE_MUTANT == 6
        double p = exp(m - s[j]); /* mutant: sign error in the exponent */
#else
        double p = exp(s[j] - m);
#endif
        const uint16_t* vj = Vh + j * d;
        for (int64_t k = 0; k < d; ++k) o[k] += p * bf16_to_double(vj[k]);
    }
    for (int64_t k = 0; k < d; ++k) o[k] /= l;
#if ORACLE_MUTANT == 7
    *lse_out = m + log2(l); /* mutant: log base 2 in the log-sum-exp */
#else
    *lse_out = m + log(l);
#endif
}

static void* attn_worker(void* arg) {
    attn_job* jb = (attn_job*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    double* q = (double*)malloc(sizeof(double) * (size_t)(jb->d > 0 ? jb->d : 1));
    if (!s || !q) { jb->err = 1; free(s); free(q); return NULL; }
    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        int64_t flat = jb->rows ? jb->rows[r] : r;
        attn_one_row(jb, flat, jb->O + r * jb->d, jb->LSE + r, s, q);
    }
    free(s); free(q);
    return NULL;
}

/*
 * Q: bf16 bit patterns [B, H, Nq, d]; K, V: [B, H_kv, Nk, d]; all contiguous; H_kv divides H
 * and query head h reads key/value head h / (H / H_kv).
 * Query i of a head attends to keys j < Nk, or, when causal, to keys j <= i + (Nk - Nq) (the
 * Nq queries are the last Nq of the Nk positions; Nq == Nk is the usual square mask), and, when
 * kv_lens is given, only to keys j < kv_lens[b], and, when mask is given (uint8, 1 = allowed),
 * only to keys with mask[b*mask_bs + h*mask_hs + i*Nk + j] != 0 (a stride of 0 repeats the
 * mask over batches or heads).  A row with no allowed key gets O = 0 and LSE = -inf.
 * rows == NULL: compute all B*H*Nq rows; O is [B*H*Nq, d] and LSE [B*H*Nq].
 * rows != NULL: compute the nrows listed flat row indices (b*H + h)*Nq + i; O is [nrows, d].
 * Returns 0, or -1 on bad arguments (including a listed row out of range).
 */
int oracle_attn4(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B, int64_t H,
                 int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d, double scale, int causal,
                 const int32_t* kv_lens, const uint8_t* mask, int64_t mask_bs, int64_t mask_hs,
                 const int64_t* rows, int64_t nrows, double* O, double* LSE, int nthreads) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 1) return -1;
    if (H > 0 && (H_kv < 1 || H % H_kv != 0)) return -1;
    const int64_t total = B * H * Nq;
    const int64_t n = rows ? nrows : total;
    if (n < 0) return -1;
    if (n == 0) return 0;
    if (!Q || !O || !LSE || (Nk > 0 && (!K || !V))) return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return -1;
    int nt = resolve_threads(nthreads);
    if (nt > n) nt = (int)n;
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    attn_job* jobs = (attn_job*)calloc((size_t)nt, sizeof(attn_job));
    if (!th || !jobs) { free(th); free(jobs); return -1; }
    for (int t = 0; t < nt; ++t) {
        attn_job* jb = &jobs[t];
        jb->Q = Q; jb->K = K; jb->V = V; jb->H = H; jb->H_kv = H_kv; jb->N = Nq; jb->Nk = Nk;
        jb->d = d; jb->scale = scale; jb->causal = causal; jb->kv_lens = kv_lens;
        jb->mask = mask; jb->mask_bs = mask_bs; jb->mask_hs = mask_hs;
        jb->rows = rows; jb->O = O; jb->LSE = LSE;
        jb->r0 = n * t / nt;
        jb->r1 = n * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    attn_worker(&jobs[0]);
    int err = 0;
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nt; ++t) err |= jobs[t].err;
    free(th); free(jobs);
    return err ? -1 : 0;
}

/* As oracle_attn4 without an explicit mask. */
int oracle_attn3(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B, int64_t H,
                 int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d, double scale, int causal,
                 const int32_t* kv_lens, const int64_t* rows, int64_t nrows, double* O,
                 double* LSE, int nthreads) {
    return oracle_attn4(Q, K, V, B, H, H_kv, Nq, Nk, d, scale, causal, kv_lens, NULL, 0, 0, rows,
                        nrows, O, LSE, nthreads);
}

/* ------------------------------------------------------------------------------------------ */
/* Attention gradients.                                                                        */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *Q, *K, *V, *dO;
    int64_t H, H_kv, N, d;
    double scale;
    int causal;
    const int32_t* kv_lens; /* [B] valid keys per sequence, or NULL (all N) */
    double *dQ, *dK, *dV;
    int64_t g0, g1; /* key/value heads [g0, g1) of the flat (b*H_kv + hk) index */
    int err;
} bwd_job;

static void* bwd_worker(void* arg) {
    bwd_job* jb = (bwd_job*)arg;
    const int64_t N = jb->N, d = jb->d, group = jb->H / jb->H_kv;
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    double* g = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !q || !o || !g) { jb->err = 1; free(s); free(q); free(o); free(g); return NULL; }
    for (int64_t bhk = jb->g0; bhk < jb->g1; ++bhk) {
        const int64_t b = bhk / jb->H_kv, hk = bhk % jb->H_kv;
        const uint16_t* Kh = jb->K + bhk * N * d;
        const uint16_t* Vh = jb->V + bhk * N * d;
        double* dKh = jb->dK + bhk * N * d;
        double* dVh = jb->dV + bhk * N * d;
        for (int64_t t = 0; t < N * d; ++t) { dKh[t] = 0.0; dVh[t] = 0.0; }
        /* keys j < len of this sequence take part */
        int64_t len = N;
#if ORACLE_MUTANT != 22
        if (jb->kv_lens) {
            len = jb->kv_lens[b];
            if (len < 0) len = 0;
            if (len > N) len = N;
        }
#endif
        /* the query heads that share this key/value head: their key and value gradients add */
        for (int64_t hq = hk * group; hq < (hk + 1) * group; ++hq) {
            const int64_t bh = b * jb->H + hq;
            const uint16_t* Qh = jb->Q + bh * N * d;
            const uint16_t* Gh = jb->dO + bh * N * d;
            double* dQh = jb->dQ + bh * N * d;
            for (int64_t t = 0; t < N * d; ++t) dQh[t] = 0.0;
#if ORACLE_MUTANT == 21
            /* mutant: the shared head keeps only the last query head's part */
            for (int64_t t = 0; t < N * d; ++t) { dKh[t] = 0.0; dVh[t] = 0.0; }
#endif
            for (int64_t i = 0; i < N; ++i) {
                int64_t nk = jb->causal ? i + 1 : N;
                if (nk > len) nk = len;
                if (nk == 0) continue; /* no allowed key: O_i = 0 and the row adds nothing */
                for (int64_t k = 0; k < d; ++k) {
                    q[k] = bf16_to_double(Qh[i * d + k]);
                    g[k] = bf16_to_double(Gh[i * d + k]);
                }
                /* the shares P_ij of row i (three passes, as the forward definition) */
                double m = -INFINITY;
                for (int64_t j = 0; j < nk; ++j) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < d; ++k) acc += q[k] * bf16_to_double(Kh[j * d + k]);
                    s[j] = jb->scale * acc;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j < nk; ++j) l += exp(s[j] - m);
                for (int64_t j = 0; j < nk; ++j) s[j] = exp(s[j] - m) / l; /* s holds P_ij */
                /* O_i and D_i = dO_i . O_i */
                for (int64_t k = 0; k < d; ++k) o[k] = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    for (int64_t k = 0; k < d; ++k) o[k] += s[j] * bf16_to_double(Vh[j * d + k]);
                double D = 0.0;
                for (int64_t k = 0; k < d; ++k) D += g[k] * o[k];
#if ORACLE_MUTANT == 16
                D = 0.0; /* mutant: drops the D_i term */
#endif
                for (int64_t j = 0; j < nk; ++j) {
                    const double p = s[j];
                    double dp = 0.0;
                    for (int64_t k = 0; k < d; ++k) {
                        dp += g[k] * bf16_to_double(Vh[j * d + k]);
                        dVh[j * d + k] += p * g[k];
                    }
#if ORACLE_MUTANT == 17
                    const double ds = p * (D - dp); /* mutant: sign of dS flipped */
#else
                    const double ds = p * (dp - D);
#endif
#if ORACLE_MUTANT == 18
                    const double sc = 1.0; /* mutant: forgets the scale in dQ and dK */
#else
                    const double sc = jb->scale;
#endif
                    for (int64_t k = 0; k < d; ++k) {
                        dQh[i * d + k] += sc * ds * bf16_to_double(Kh[j * d + k]);
                        dKh[j * d + k] += sc * ds * q[k];
                    }
                }
            }
        }
    }
    free(s); free(q); free(o); free(g);
    return NULL;
}

/*
 * Gradients of O = softmax(scale Q K^T [mask]) V with respect to Q, K and V for the output
 * gradient dO, the derivative of the definition (the backward pass of "FlashAttention"
 * (paweldubiel.com notes), "Mechanism and details"): per row, P = the softmax shares,
 * D_i = dO_i . O_i, dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij k_j,
 * dK_j = scale sum_i dS_ij q_i, dV_j = sum_i P_ij dO_i.  Q, dO: bf16 bit patterns [B, H, N, d];
 * K, V: [B, H_kv, N, d] with H_kv dividing H (query head h reads key/value head h / (H / H_kv),
 * and the key and value gradients of a shared head sum over its query heads); kv_lens: NULL or
 * int32 [B], keys j >= kv_lens[b] excluded (clamped to [0, N]); causal: key j allowed for query
 * i only when j <= i.  A row with no allowed key contributes nothing (dQ_i = 0).  dQ fp64
 * [B, H, N, d]; dK, dV fp64 [B, H_kv, N, d].  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_bwd2(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                     const uint16_t* dO, int64_t B, int64_t H, int64_t H_kv, int64_t N, int64_t d,
                     double scale, int causal, const int32_t* kv_lens, double* dQ, double* dK,
                     double* dV, int nthreads) {
    if (B < 0 || H < 0 || H_kv < 1 || N < 0 || d < 1 || (H > 0 && H % H_kv != 0)) return -1;
    const int64_t kv_heads = B * H_kv;
    if (B * H == 0 || N == 0) return 0;
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return -1;
    int nt = resolve_threads(nthreads);
    if (nt > kv_heads) nt = (int)kv_heads;
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    bwd_job* jobs = (bwd_job*)calloc((size_t)nt, sizeof(bwd_job));
    if (!th || !jobs) { free(th); free(jobs); return -1; }
    for (int t = 0; t < nt; ++t) {
        bwd_job* jb = &jobs[t];
        jb->Q = Q; jb->K = K; jb->V = V; jb->dO = dO; jb->H = H; jb->H_kv = H_kv; jb->N = N;
        jb->d = d; jb->scale = scale; jb->causal = causal; jb->kv_lens = kv_lens;
        jb->dQ = dQ; jb->dK = dK; jb->dV = dV;
        jb->g0 = kv_heads * t / nt;
        jb->g1 = kv_heads * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, bwd_worker, &jobs[t]);
    bwd_worker(&jobs[0]);
    int err = 0;
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nt; ++t) err |= jobs[t].err;
    free(th); free(jobs);
    return err ? -1 : 0;
}

/* Every query head with its own key/value head, every key valid. */
int oracle_attn_bwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const uint16_t* dO,
                    int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                    double* dQ, double* dK, double* dV, int nthreads) {
    return oracle_attn_bwd2(Q, K, V, dO, B, H, H, N, d, scale, causal, NULL, dQ, dK, dV,
                            nthreads);
}

/* Every query head with its own key/value head, every key valid. */
int oracle_attn2(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B, int64_t H,
                 int64_t Nq, int64_t Nk, int64_t d, double scale, int causal, const int64_t* rows,
                 int64_t nrows, double* O, double* LSE, int nthreads) {
    return oracle_attn3(Q, K, V, B, H, H, Nq, Nk, d, scale, causal, NULL, rows, nrows, O, LSE,
                        nthreads);
}

/* Square attention: queries and keys are the same N positions. */
int oracle_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B, int64_t H,
                int64_t N, int64_t d, double scale, int causal, const int64_t* rows,
                int64_t nrows, double* O, double* LSE, int nthreads) {
    return oracle_attn2(Q, K, V, B, H, N, N, d, scale, causal, rows, nrows, O, LSE, nthreads);
}

/* ------------------------------------------------------------------------------------------ */
/* The streaming state of one score row, block by block, and the merge of two states.          */
/* ------------------------------------------------------------------------------------------ */

/*
 * Reads the n scores s[] with their value rows v[n*dv] in blocks of `block` and keeps the
 * state (m, l, acc): m the largest score so far, l = sum exp(s_j - m), acc = sum exp(s_j - m)
 * v_j over the scores read so far.  Per block: m_new = max(m, max of the block); a block that
 * leaves m_new = -inf adds nothing; alpha = exp(m - m_new) rescales l and acc alike; the block's
 * own terms p = exp(s - m_new) are added.
 *
 * If trace arrays are given they receive the state after every block (ceil(n/block) entries;
 * trace_acc has dv per entry): m, alpha used, the block's own sum of p, l, acc.  A block that
 * was skipped by the -inf guard records alpha = NAN (no rescale happened) and psum = 0.
 * Returns the number of blocks, or -1 on bad arguments.
 */
int64_t oracle_online_state(const double* s, const double* v, int64_t n, int64_t dv,
                            int64_t block, double* m_out, double* l_out, double* acc_out,
                            double* trace_m, double* trace_alpha, double* trace_psum,
                            double* trace_l, double* trace_acc) {
    if (n < 0 || dv < 0 || block < 1 || !m_out || !l_out) return -1;
    if (dv > 0 && (!acc_out || (n > 0 && !v))) return -1;
    double m = -INFINITY, l = 0.0;
    for (int64_t k = 0; k < dv; ++k) acc_out[k] = 0.0;
    int64_t nb = 0;
    for (int64_t i0 = 0; i0 < n; i0 += block, ++nb) {
        int64_t i1 = i0 + block < n ? i0 + block : n;
        double bmax = -INFINITY;
        for (int64_t j = i0; j < i1; ++j)
            if (s[j] > bmax) bmax = s[j];
        double m_new = m > bmax ? m : bmax;
        double alpha = NAN, psum = 0.0;
#if ORACLE_MUTANT == 10
        int skip = 0; /* mutant: no -inf guard */
#else
        int skip = (m_new == -INFINITY); /* nothing finite yet: the block adds nothing */
#endif
        if (!skip) {
#if ORACLE_MUTANT == 9
            double m_p = (m == -INFINITY) ? m_new : m; /* mutant: p against the old max */
#else
            double m_p = m_new;
#endif
            alpha = exp(m - m_new);
            for (int64_t j = i0; j < i1; ++j) psum += exp(s[j] - m_p);
#if ORACLE_MUTANT == 8
            l = l + psum; /* mutant: drops the rescale of l */
#else
            l = l * alpha + psum;
#endif
            for (int64_t k = 0; k < dv; ++k) {
                double add = 0.0;
                for (int64_t j = i0; j < i1; ++j) add += exp(s[j] - m_p) * v[j * dv + k];
                acc_out[k] = acc_out[k] * alpha + add;
            }
            m = m_new;
        }
        if (trace_m) trace_m[nb] = m;
        if (trace_alpha) trace_alpha[nb] = alpha;
        if (trace_psum) trace_psum[nb] = psum;
        if (trace_l) trace_l[nb] = l;
        if (trace_acc)
            for (int64_t k = 0; k < dv; ++k) trace_acc[nb * dv + k] = acc_out[k];
    }
    *m_out = m;
    *l_out = l;
    return nb;
}

/*
 * Merge of two states built from disjoint parts of one row: m = max(m_a, m_b); each side's l
 * and acc are rescaled by exp(its m - m) and added.  If both are empty (m = -inf) the result is
 * state a.  Output may alias either input.
 */
int oracle_merge(double m_a, double l_a, const double* acc_a, double m_b, double l_b,
                 const double* acc_b, int64_t dv, double* m_out, double* l_out,
                 double* acc_out) {
    if (dv < 0 || !m_out || !l_out || (dv > 0 && (!acc_a || !acc_b || !acc_out))) return -1;
    double m = m_a > m_b ? m_a : m_b;
    if (m == -INFINITY) {
        *m_out = m_a;
        *l_out = l_a;
        for (int64_t k = 0; k < dv; ++k) acc_out[k] = acc_a[k];
        return 0;
    }
    double wa = exp(m_a - m), wb = exp(m_b - m);
    *m_out = m;
#if ORACLE_MUTANT == 11
    wb = wa; /* mutant: weighs both sides by the first side's factor */
#endif
    *l_out = l_a * wa + l_b * wb;
    for (int64_t k = 0; k < dv; ++k) acc_out[k] = acc_a[k] * wa + acc_b[k] * wb;
    return 0;
}
