/*
 * splash_oracle.c -- the CPU oracle for block-sparse (Splash-style) masked
 * attention: mask tables, forward pass and backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, __graft_entry__.smoke() and the CPU-baseline leg
 * of bench.py do.  It shares no code, header, table or constant with the CUDA
 * library under block_sparse_flash_gb300/.
 *
 * It is deliberately plain and slow: every floating-point value is an IEEE
 * double, every block is classified by looking at every one of its elements,
 * and attention is computed by materialising score panels, masking them and
 * running a two-pass (max, then sum) softmax.
 *
 * Sources (cited by page title and section):
 *   [L13]  "Pallas Kernels and Splash Attention" -- CMU 11-868 Lecture 13
 *          study notes (semidirectx.com).
 *   [OPS]  "The maths and infra behind core LLM operations" (joto.ai blog:
 *          RMSNorm / Softmax / Causal Mask / Sampling).
 *
 * Readings taken where the pages leave a step open (each is restated in the
 * design notes of the repository):
 *   - joint mask = AND of causal, local window and segment equality [L13 §6.4];
 *   - causal keeps key j <= query i, both 0-based from the same origin;
 *   - the local window is given as inclusive (left, right) distances; a
 *     negative distance means "unbounded on that side";
 *   - masked scores are excluded from the softmax (the -inf reading of
 *     [OPS] "Causal Mask"), so a row with no allowed key has O = 0 and
 *     LSE = -inf;
 *   - the scale multiplies q.k before the soft cap: s = cap*tanh(scale*q.k/cap)
 *     [L13 §5.2 step 2 and §5.4];
 *   - LSE is the natural-log log-sum-exp of the scaled (and capped) scores,
 *     LSE = m + ln(l) [OPS] "LSE and Online Softmax";
 *   - a GQA query head h reads key/value head h / (Hq/Hkv) [L13 §5.2];
 *   - lengths that are not a multiple of the block: the block grid is padded
 *     to whole blocks and padding positions are masked [L13 §2.3], so a block
 *     with padding is never full;
 *   - MaskInfo: block class 0 = empty, 1 = partial, 2 = full; active blocks in
 *     row-major order (q-block ascending, then kv-block ascending); bounds
 *     flags mark the first and last active block of each q-block row; partial
 *     patterns are deduplicated by exact content in first-occurrence order;
 *     mask_next is -1 for full blocks [L13 §6.2, §6.3].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2
#define ORACLE_ERR_CAPACITY 3

/* The mask specification.  Segment arrays are host arrays of shape
 * [batch][Lq] and [batch][Lk]; when q_seg is NULL there is no document mask
 * and one MaskInfo serves every batch row. */
typedef struct {
    int32_t causal;
    int64_t window_left;
    int64_t window_right;
    const int32_t *q_seg;
    const int32_t *kv_seg;
    int32_t batch;
} oracle_mask_spec;

/* ------------------------------------------------------------------------ */
/* The joint mask predicate.                                                 */
/* [L13 §6.1] causal / local masks; [L13 §6.4] segment IDs allow only       */
/* q_id == kv_id, and masks are joined by logical AND.                       */
/* ------------------------------------------------------------------------ */
static int allowed(const oracle_mask_spec *sp, int64_t b, int64_t Lq, int64_t Lk,
                   int64_t i, int64_t j)
{
    if (sp->causal && j > i) return 0;
    if (sp->window_left >= 0 && i - j > sp->window_left) return 0;
    if (sp->window_right >= 0 && j - i > sp->window_right) return 0;
    if (sp->q_seg != NULL && sp->q_seg[b * Lq + i] != sp->kv_seg[b * Lk + j]) return 0;
    return 1;
}

int oracle_allowed(const oracle_mask_spec *sp, int64_t b, int64_t Lq, int64_t Lk,
                   int64_t i, int64_t j)
{
    return allowed(sp, b, Lq, Lk, i, j);
}

/* The predicate on the padded block grid: when Lq or Lk is not a multiple of
 * the block, the last q-block / kv-block extends past the sequence and its
 * padding positions are masked ([L13 §2.3]: ragged edges are padded so that
 * every block has the same size; padding contributes nothing). */
static int allowed_padded(const oracle_mask_spec *sp, int64_t b, int64_t Lq, int64_t Lk,
                          int64_t i, int64_t j)
{
    if (i >= Lq || j >= Lk) return 0;
    return allowed(sp, b, Lq, Lk, i, j);
}

static int64_t ceil_div(int64_t a, int64_t b)
{
    return (a + b - 1) / b;
}

static int64_t batch_rows_of(const oracle_mask_spec *sp)
{
    return sp->q_seg != NULL ? sp->batch : 1;
}

/* ------------------------------------------------------------------------ */
/* MaskInfo, phase 1: classify every block by counting its allowed elements.  */
/* [L13 §6.1]: a block is empty (nothing to compute), full (no mask needed)  */
/* or partial (element mask needed).                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    const oracle_mask_spec *sp;
    int64_t Lq, Lk, bq, bk, nq, nk, nbm;
    int8_t *block_mask;
    int64_t *block_count; /* allowed elements per block */
    int64_t next;         /* next block-row to take */
    pthread_mutex_t mu;
} classify_job;

static void *classify_worker(void *arg)
{
    classify_job *jb = (classify_job *)arg;
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t row = jb->next++;
        pthread_mutex_unlock(&jb->mu);
        if (row >= jb->nbm * jb->nq) break;
        int64_t bm = row / jb->nq, r = row % jb->nq;
        for (int64_t c = 0; c < jb->nk; ++c) {
            int64_t n = 0;
            for (int64_t i = r * jb->bq; i < (r + 1) * jb->bq; ++i)
                for (int64_t j = c * jb->bk; j < (c + 1) * jb->bk; ++j)
                    n += allowed_padded(jb->sp, bm, jb->Lq, jb->Lk, i, j);
            int8_t cls = (n == 0) ? 0 : (n == jb->bq * jb->bk ? 2 : 1);
            jb->block_mask[row * jb->nk + c] = cls;
            jb->block_count[row * jb->nk + c] = n;
        }
    }
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fn, job) != 0) break;
        ++started;
    }
    if (started == 0) fn(job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return ORACLE_OK;
}

/* Fills block_mask[nbm][nq][nk] and returns the totals.  allowed_pairs is the
 * number of allowed (query, key) pairs summed over the MaskInfo batch rows. */
int oracle_mask_classify(const oracle_mask_spec *sp, int64_t Lq, int64_t Lk, int64_t bq,
                         int64_t bk, int nthreads, int8_t *block_mask,
                         int64_t *num_active, int64_t *num_partial, int64_t *allowed_pairs)
{
    if (!sp || !block_mask || bq <= 0 || bk <= 0 || Lq <= 0 || Lk <= 0) return ORACLE_ERR_ARG;
    if (sp->q_seg != NULL && (sp->kv_seg == NULL || sp->batch <= 0)) return ORACLE_ERR_ARG;
    classify_job jb;
    jb.sp = sp; jb.Lq = Lq; jb.Lk = Lk; jb.bq = bq; jb.bk = bk;
    jb.nq = ceil_div(Lq, bq); jb.nk = ceil_div(Lk, bk); jb.nbm = batch_rows_of(sp);
    jb.block_mask = block_mask;
    jb.block_count = (int64_t *)malloc(sizeof(int64_t) * (size_t)(jb.nbm * jb.nq * jb.nk));
    if (!jb.block_count) return ORACLE_ERR_NOMEM;
    jb.next = 0;
    pthread_mutex_init(&jb.mu, NULL);
    run_threads(classify_worker, &jb, nthreads);
    pthread_mutex_destroy(&jb.mu);
    int64_t a = 0, p = 0, n = 0, nb = jb.nbm * jb.nq * jb.nk;
    for (int64_t x = 0; x < nb; ++x) {
        a += block_mask[x] != 0;
        p += block_mask[x] == 1;
        n += jb.block_count[x];
    }
    free(jb.block_count);
    *num_active = a; *num_partial = p; *allowed_pairs = n;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* MaskInfo, phase 2: the sparse execution table [L13 §6.2, §6.3].            */
/* Walks block_mask in row-major order and writes the active lists, the row  */
/* pointers (CSR; row_ptr[r] .. row_ptr[r+1]-1 are row r's active blocks),    */
/* the bounds flags, and the deduplicated partial patterns.                   */
/* Arrays are caller-allocated: active arrays hold num_active entries,        */
/* patterns hold pattern_capacity blocks of bq*bk bytes.                      */
/* ------------------------------------------------------------------------ */
static uint64_t fnv1a(const uint8_t *p, size_t n)
{
    uint64_t h = 1469598103934665603ULL;
    for (size_t x = 0; x < n; ++x) { h ^= p[x]; h *= 1099511628211ULL; }
    return h;
}

int oracle_mask_table(const oracle_mask_spec *sp, int64_t Lq, int64_t Lk, int64_t bq, int64_t bk,
                      const int8_t *block_mask, int32_t *row_ptr, int32_t *active_rows,
                      int32_t *active_cols, int32_t *mask_next, uint8_t *bounds_start,
                      uint8_t *bounds_end, uint8_t *patterns, int64_t pattern_capacity,
                      int64_t *num_patterns)
{
    if (!sp || !block_mask || !row_ptr || bq <= 0 || bk <= 0 || Lq <= 0 || Lk <= 0)
        return ORACLE_ERR_ARG;
    int64_t nq = ceil_div(Lq, bq), nk = ceil_div(Lk, bk), nbm = batch_rows_of(sp);
    size_t pbytes = (size_t)(bq * bk);
    uint8_t *cand = (uint8_t *)malloc(pbytes);
    uint64_t *hashes = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(pattern_capacity > 0 ? pattern_capacity : 1));
    if (!cand || !hashes) { free(cand); free(hashes); return ORACLE_ERR_NOMEM; }
    int64_t g = 0, P = 0;
    for (int64_t bm = 0; bm < nbm; ++bm) {
        for (int64_t r = 0; r < nq; ++r) {
            int64_t row = bm * nq + r;
            row_ptr[row] = (int32_t)g;
            int64_t first = g;
            for (int64_t c = 0; c < nk; ++c) {
                int8_t cls = block_mask[row * nk + c];
                if (cls == 0) continue;
                active_rows[g] = (int32_t)r;
                active_cols[g] = (int32_t)c;
                mask_next[g] = -1;
                if (cls == 1) {
                    /* the element pattern: row = query offset, col = key offset */
                    for (int64_t di = 0; di < bq; ++di)
                        for (int64_t dj = 0; dj < bk; ++dj)
                            cand[di * bk + dj] =
                                (uint8_t)allowed_padded(sp, bm, Lq, Lk, r * bq + di, c * bk + dj);
                    uint64_t h = fnv1a(cand, pbytes);
                    int64_t found = -1;
                    for (int64_t u = 0; u < P; ++u)
                        if (hashes[u] == h && memcmp(patterns + (size_t)u * pbytes, cand, pbytes) == 0) {
                            found = u;
                            break;
                        }
                    if (found < 0) {
                        if (P >= pattern_capacity) { free(cand); free(hashes); return ORACLE_ERR_CAPACITY; }
                        memcpy(patterns + (size_t)P * pbytes, cand, pbytes);
                        hashes[P] = h;
                        found = P++;
                    }
                    mask_next[g] = (int32_t)found;
                }
                ++g;
            }
            for (int64_t x = first; x < g; ++x) {
                bounds_start[x] = (uint8_t)(x == first);
                bounds_end[x] = (uint8_t)(x == g - 1);
            }
        }
    }
    row_ptr[nbm * nq] = (int32_t)g;
    *num_patterns = P;
    free(cand);
    free(hashes);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Attention forward, the plain definition.                                   */
/* For each requested (b, hq, i): the score row s_j = scale * q_i . k_j       */
/* (soft-capped if cap > 0), masked entries excluded; two-pass softmax: m =   */
/* max s_j, l = sum exp(s_j - m), O_i = sum exp(s_j - m) v_j / l and          */
/* LSE_i = m + ln l.                                                           */
/* [L13 §5.1] safe softmax; [L13 §5.2] O = softmax(qk) v; [L13 §5.4] soft cap */
/* cap*tanh(x/cap); [L13 §6.3] residual LSE; [OPS] "LSE and Online Softmax".  */
/* Score panels of up to PANEL rows x Lk keys are materialised in f64.        */
/* ------------------------------------------------------------------------ */
#define PANEL 64

static double bf16_to_double(uint16_t x)
{
    uint32_t u = ((uint32_t)x) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t B, Hq, Hkv, Lq, Lk, dqk, dv;
    const oracle_mask_spec *sp;
    double scale, softcap;
    const int64_t *rows; /* flat (b*Hq + h)*Lq + i, sorted or not */
    int64_t nrows;
    double *out, *lse;
    int64_t next;
    pthread_mutex_t mu;
} attn_job;

static void attention_panel(attn_job *jb, int64_t x0, int64_t x1, double *S, double *kf, double *qf)
{
    (void)kf;
    for (int64_t x = x0; x < x1; ++x) {
        int64_t flat = jb->rows ? jb->rows[x] : x;
        int64_t i = flat % jb->Lq;
        int64_t bh = flat / jb->Lq;
        int64_t h = bh % jb->Hq, b = bh / jb->Hq;
        int64_t kvh = h / (jb->Hq / jb->Hkv);
        int64_t bm = jb->sp->q_seg != NULL ? b : 0;
        const uint16_t *qrow = jb->q + ((b * jb->Hq + h) * jb->Lq + i) * jb->dqk;
        for (int64_t d = 0; d < jb->dqk; ++d) qf[d] = bf16_to_double(qrow[d]);
        double *srow = S + (x - x0) * jb->Lk;
        /* 1. scores (materialised) */
        for (int64_t j = 0; j < jb->Lk; ++j) {
            if (!allowed(jb->sp, bm, jb->Lq, jb->Lk, i, j)) { srow[j] = -INFINITY; continue; }
            const uint16_t *krow = jb->k + ((b * jb->Hkv + kvh) * jb->Lk + j) * jb->dqk;
            double dot = 0.0;
            for (int64_t d = 0; d < jb->dqk; ++d) dot += qf[d] * bf16_to_double(krow[d]);
            double s = jb->scale * dot;
            if (jb->softcap > 0.0) s = jb->softcap * tanh(s / jb->softcap);
            srow[j] = s;
        }
        /* 2. pass one: the row maximum over allowed keys */
        double m = -INFINITY;
        for (int64_t j = 0; j < jb->Lk; ++j)
            if (srow[j] > m) m = srow[j];
        double *o = jb->out + x * jb->dv;
        for (int64_t d = 0; d < jb->dv; ++d) o[d] = 0.0;
        if (m == -INFINITY) { /* no allowed key */
            jb->lse[x] = -INFINITY;
            continue;
        }
        /* 3. pass two: denominators and the weighted sum of values */
        double l = 0.0;
        for (int64_t j = 0; j < jb->Lk; ++j) {
            if (srow[j] == -INFINITY) continue;
            double p = exp(srow[j] - m);
            l += p;
            const uint16_t *vrow = jb->v + ((b * jb->Hkv + kvh) * jb->Lk + j) * jb->dv;
            for (int64_t d = 0; d < jb->dv; ++d) o[d] += p * bf16_to_double(vrow[d]);
        }
        for (int64_t d = 0; d < jb->dv; ++d) o[d] /= l;
        jb->lse[x] = m + log(l);
    }
}

static void *attention_worker(void *arg)
{
    attn_job *jb = (attn_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(PANEL * jb->Lk));
    double *qf = (double *)malloc(sizeof(double) * (size_t)jb->dqk);
    if (!S || !qf) { free(S); free(qf); return NULL; }
    for (;;) {
        pthread_mutex_lock(&jb->mu);
        int64_t x0 = jb->next;
        jb->next += PANEL;
        pthread_mutex_unlock(&jb->mu);
        if (x0 >= jb->nrows) break;
        int64_t x1 = x0 + PANEL < jb->nrows ? x0 + PANEL : jb->nrows;
        attention_panel(jb, x0, x1, S, NULL, qf);
    }
    free(S);
    free(qf);
    return NULL;
}

/* q, k, v are bf16 bit patterns: q [B][Hq][Lq][dqk], k [B][Hkv][Lk][dqk],
 * v [B][Hkv][Lk][dv].  rows (optional) lists flat query rows
 * (b*Hq + h)*Lq + i; when NULL every row is computed in order and nrows must
 * be B*Hq*Lq.  out is [nrows][dv] f64, lse is [nrows] f64. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lk, int64_t dqk, int64_t dv,
                     const oracle_mask_spec *sp, double scale, double softcap,
                     const int64_t *rows, int64_t nrows, int nthreads, double *out, double *lse)
{
    if (!q || !k || !v || !sp || !out || !lse || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv ||
        Lq <= 0 || Lk <= 0 || dqk <= 0 || dv <= 0 || nrows < 0)
        return ORACLE_ERR_ARG;
    if (!rows && nrows != B * Hq * Lq) return ORACLE_ERR_ARG;
    if (sp->q_seg != NULL && (sp->kv_seg == NULL || sp->batch != B)) return ORACLE_ERR_ARG;
    if (rows)
        for (int64_t x = 0; x < nrows; ++x)
            if (rows[x] < 0 || rows[x] >= B * Hq * Lq) return ORACLE_ERR_ARG;
    attn_job jb;
    jb.q = q; jb.k = k; jb.v = v;
    jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.Lq = Lq; jb.Lk = Lk; jb.dqk = dqk; jb.dv = dv;
    jb.sp = sp; jb.scale = scale; jb.softcap = softcap;
    jb.rows = rows; jb.nrows = nrows; jb.out = out; jb.lse = lse;
    jb.next = 0;
    pthread_mutex_init(&jb.mu, NULL);
    run_threads(attention_worker, &jb, nthreads);
    pthread_mutex_destroy(&jb.mu);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Backward pass of one (batch b, query head h): the gradients of
 *   out_i = sum_j P_ij v_j,  P_ij = exp(s_ij) / sum_j' exp(s_ij')  (allowed j)
 * with respect to q, k and v, for an upstream gradient dout.  Plain calculus
 * on the forward's definition (the softmax Jacobian):
 *   dP_ij = dout_i . v_j,  D_i = sum_j P_ij dP_ij,  dS_ij = P_ij (dP_ij - D_i),
 *   with the soft cap s = cap tanh(u/cap), u = scale q.k: dU_ij = dS_ij (1 - t_ij^2),
 *   t = tanh(u/cap) (without it dU = dS);
 *   dq_i = scale sum_j dU_ij k_j,  dk_j = scale sum_i dU_ij q_i,  dv_j = sum_i P_ij dout_i.
 * P is recomputed from the row's log-sum-exp, P_ij = exp(s_ij - LSE_i) -- the
 * residual the forward keeps for its backward ([L13] §6.3; [OPS] "LSE and
 * Online Softmax": the backward rebuilds the probabilities from LSE instead
 * of storing them).  Pass A runs over query rows (LSE, D, dq); pass B over key
 * rows (dk, dv), each row owned by one thread. */

typedef struct {
    const double *q, *k, *v, *dout, *delta_in;
    int64_t b, Lq, Lk, dqk, dv;
    const oracle_mask_spec *sp;
    double scale, softcap;
    double *dq, *dk, *dvo, *lse, *delta;
    int64_t next, total;
    pthread_mutex_t mu;
} bwd_job;

static int64_t bwd_take(bwd_job *jb)
{
    pthread_mutex_lock(&jb->mu);
    int64_t x = jb->next++;
    pthread_mutex_unlock(&jb->mu);
    return x < jb->total ? x : -1;
}

/* score s and tanh value t of (i, j); returns 0 when the pair is masked */
static int bwd_score(const bwd_job *jb, int64_t i, int64_t j, double *s, double *t)
{
    if (!allowed(jb->sp, jb->b, jb->Lq, jb->Lk, i, j)) return 0;
    const double *qi = jb->q + i * jb->dqk, *kj = jb->k + j * jb->dqk;
    double dot = 0.0;
    for (int64_t d = 0; d < jb->dqk; ++d) dot += qi[d] * kj[d];
    double u = jb->scale * dot;
    if (jb->softcap > 0.0) {
        *t = tanh(u / jb->softcap);
        *s = jb->softcap * *t;
    } else {
        *t = 0.0;
        *s = u;
    }
    return 1;
}

static double bwd_dp(const bwd_job *jb, int64_t i, int64_t j)
{
    const double *g = jb->dout + i * jb->dv, *vj = jb->v + j * jb->dv;
    double acc = 0.0;
    for (int64_t d = 0; d < jb->dv; ++d) acc += g[d] * vj[d];
    return acc;
}

static void *bwd_rows_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)jb->Lk);
    double *t = (double *)malloc(sizeof(double) * (size_t)jb->Lk);
    unsigned char *ok = (unsigned char *)malloc((size_t)jb->Lk);
    if (!s || !t || !ok) { free(s); free(t); free(ok); return NULL; }
    for (int64_t i; (i = bwd_take(jb)) >= 0;) {
        double *dqi = jb->dq + i * jb->dqk;
        for (int64_t d = 0; d < jb->dqk; ++d) dqi[d] = 0.0;
        double m = -INFINITY;
        for (int64_t j = 0; j < jb->Lk; ++j) {
            ok[j] = (unsigned char)bwd_score(jb, i, j, &s[j], &t[j]);
            if (ok[j] && s[j] > m) m = s[j];
        }
        if (m == -INFINITY) { /* no allowed key: no gradient flows */
            jb->lse[i] = -INFINITY;
            jb->delta[i] = 0.0;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < jb->Lk; ++j)
            if (ok[j]) l += exp(s[j] - m);
        double lse = m + log(l), D = 0.0;
        if (jb->delta_in) { /* D given (e.g. dout_i . out_i of a stored output) */
            D = jb->delta_in[i];
        } else {
            for (int64_t j = 0; j < jb->Lk; ++j)
                if (ok[j]) D += exp(s[j] - lse) * bwd_dp(jb, i, j);
        }
        jb->lse[i] = lse;
        jb->delta[i] = D;
        for (int64_t j = 0; j < jb->Lk; ++j) {
            if (!ok[j]) continue;
            double p = exp(s[j] - lse);
            double du = p * (bwd_dp(jb, i, j) - D);
            if (jb->softcap > 0.0) du *= 1.0 - t[j] * t[j];
            const double *kj = jb->k + j * jb->dqk;
            for (int64_t d = 0; d < jb->dqk; ++d) dqi[d] += jb->scale * du * kj[d];
        }
    }
    free(s); free(t); free(ok);
    return NULL;
}

static void *bwd_keys_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    for (int64_t j; (j = bwd_take(jb)) >= 0;) {
        double *dkj = jb->dk + j * jb->dqk, *dvj = jb->dvo + j * jb->dv;
        for (int64_t d = 0; d < jb->dqk; ++d) dkj[d] = 0.0;
        for (int64_t d = 0; d < jb->dv; ++d) dvj[d] = 0.0;
        for (int64_t i = 0; i < jb->Lq; ++i) {
            double s, t;
            if (jb->lse[i] == -INFINITY || !bwd_score(jb, i, j, &s, &t)) continue;
            double p = exp(s - jb->lse[i]);
            double du = p * (bwd_dp(jb, i, j) - jb->delta[i]);
            if (jb->softcap > 0.0) du *= 1.0 - t * t;
            const double *g = jb->dout + i * jb->dv, *qi = jb->q + i * jb->dqk;
            for (int64_t d = 0; d < jb->dv; ++d) dvj[d] += p * g[d];
            for (int64_t d = 0; d < jb->dqk; ++d) dkj[d] += jb->scale * du * qi[d];
        }
    }
    return NULL;
}

/* q [Lq][dqk] and dout [Lq][dv] are head h's rows of batch b; k [Lk][dqk] and
 * v [Lk][dv] those of its key/value head; all f64.  b selects the segment-ID
 * batch row (ignored without segment IDs).  delta_in [Lq] is optional: when
 * given, D_i is taken from it (for instance dout_i . out_i of a stored
 * forward output); when NULL, D_i = sum_j P_ij dP_ij exactly.  Writes
 * dq [Lq][dqk], this head's contributions dk [Lk][dqk] and
 * dv [Lk][dv] (a GQA group sums them), the row log-sum-exp lse [Lq] and
 * D = delta [Lq]. */
int oracle_attention_bwd_head(const double *q, const double *k, const double *v, const double *dout,
                              const double *delta_in, int64_t b, int64_t Lq, int64_t Lk, int64_t dqk, int64_t dv,
                              const oracle_mask_spec *sp, double scale, double softcap, int nthreads,
                              double *dq, double *dk, double *dvo, double *lse, double *delta)
{
    if (!q || !k || !v || !dout || !sp || !dq || !dk || !dvo || !lse || !delta || Lq <= 0 || Lk <= 0 ||
        dqk <= 0 || dv <= 0 || b < 0)
        return ORACLE_ERR_ARG;
    if (sp->q_seg != NULL && (sp->kv_seg == NULL || b >= sp->batch)) return ORACLE_ERR_ARG;
    bwd_job jb;
    jb.q = q; jb.k = k; jb.v = v; jb.dout = dout; jb.delta_in = delta_in;
    jb.b = sp->q_seg != NULL ? b : 0;
    jb.Lq = Lq; jb.Lk = Lk; jb.dqk = dqk; jb.dv = dv;
    jb.sp = sp; jb.scale = scale; jb.softcap = softcap;
    jb.dq = dq; jb.dk = dk; jb.dvo = dvo; jb.lse = lse; jb.delta = delta;
    pthread_mutex_init(&jb.mu, NULL);
    jb.next = 0; jb.total = Lq;
    run_threads(bwd_rows_worker, &jb, nthreads);
    jb.next = 0; jb.total = Lk;
    run_threads(bwd_keys_worker, &jb, nthreads);
    pthread_mutex_destroy(&jb.mu);
    return ORACLE_OK;
}
