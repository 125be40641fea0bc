/*
 * CPU oracle for the DSA lightning-indexer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA product path
 * never links, calls or includes it, and this file shares no code with it.
 *
 * Plain, slow, obviously correct: every product and sum in double precision,
 * straight loops in the order the definition is written, a library sort for
 * the selection.  bf16 inputs are widened exactly to double; the only
 * rounding to fp32 happens when a score is stored into an fp32 output.
 *
 * What it computes (all page references are to the NeMo AutoModel page
 * "nemo_automodel.components.models.deepseek_v4.kernels.tilelang_indexer",
 * unless another page is named):
 *
 *  - Layouts, from the `V4IndexerFunction` docstring and the
 *    `v4_lighting_indexer` parameter list:
 *        q [S, B, H, D] bf16, k [S_kv, B, D] bf16, w [S, B, H] fp32,
 *        topk_indices [B, S, topk] int32, returned scores [B, S, topk] fp32.
 *  - The lightning-indexer score of query t against compressed key j:
 *        I[t, j] = sum_h w[t, h] * ReLU( sum_d q[t, h, d] * k[j, d] )
 *    (the pages name the "lighting_indexer" but do not print the formula;
 *    this is the DeepSeek Sparse Attention lightning-indexer definition).
 *  - Causal masking over compressed keys (the module summary says the
 *    indexer was moved onto V4's SBHD layout with causal masking; the
 *    `compress_ratio` parameter is 4 on C4 layers): compressed key j
 *    summarises source tokens [j*r, (j+1)*r), and a key counts only when its
 *    whole block is at or before the query position, (j+1)*r - 1 <= t.  The
 *    metrale.ai page "Module glm5next_dsa", section "Checkpoint and kernel
 *    facts", applies the same rule to pools: an incomplete pool at the end
 *    does not count.
 *  - Top-k: the `topk` visible keys with the largest score, returned in
 *    descending score order, equal scores ordered by the lower key index
 *    first; slots past the number of visible keys hold index -1 (the page
 *    "Module glm5next_dsa" marks an invalid index with -1, section "Shape of
 *    the pipeline", and fills the whole index row with -1 before storing the
 *    real indices, section "Checkpoint and kernel facts") and score -inf.
 *  - Given indices (`topk_indices` parameter, and `pytorch_extract_topk_scores
 *    (logits, topk_indices, dim=-1)`): the score of each given slot is the
 *    logit at that index, -inf where the index is -1, out of range or not
 *    visible (a masked logit is -inf); the indices are returned unchanged.
 *
 * Query positions: prefill rows sit at position t = s; when q_pos is given,
 * row s of sequence b sits at position q_pos[b] + s (decode rows).
 *
 * Key validity (the pool variant, page "Module glm5next_dsa": "index_scores
 * -> [Q, P] scores + candidate validity"): when key_valid is given, a key
 * whose flag is 0 is not a candidate -- it is treated like a key that is not
 * visible (no top-k slot, -inf when asked for by index or in the logits).
 *
 * The pool variant's other two steps (same page, "Shape of the pipeline"
 * and "Checkpoint and kernel facts") are oracle_kpool_compress and
 * oracle_expand_selection below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* exact widening of a bf16 bit pattern: bf16 is the top half of an fp32 */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* causal visibility of compressed key j for a query at position t */
int oracle_key_visible(long long j, long long t, int ratio)
{
    return (j + 1) * (long long)ratio - 1 <= t;
}

static long long row_position(const int32_t *q_pos, int b, int s)
{
    return q_pos ? (long long)q_pos[b] + s : (long long)s;
}

typedef struct {
    const uint16_t *q;
    const uint16_t *k;
    const float *w;
    int S, B, H, D, S_kv, ratio;
    const uint8_t *key_valid; /* [S_kv, B] or NULL (every key valid) */
} problem_t;

/* key j of sequence b is a candidate for a query at position t */
static int key_candidate(const problem_t *p, long long j, int b, long long t)
{
    if (!oracle_key_visible(j, t, p->ratio)) return 0;
    return !p->key_valid || p->key_valid[(size_t)j * p->B + b] != 0;
}

/* I[t, j] for one (row, key) pair, the definition written out */
static double score_one(const problem_t *p, int b, int s, long long j)
{
    double total = 0.0;
    for (int h = 0; h < p->H; ++h) {
        const uint16_t *qh = p->q + (((size_t)s * p->B + b) * p->H + h) * p->D;
        const uint16_t *kj = p->k + ((size_t)j * p->B + b) * p->D;
        double dot = 0.0;
        for (int d = 0; d < p->D; ++d)
            dot += bf16_to_double(qh[d]) * bf16_to_double(kj[d]);
        double relu = dot > 0.0 ? dot : 0.0;
        double wt = (double)p->w[((size_t)s * p->B + b) * p->H + h];
        total += wt * relu;
    }
    return total;
}

typedef struct {
    double score;
    int32_t j;
} cand_t;

/* descending score, then ascending key index (equal scores: lower j first) */
static int cand_cmp(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

/* ---- row-parallel driver ------------------------------------------------ */

typedef struct {
    const problem_t *p;
    const int32_t *q_pos;
    const int64_t *rows; /* row id = b * S + s */
    long long n_rows;
    int topk;
    const int32_t *in_idx; /* [B, S, topk] or NULL */
    /* outputs, one line of `topk` per requested row */
    int32_t *out_idx;
    float *out_scores;
    double *out_scores_f64;
    double *out_next; /* score of the (topk+1)-th visible key, or -inf */
    int32_t *out_nvis;
    double *logits; /* [n_rows, S_kv] or NULL */
    long long next_row;
    pthread_mutex_t lock;
} job_t;

static void do_row(job_t *jb, long long r)
{
    const problem_t *p = jb->p;
    long long row = jb->rows[r];
    int b = (int)(row / p->S), s = (int)(row % p->S);
    long long t = row_position(jb->q_pos, b, s);
    int topk = jb->topk;

    if (jb->logits) {
        double *L = jb->logits + (size_t)r * p->S_kv;
        for (long long j = 0; j < p->S_kv; ++j)
            L[j] = key_candidate(p, j, b, t) ? score_one(p, b, s, j)
                                             : -INFINITY;
    }

    if (jb->in_idx) {
        const int32_t *given = jb->in_idx + ((size_t)b * p->S + s) * topk;
        int32_t nvis = 0;
        for (long long j = 0; j < p->S_kv; ++j)
            nvis += key_candidate(p, j, b, t);
        for (int i = 0; i < topk; ++i) {
            int32_t j = given[i];
            double v = -INFINITY;
            if (j >= 0 && j < p->S_kv && key_candidate(p, j, b, t))
                v = score_one(p, b, s, j);
            if (jb->out_idx) jb->out_idx[(size_t)r * topk + i] = j;
            if (jb->out_scores) jb->out_scores[(size_t)r * topk + i] = (float)v;
            if (jb->out_scores_f64) jb->out_scores_f64[(size_t)r * topk + i] = v;
        }
        if (jb->out_nvis) jb->out_nvis[r] = nvis;
        if (jb->out_next) jb->out_next[r] = -INFINITY;
        return;
    }

    if (!jb->out_idx && !jb->out_scores && !jb->out_scores_f64) return;

    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(p->S_kv > 0 ? p->S_kv : 1));
    long long n = 0;
    for (long long j = 0; j < p->S_kv; ++j) {
        if (!key_candidate(p, j, b, t)) continue;
        c[n].score = jb->logits ? jb->logits[(size_t)r * p->S_kv + j]
                                : score_one(p, b, s, j);
        c[n].j = (int32_t)j;
        ++n;
    }
    qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
    for (int i = 0; i < topk; ++i) {
        int32_t j = i < n ? c[i].j : -1;
        double v = i < n ? c[i].score : -INFINITY;
        if (jb->out_idx) jb->out_idx[(size_t)r * topk + i] = j;
        if (jb->out_scores) jb->out_scores[(size_t)r * topk + i] = (float)v;
        if (jb->out_scores_f64) jb->out_scores_f64[(size_t)r * topk + i] = v;
    }
    if (jb->out_next) jb->out_next[r] = topk < n ? c[topk].score : -INFINITY;
    if (jb->out_nvis) jb->out_nvis[r] = (int32_t)n;
    free(c);
}

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&jb->lock);
        long long r = jb->next_row++;
        pthread_mutex_unlock(&jb->lock);
        if (r >= jb->n_rows) break;
        do_row(jb, r);
    }
    return NULL;
}

/*
 * The whole forward for a list of rows.
 *
 * q, k: bf16 bit patterns; w fp32; q_pos [B] or NULL; rows: row ids b*S+s.
 * key_valid: [S_kv, B] uint8 or NULL (every key a candidate).
 * in_idx NULL -> top-k path; else the given-indices path.
 * Any output pointer may be NULL.  Per requested row r:
 *   out_idx[r*topk + i], out_scores[...] (fp32), out_scores_f64[...] (fp64),
 *   out_next[r] = (topk+1)-th visible score (-inf if none; top-k path),
 *   out_nvis[r] = number of candidate (visible and valid) keys,
 *   logits[r*S_kv + j] = I[t, j] or -inf where key j is not a candidate.
 * Returns the number of threads used.
 */
int oracle_indexer_fwd(const uint16_t *q, const uint16_t *k, const float *w,
                       int S, int B, int H, int D, int S_kv, int ratio,
                       int topk, const int32_t *q_pos,
                       const uint8_t *key_valid, const int32_t *in_idx,
                       const int64_t *rows, long long n_rows,
                       int32_t *out_idx, float *out_scores,
                       double *out_scores_f64, double *out_next,
                       int32_t *out_nvis, double *logits, int n_threads)
{
    problem_t p = {q, k, w, S, B, H, D, S_kv, ratio, key_valid};
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.p = &p;
    jb.q_pos = q_pos;
    jb.rows = rows;
    jb.n_rows = n_rows;
    jb.topk = topk;
    jb.in_idx = in_idx;
    jb.out_idx = out_idx;
    jb.out_scores = out_scores;
    jb.out_scores_f64 = out_scores_f64;
    jb.out_next = out_next;
    jb.out_nvis = out_nvis;
    jb.logits = logits;
    jb.next_row = 0;
    pthread_mutex_init(&jb.lock, NULL);

    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long long)n_threads > n_rows) n_threads = n_rows > 0 ? (int)n_rows : 1;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, worker, &jb) == 0) ++started;
    worker(&jb);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&jb.lock);
    return started + 1;
}

/*
 * Backward of the given-slots forward (V4IndexerFunction.backward, page
 * "nemo_automodel.components.models.deepseek_v4.kernels.tilelang_indexer":
 * the gradient of a loss with respect to index_q, index_k and weights given
 * the gradient of the returned scores).  The pages print no formula; this is
 * the derivative of the score definition above, slot by slot:
 *
 *   slot (b, s, i) with key j = idx[b, s, i] that is in [0, S_kv) and
 *   visible at the row's position, upstream gradient g = grad_scores[b,s,i]:
 *     dot_h = sum_d q[s,b,h,d] * k[j,b,d]
 *     grad_w[s,b,h]   += g * max(dot_h, 0)
 *     if dot_h > 0 (ReLU'(0) = 0):
 *       grad_q[s,b,h,:] += g * w[s,b,h] * k[j,b,:]
 *       grad_k[j,b,:]   += g * w[s,b,h] * q[s,b,h,:]
 *   other slots (-1, out of range, not visible) contribute nothing.
 *
 * All in double, single-threaded (grad_k sums over rows).  abs_q, abs_k and
 * abs_w (may be NULL) receive the same sums over the absolute values of the
 * terms, the scale an implementation's rounding error is measured against.
 * The outputs are overwritten (zeroed first).
 */
void oracle_indexer_bwd(const uint16_t *q, const uint16_t *k, const float *w,
                        int S, int B, int H, int D, int S_kv, int ratio,
                        int topk, const int32_t *q_pos, const int32_t *idx,
                        const float *grad_scores, double *grad_q,
                        double *grad_k, double *grad_w, double *abs_q,
                        double *abs_k, double *abs_w)
{
    const size_t nq = (size_t)S * B * H * D, nk = (size_t)S_kv * B * D;
    const size_t nw = (size_t)S * B * H;
    memset(grad_q, 0, nq * sizeof(double));
    memset(grad_k, 0, nk * sizeof(double));
    memset(grad_w, 0, nw * sizeof(double));
    if (abs_q) memset(abs_q, 0, nq * sizeof(double));
    if (abs_k) memset(abs_k, 0, nk * sizeof(double));
    if (abs_w) memset(abs_w, 0, nw * sizeof(double));
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < S; ++s) {
            const long long t = row_position(q_pos, b, s);
            for (int i = 0; i < topk; ++i) {
                const size_t slot = ((size_t)b * S + s) * topk + i;
                const long long j = idx[slot];
                if (j < 0 || j >= S_kv || !oracle_key_visible(j, t, ratio))
                    continue;
                const double g = (double)grad_scores[slot];
                const uint16_t *kj = k + ((size_t)j * B + b) * D;
                for (int h = 0; h < H; ++h) {
                    const size_t qo = (((size_t)s * B + b) * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += bf16_to_double(q[qo + d]) * bf16_to_double(kj[d]);
                    const size_t wo = ((size_t)s * B + b) * H + h;
                    const double relu = dot > 0.0 ? dot : 0.0;
                    grad_w[wo] += g * relu;
                    if (abs_w) abs_w[wo] += fabs(g * relu);
                    if (dot <= 0.0) continue;
                    const double c = g * (double)w[wo];
                    for (int d = 0; d < D; ++d) {
                        const double tq = c * bf16_to_double(kj[d]);
                        const double tk = c * bf16_to_double(q[qo + d]);
                        grad_q[qo + d] += tq;
                        grad_k[((size_t)j * B + b) * D + d] += tk;
                        if (abs_q) abs_q[qo + d] += fabs(tq);
                        if (abs_k) abs_k[((size_t)j * B + b) * D + d] += fabs(tk);
                    }
                }
            }
        }
    }
}

/*
 * Pool compression (page "Module glm5next_dsa": kpool_compress in "Shape of
 * the pipeline"; section "Checkpoint and kernel facts": the softmax of a
 * pool is taken across its slots separately for each channel, pools begin
 * at first_key, and a pool is a candidate only when all of its slots are
 * valid).
 *
 * Pool p of sequence b covers the tokens first_key + p*kpool + s,
 * s = 0..kpool-1; there are P = (T - first_key) / kpool whole pools (an
 * incomplete pool at the end is dropped).  For channel c, with the slot logits
 * z_s = gate[token_s, b, c] + ape[s, c]:
 *     key[p, b, c] = sum_s softmax_s(z)_s * k[token_s, b, c]
 * (the page names the inputs k, gate, valid and ape and the softmax axis; the
 * logit of a slot being its gate plus its slot-position embedding is the
 * reading of "ape").  valid_out[p, b] = 1 iff valid[token_s, b] != 0 for
 * every slot (valid NULL: every token valid).
 *
 * k [T, B, D] bf16 bits, gate [T, B, D] fp32, ape [kpool, D] fp32,
 * valid [T, B] uint8 or NULL; out_keys [P, B, D] double, out_valid [P, B].
 * Returns P.
 */
long long oracle_kpool_compress(const uint16_t *k, const float *gate,
                                const float *ape, const uint8_t *valid,
                                int T, int B, int D, int kpool, int first_key,
                                double *out_keys, uint8_t *out_valid)
{
    long long P = T > first_key ? (long long)(T - first_key) / kpool : 0;
    for (long long p = 0; p < P; ++p) {
        for (int b = 0; b < B; ++b) {
            int all_valid = 1;
            for (int s = 0; s < kpool; ++s) {
                long long tok = first_key + p * kpool + s;
                if (valid && valid[(size_t)tok * B + b] == 0) all_valid = 0;
            }
            if (out_valid) out_valid[(size_t)p * B + b] = (uint8_t)all_valid;
            for (int c = 0; c < D; ++c) {
                /* softmax over the slots, written with the usual max shift */
                double zmax = -INFINITY;
                for (int s = 0; s < kpool; ++s) {
                    long long tok = first_key + p * kpool + s;
                    double z = (double)gate[((size_t)tok * B + b) * D + c] +
                               (double)ape[(size_t)s * D + c];
                    if (z > zmax) zmax = z;
                }
                double den = 0.0, num = 0.0;
                for (int s = 0; s < kpool; ++s) {
                    long long tok = first_key + p * kpool + s;
                    double z = (double)gate[((size_t)tok * B + b) * D + c] +
                               (double)ape[(size_t)s * D + c];
                    double e = exp(z - zmax);
                    den += e;
                    num += e * bf16_to_double(k[((size_t)tok * B + b) * D + c]);
                }
                out_keys[((size_t)p * B + b) * D + c] = num / den;
            }
        }
    }
    return P;
}

/*
 * Selection expansion (page "Module glm5next_dsa": expand_selection in
 * "Shape of the pipeline", where -1 marks an invalid id; section
 * "Checkpoint and kernel facts": the expansion fills its whole output row
 * with -1 first, so no slot is left unwritten).  Each row's select_k pool ids become select_k * kpool token
 * ids: slot i*kpool + s holds first_key + pool_i*kpool + s, or -1 when
 * pool_i is -1.
 */
void oracle_expand_selection(const int32_t *pools, long long rows,
                             int select_k, int kpool, int first_key,
                             int32_t *out_tokens)
{
    const long long width = (long long)select_k * kpool;
    for (long long r = 0; r < rows; ++r) {
        int32_t *out = out_tokens + (size_t)r * width;
        for (long long i = 0; i < width; ++i) out[i] = -1;
        for (int i = 0; i < select_k; ++i) {
            int32_t pool = pools[(size_t)r * select_k + i];
            if (pool < 0) continue;
            for (int s = 0; s < kpool; ++s)
                out[(size_t)i * kpool + s] =
                    (int32_t)((long long)first_key + (long long)pool * kpool + s);
        }
    }
}

/*
 * Sparse MLA forward over the selected tokens (page "Module glm5next_dsa",
 * "Shape of the pipeline": the selected tokens feed an MLA attention
 * without the rotary part, over those tokens only; the
 * NeMo AutoModel pages list tilelang_sparse_mla_fwd after the indexer; the
 * latent width is kv_lora_rank, section "Constants", KERNEL_KV_LORA_DIM).
 * The pages print no formula; this is attention in the MLA latent space
 * with no rotary part, the latent row of a selected token serving as both
 * key and value:
 *
 *   for row (b, s), head h, and the slots i whose token j_i = idx[b,s,i]
 *   lies in [0, T) (-1 and out-of-range slots are skipped; repeated tokens
 *   count once per slot):
 *     x_i = scale * sum_d q[s,b,h,d] * c[j_i,b,d]
 *     o[s,b,h,:] = sum_i softmax(x)_i * c[j_i,b,:]
 *     lse[s,b,h] = log sum_i exp(x_i)           (natural log)
 *   a row with no such slot: o = 0, lse = -inf.
 *
 * q [S, B, H, Dc] bf16 bits, c [T, B, Dc] bf16 bits, idx [B, S, topk];
 * out_o [S, B, H, Dc] double, out_lse [S, B, H] double.  Rows in parallel.
 */
typedef struct {
    const uint16_t *q, *c;
    const int32_t *idx;
    int S, B, H, Dc, T, topk;
    double scale;
    double *o, *lse;
    long long next;
    pthread_mutex_t lock;
} mla_job_t;

static void mla_row(mla_job_t *jb, long long row)
{
    const int b = (int)(row / jb->S), s = (int)(row % jb->S);
    const int32_t *sel = jb->idx + ((size_t)b * jb->S + s) * jb->topk;
    double *x = (double *)malloc(sizeof(double) * (size_t)(jb->topk > 0 ? jb->topk : 1));
    for (int h = 0; h < jb->H; ++h) {
        const uint16_t *qh = jb->q + (((size_t)s * jb->B + b) * jb->H + h) * jb->Dc;
        double *oh = jb->o + (((size_t)s * jb->B + b) * jb->H + h) * jb->Dc;
        double xmax = -INFINITY;
        int n = 0;
        for (int i = 0; i < jb->topk; ++i) {
            const int32_t j = sel[i];
            x[i] = -INFINITY;
            if (j < 0 || j >= jb->T) continue;
            const uint16_t *cj = jb->c + ((size_t)j * jb->B + b) * jb->Dc;
            double dot = 0.0;
            for (int d = 0; d < jb->Dc; ++d)
                dot += bf16_to_double(qh[d]) * bf16_to_double(cj[d]);
            x[i] = jb->scale * dot;
            if (x[i] > xmax) xmax = x[i];
            ++n;
        }
        for (int d = 0; d < jb->Dc; ++d) oh[d] = 0.0;
        if (n == 0) {
            jb->lse[((size_t)s * jb->B + b) * jb->H + h] = -INFINITY;
            continue;
        }
        double den = 0.0;
        for (int i = 0; i < jb->topk; ++i) {
            const int32_t j = sel[i];
            if (j < 0 || j >= jb->T) continue;
            const double e = exp(x[i] - xmax);
            den += e;
            const uint16_t *cj = jb->c + ((size_t)j * jb->B + b) * jb->Dc;
            for (int d = 0; d < jb->Dc; ++d) oh[d] += e * bf16_to_double(cj[d]);
        }
        for (int d = 0; d < jb->Dc; ++d) oh[d] /= den;
        jb->lse[((size_t)s * jb->B + b) * jb->H + h] = xmax + log(den);
    }
    free(x);
}

static void *mla_worker(void *arg)
{
    mla_job_t *jb = (mla_job_t *)arg;
    const long long rows = (long long)jb->S * jb->B;
    for (;;) {
        pthread_mutex_lock(&jb->lock);
        long long r = jb->next++;
        pthread_mutex_unlock(&jb->lock);
        if (r >= rows) break;
        mla_row(jb, r);
    }
    return NULL;
}

int oracle_sparse_mla_fwd(const uint16_t *q, const uint16_t *c,
                          const int32_t *idx, int S, int B, int H, int Dc,
                          int T, int topk, double scale, double *out_o,
                          double *out_lse, int n_threads)
{
    mla_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.c = c; jb.idx = idx;
    jb.S = S; jb.B = B; jb.H = H; jb.Dc = Dc; jb.T = T; jb.topk = topk;
    jb.scale = scale; jb.o = out_o; jb.lse = out_lse; jb.next = 0;
    pthread_mutex_init(&jb.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&th[started], NULL, mla_worker, &jb) == 0) ++started;
    mla_worker(&jb);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&jb.lock);
    return started + 1;
}
