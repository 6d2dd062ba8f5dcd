/*
 * fp64 CPU oracle for MLA tree-verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path calls, links or
 * loads this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes (page "The Shared Memory Ceiling", sections "Technical
 * Deep Dive" and "Assumptions and Correctness"): the naive form of the
 * verify attention, which holds the FULL score row of one (query, head) pair,
 * takes its maximum and normaliser, and forms the weighted sum of the values.
 * The MLA specifics (section "The Broader Context"): every head attends to
 * one shared latent KV row made of a 512-dim c_kv and a 64-dim k_rope; the
 * query is already in the latent space (q_lat, q_rope); V is c_kv.  A draft
 * tree token sees the whole prefix and, among the tree tokens, only its
 * ancestors and itself (ancestor-or-self mask given by a parent array).
 *
 * For request b with prefix P = seq_len - n_tree, node i and head h:
 *   visible V = {0..P-1} u {P + j : j in anc*(i)},  anc*(i) = {i, par(i), ...}
 *   s_t   = scale * (q_lat . c_t + q_rope . r_t)             for t in V
 *   lse   = m + ln sum_t exp(s_t - m),  m = max_t s_t       (natural log)
 *   out_d = sum_t exp(s_t - lse) * c_t[d]
 * KV row t of request b is kv[block_table[b][t / page] * page + t % page].
 * Everything is evaluated in double; the bf16 inputs widen exactly.
 *
 * A key range [key_begin, key_end) restricts V to positions inside it (the
 * split-KV partial of that range).  mla_oracle_combine merges such partials
 * with the log-sum-exp weights of flash-decoding.
 *
 * Sparse (top-k) variant, mla_oracle_verify_sparse_rows (page "The SMEM
 * Ceiling", section "The Problem Space": during decode each token attends to
 * a sparse set of previous tokens chosen by a top-k index selection): tree
 * token g carries topk slots topk_idx[g][0..topk); each slot holding a prefix
 * position t in [0, P) contributes that key once (a position listed twice
 * counts twice), -1 marks an unused slot.  The prefix part of V is replaced by
 * these slots; the ancestor-or-self tree keys stay visible as above.
 *
 * Returns 0 on success; 1 for an invalid argument; 6 for an invalid draft
 * tree or length (parent outside [-1, i), n_tree > seq_len, negative sizes);
 * 7 for a block-table entry outside [0, num_pages); 9 for a top-k slot that is
 * neither -1 nor a prefix position.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0 /* non-zero only in deliberately broken test builds */
#endif

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_BAD_TREE = 6, OR_BAD_BLOCK = 7, OR_BAD_INDEX = 9 };

typedef struct {
    const uint16_t *q_lat, *q_rope, *kv;
    const int32_t *block_table, *seq_lens, *parent, *n_tree;
    const int32_t *topk_idx;  /* [total_q][topk] or NULL (dense: the whole prefix) */
    int64_t topk;
    int64_t batch, total_q, heads, dl, dr, page, max_pages, num_pages;
    double scale;
    int64_t *q_off;   /* [batch + 1] first q index of each request */
    int64_t *q_req;   /* [total_q]   request of each q index        */
} problem_t;

static double widen(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* KV row of logical position t of request b, or NULL if its page id is invalid. */
static const uint16_t *kv_row(const problem_t *p, int64_t b, int64_t t)
{
#if ORACLE_MUTANT == 6
    int64_t slot = p->block_table[0 * p->max_pages + t / p->page];
#else
    int64_t slot = p->block_table[b * p->max_pages + t / p->page];
#endif
    if (slot < 0 || slot >= p->num_pages) return NULL;
    return p->kv + (slot * p->page + t % p->page) * (p->dl + p->dr);
}

/* One output row: q index g, head h, keys restricted to [k0, k1). */
static int one_row(const problem_t *p, int64_t g, int64_t h, int64_t k0, int64_t k1,
                   int64_t *keys, double *score, double *out, double *lse)
{
    const int64_t b = p->q_req[g];
    const int64_t base = p->q_off[b];
    const int64_t i = g - base;
    const int64_t T = p->n_tree[b];
    const int64_t L = p->seq_lens[b];
    const int64_t P = L - T;
    const int64_t D = p->dl + p->dr;
    int64_t n = 0;

    if (p->topk > 0) {
        /* the listed prefix positions, one key per slot */
        for (int64_t sl = 0; sl < p->topk; ++sl) {
            int64_t t = p->topk_idx[g * p->topk + sl];
#if ORACLE_MUTANT == 11
            if (t >= 0 && t + 1 < P) t += 1;        /* every listed position off by one */
#elif ORACLE_MUTANT == 12
            if (t < 0 && P > 0) t = 0;              /* unused slots attend to position 0 */
#endif
            if (t >= 0 && t >= k0 && t < k1) keys[n++] = t;
        }
    } else {
        /* the whole prefix is visible */
        for (int64_t t = (k0 > 0 ? k0 : 0); t < P && t < k1; ++t) keys[n++] = t;
    }
    /* ancestor-or-self walk up the parent array */
#if ORACLE_MUTANT == 2
    int64_t j = p->parent[base + i];      /* forgets the node itself */
#else
    int64_t j = i;
#endif
    int64_t steps = 0;
    while (j >= 0) {
        if (++steps > T) return OR_BAD_TREE;
#if ORACLE_MUTANT == 9
        int64_t t = P + j - 1;
#else
        int64_t t = P + j;
#endif
        if (t >= k0 && t < k1) keys[n++] = t;
        int64_t up = p->parent[base + j];
        if (up < -1 || up >= j) return OR_BAD_TREE;
#if ORACLE_MUTANT == 3
        break;                              /* stops after the first link */
#endif
        j = up;
    }

    const uint16_t *ql = p->q_lat + (g * p->heads + h) * p->dl;
    const uint16_t *qr = p->q_rope + (g * p->heads + h) * p->dr;
    for (int64_t k = 0; k < n; ++k) {
        const uint16_t *row = kv_row(p, b, keys[k]);
        if (!row) return OR_BAD_BLOCK;
        double s = 0.0;
        for (int64_t d = 0; d < p->dl; ++d) s += widen(ql[d]) * widen(row[d]);
#if ORACLE_MUTANT != 1
        for (int64_t d = 0; d < p->dr; ++d) s += widen(qr[d]) * widen(row[p->dl + d]);
#endif
#if ORACLE_MUTANT == 4
        score[k] = s;
#else
        score[k] = p->scale * s;
#endif
    }

    for (int64_t d = 0; d < p->dl; ++d) out[d] = 0.0;
    if (n == 0) {           /* nothing visible in this key range */
        *lse = -INFINITY;
        return OR_OK;
    }
    double m = score[0];
    for (int64_t k = 1; k < n; ++k) if (score[k] > m) m = score[k];
    double z = 0.0;
    for (int64_t k = 0; k < n; ++k) z += exp(score[k] - m);
    double l = m + log(z);
#if ORACLE_MUTANT == 5
    *lse = l / log(2.0);
#else
    *lse = l;
#endif
    for (int64_t k = 0; k < n; ++k) {
        const uint16_t *row = kv_row(p, b, keys[k]);
#if ORACLE_MUTANT == 7
        double w = exp(score[k] - m);       /* never normalised */
#else
        double w = exp(score[k] - l);
#endif
#if ORACLE_MUTANT == 8
        for (int64_t d = 0; d < p->dl; ++d) out[d] += w * widen(row[(d + p->dr) % D]);
#else
        for (int64_t d = 0; d < p->dl; ++d) out[d] += w * widen(row[d]);
#endif
    }
    (void)D;
    return OR_OK;
}

typedef struct {
    const problem_t *p;
    const int64_t *rows;
    int64_t n_rows, k0, k1;
    double *out, *lse;
    int64_t next;           /* shared work counter */
    int status;
} job_t;

static void *worker(void *arg)
{
    job_t *job = (job_t *)arg;
    const problem_t *p = job->p;
    int64_t maxlen = 1;
    for (int64_t b = 0; b < p->batch; ++b)
        if (p->seq_lens[b] > maxlen) maxlen = p->seq_lens[b];
    if (p->topk + 64 > maxlen) maxlen = p->topk + 64;   /* slots may repeat positions */
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(maxlen + 1));
    double *score = (double *)malloc(sizeof(double) * (size_t)(maxlen + 1));
    if (!keys || !score) {
        __atomic_store_n(&job->status, OR_BAD_ARG, __ATOMIC_RELAXED);
        free(keys);
        free(score);
        return NULL;
    }
    for (;;) {
        int64_t r = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (r >= job->n_rows) break;
        int64_t row = job->rows[r];
        int st = one_row(p, row / p->heads, row % p->heads, job->k0, job->k1, keys, score,
                         job->out + r * p->dl, job->lse + r);
        if (st) __atomic_store_n(&job->status, st, __ATOMIC_RELAXED);
    }
    free(keys);
    free(score);
    return NULL;
}

/* Check sizes and the tree of every request; fill q_off / q_req. */
static int prepare(problem_t *p)
{
    if (p->batch < 0 || p->heads <= 0 || p->dl <= 0 || p->dr < 0 || p->page <= 0) return OR_BAD_ARG;
    int64_t acc = 0;
    for (int64_t b = 0; b < p->batch; ++b) {
        int64_t T = p->n_tree[b], L = p->seq_lens[b];
        if (T < 0 || L < T) return OR_BAD_TREE;
        if ((L + p->page - 1) / p->page > p->max_pages) return OR_BAD_ARG;
        p->q_off[b] = acc;
        for (int64_t j = 0; j < T && acc + j < p->total_q; ++j) p->q_req[acc + j] = b;
        acc += T;
    }
    p->q_off[p->batch] = acc;
    if (acc != p->total_q) return OR_BAD_ARG;
    for (int64_t b = 0; b < p->batch; ++b)
        for (int64_t j = 0; j < p->n_tree[b]; ++j) {
            int64_t up = p->parent[p->q_off[b] + j];
            if (up < -1 || up >= j) return OR_BAD_TREE;
        }
    if (p->topk > 0)
        for (int64_t b = 0; b < p->batch; ++b) {
            const int64_t P = p->seq_lens[b] - p->n_tree[b];
            for (int64_t g = p->q_off[b]; g < p->q_off[b + 1]; ++g)
                for (int64_t sl = 0; sl < p->topk; ++sl) {
                    int64_t t = p->topk_idx[g * p->topk + sl];
                    if (t < -1 || t >= P) return OR_BAD_INDEX;
                }
        }
    for (int64_t b = 0; b < p->batch; ++b) {
        int64_t pages = (p->seq_lens[b] + p->page - 1) / p->page;
        for (int64_t k = 0; k < pages; ++k) {
            int64_t slot = p->block_table[b * p->max_pages + k];
            if (slot < 0 || slot >= p->num_pages) return OR_BAD_BLOCK;
        }
    }
    return OR_OK;
}

int mla_oracle_check(const int32_t *block_table, const int32_t *seq_lens,
                     const int32_t *tree_parent, const int32_t *n_tree,
                     int64_t batch, int64_t total_q, int64_t page_size,
                     int64_t max_pages_per_seq, int64_t num_pages)
{
    problem_t p;
    memset(&p, 0, sizeof p);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.parent = tree_parent;
    p.n_tree = n_tree;
    p.batch = batch;
    p.total_q = total_q;
    p.heads = 1;
    p.dl = 1;
    p.page = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.q_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(batch + 1));
    p.q_req = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total_q + 1));
    int st = (p.q_off && p.q_req) ? prepare(&p) : OR_BAD_ARG;
    free(p.q_off);
    free(p.q_req);
    return st;
}

static int verify_rows(const uint16_t *q_lat, const uint16_t *q_rope, const uint16_t *kv_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *tree_parent, const int32_t *n_tree, double scale,
                       int64_t batch, int64_t total_q, int64_t num_heads, int64_t d_latent,
                       int64_t d_rope, int64_t page_size, int64_t max_pages_per_seq,
                       int64_t num_pages, const int64_t *rows, int64_t n_rows,
                       int64_t key_begin, int64_t key_end, double *out, double *lse,
                       int threads, const int32_t *topk_idx, int64_t topk)
{
    problem_t p;
    memset(&p, 0, sizeof p);
    p.q_lat = q_lat;
    p.q_rope = q_rope;
    p.kv = kv_cache;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.parent = tree_parent;
    p.n_tree = n_tree;
    p.batch = batch;
    p.total_q = total_q;
    p.heads = num_heads;
    p.dl = d_latent;
    p.dr = d_rope;
    p.page = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.scale = scale;
    p.topk_idx = topk_idx;
    p.topk = topk;
    if (topk < 0 || (topk > 0 && !topk_idx)) return OR_BAD_ARG;
    if (n_rows < 0 || (n_rows > 0 && (!rows || !out || !lse))) return OR_BAD_ARG;
    p.q_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(batch + 1));
    p.q_req = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total_q + 1));
    int st = (p.q_off && p.q_req) ? prepare(&p) : OR_BAD_ARG;
    for (int64_t r = 0; st == OR_OK && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= total_q * num_heads) st = OR_BAD_ARG;
    if (st == OR_OK && n_rows > 0) {
        long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
        int nt = threads > 0 ? threads : (int)(ncpu > 0 ? ncpu : 1);
        if (nt > n_rows) nt = (int)n_rows;
        job_t job = {&p, rows, n_rows, key_begin, key_end, out, lse, 0, OR_OK};
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
        int started = 0;
        for (int k = 0; tid && k < nt; ++k)
            if (pthread_create(&tid[k], NULL, worker, &job) == 0) ++started;
        if (started == 0) worker(&job);
        for (int k = 0; k < started; ++k) pthread_join(tid[k], NULL);
        free(tid);
        st = job.status;
    }
    free(p.q_off);
    free(p.q_req);
    return st;
}

int mla_oracle_verify_rows(const uint16_t *q_lat, const uint16_t *q_rope, const uint16_t *kv_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *tree_parent, const int32_t *n_tree, double scale,
                           int64_t batch, int64_t total_q, int64_t num_heads, int64_t d_latent,
                           int64_t d_rope, int64_t page_size, int64_t max_pages_per_seq,
                           int64_t num_pages, const int64_t *rows, int64_t n_rows,
                           int64_t key_begin, int64_t key_end, double *out, double *lse,
                           int threads)
{
    return verify_rows(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, batch,
                       total_q, num_heads, d_latent, d_rope, page_size, max_pages_per_seq, num_pages, rows,
                       n_rows, key_begin, key_end, out, lse, threads, NULL, 0);
}

int mla_oracle_verify_sparse_rows(const uint16_t *q_lat, const uint16_t *q_rope, const uint16_t *kv_cache,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  const int32_t *tree_parent, const int32_t *n_tree,
                                  const int32_t *topk_idx, int64_t topk, double scale,
                                  int64_t batch, int64_t total_q, int64_t num_heads, int64_t d_latent,
                                  int64_t d_rope, int64_t page_size, int64_t max_pages_per_seq,
                                  int64_t num_pages, const int64_t *rows, int64_t n_rows,
                                  double *out, double *lse, int threads)
{
    if (topk <= 0) return OR_BAD_ARG;
    return verify_rows(q_lat, q_rope, kv_cache, block_table, seq_lens, tree_parent, n_tree, scale, batch,
                       total_q, num_heads, d_latent, d_rope, page_size, max_pages_per_seq, num_pages, rows,
                       n_rows, 0, INT64_MAX, out, lse, threads, topk_idx, topk);
}

/* Flash-decoding merge of split partials: part_out [n_splits][rows][dv] holds
 * each split's normalised output, part_lse [n_splits][rows] its log-sum-exp
 * (-inf for a split that saw no key). */
int mla_oracle_combine(const double *part_out, const double *part_lse, int64_t n_splits,
                       int64_t rows, int64_t dv, double *out, double *lse)
{
    if (n_splits <= 0 || rows < 0 || dv <= 0) return OR_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int64_t s = 0; s < n_splits; ++s)
            if (part_lse[s * rows + r] > m) m = part_lse[s * rows + r];
        double *o = out + r * dv;
        for (int64_t d = 0; d < dv; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int64_t s = 0; s < n_splits; ++s) z += exp(part_lse[s * rows + r] - m);
#if ORACLE_MUTANT == 10
        double l = m;
#else
        double l = m + log(z);
#endif
        lse[r] = l;
        for (int64_t s = 0; s < n_splits; ++s) {
            double w = exp(part_lse[s * rows + r] - l);
            const double *src = part_out + (s * rows + r) * dv;
            for (int64_t d = 0; d < dv; ++d) o[d] += w * src[d];
        }
    }
    return OR_OK;
}

int mla_oracle_mutant(void) { return ORACLE_MUTANT; }
