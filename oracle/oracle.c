/*
 * oracle.c -- fp64 CPU oracle for shared-prefix fan-out attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The product path
 * (the CUDA library) never calls it, links it or shares code with it.
 *
 * What it computes is the plain definition of attention over each branch's
 * logical context, with no tiling, no online softmax and no batching:
 *
 *   - Fork ("AHBM Agentic Runtime Architecture", section 3.1 "Fan-out context
 *     structure"): branch b's page table is the shared prefix pages followed by
 *     its own private pages; shared pages are referenced, never copied.
 *   - Row independence (same page, section 3.2 "Sub-agent query batching" and
 *     section 3.4 "Online softmax merge"): every query row attends on its own;
 *     batching rows changes the execution shape, not the result.  So the oracle
 *     simply loops over rows.
 *   - GQA (ADR-0060, section 0 "reference dimensions", and TL;DR): query head h
 *     reads KV head h / G, G = H_q / H_kv. Here written as an explicit
 *     head broadcast, not a fold of rows into M.
 *   - Causality (ADR-0060, section 5.4 "PREFILL, no SP"): key j is visible to
 *     a query at absolute position pos iff j <= pos (the diagonal is visible:
 *     a token's own K/V is in the cache before the kernel runs, section 0.5.1
 *     precondition P3). New query tokens are the tail of their branch's
 *     suffix: pos = P + S_b - T_b + t.
 *   - Softmax with scale (ADR-0060, section 0.5.3 "softmax_scale"):
 *     s_j = scale * <q, k_j>, out = sum_j exp(s_j - M) v_j / Z,
 *     M = max_j s_j, Z = sum_j exp(s_j - M); lse = M + ln Z (natural log).
 *     Two passes (max, then exp-sum), all in double from the exact bf16 values.
 *   - Cache append (ADR-0060, section 0.5.1, precondition P3: the new K/V rows
 *     are written before attention runs, so attention is a pure read): a
 *     branch's new tokens go to the next positions of its private suffix,
 *     with pages taken from the free list as the suffix grows.
 *   - Partial state and merge (ADR-0060, section 4 "Reduction", and
 *     "AHBM Agentic Runtime Architecture" section 3.4): a partial over a key
 *     subset is (m, l, o) with o unnormalised; two partials merge as
 *     m = max(m_a, m_b), s_a = exp(m_a - m), s_b = exp(m_b - m),
 *     l = l_a s_a + l_b s_b, o = o_a s_a + o_b s_b; the final output is o / l.
 *
 * Layouts (all row-major, bf16 given as uint16 bit patterns):
 *   q        [R][H_q][d]                R = sum_b T_b, rows grouped by branch
 *   k_pool   [num_pages][H_kv][page][d] (v_pool the same)
 *   table    [B][max_pages]             physical page ids, -1 = unused
 *   out      [n][H_q][d] double, lse [n][H_q] double, for the n tokens asked for
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Branch page tables: prefix pages, then each branch's private pages taken in
 * order from the free list (branch 0 first). Returns 0, or -1 when the free
 * list or the table width is too small. */
int oracle_fork(const int32_t *prefix_pages, int32_t n_prefix_pages, int32_t num_branches,
                const int32_t *suffix_lens, int32_t page_size, const int32_t *free_pages,
                int32_t n_free, int32_t *table, int32_t max_pages) {
    int32_t next_free = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        int32_t n_private = (suffix_lens[b] + page_size - 1) / page_size;
        if (n_prefix_pages + n_private > max_pages) return -1;
        if (next_free + n_private > n_free) return -1;
        int32_t *row = table + (int64_t)b * max_pages;
        for (int32_t i = 0; i < max_pages; ++i) row[i] = -1;
        for (int32_t i = 0; i < n_prefix_pages; ++i) row[i] = prefix_pages[i];
        for (int32_t i = 0; i < n_private; ++i) row[n_prefix_pages + i] = free_pages[next_free++];
    }
    return 0;
}

/* Logical key j of branch b, KV head h: its d-vector in the pool. */
static const uint16_t *kv_row(const uint16_t *pool, const int32_t *table, int32_t max_pages,
                              int32_t b, int32_t j, int32_t h, int32_t H_kv, int32_t page,
                              int32_t d) {
    int32_t phys = table[(int64_t)b * max_pages + j / page];
    int64_t off = (((int64_t)phys * H_kv + h) * page + (j % page)) * (int64_t)d;
    return pool + off;
}

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *table;
    int32_t max_pages, P;
    const int32_t *S, *T;
    int32_t B, H_q, H_kv, d, page;
    double scale;
    int causal;
} problem;

/* branch of global token r and its index t inside the branch */
static void locate(const problem *pb, int32_t r, int32_t *b_out, int32_t *t_out) {
    int32_t start = 0;
    for (int32_t b = 0; b < pb->B; ++b) {
        if (r < start + pb->T[b]) {
            *b_out = b;
            *t_out = r - start;
            return;
        }
        start += pb->T[b];
    }
    *b_out = -1;
    *t_out = -1;
}

/* Number of keys visible to token r: keys 0 .. n-1 of its branch. */
static int32_t visible_keys(const problem *pb, int32_t b, int32_t t) {
    int32_t n = pb->P + pb->S[b];
    if (pb->causal) {
        int32_t pos = pb->P + pb->S[b] - pb->T[b] + t;
        if (pos + 1 < n) n = pos + 1;
    }
    return n;
}

/* Scores of (token r, query head h) against keys [lo, hi) of its branch. */
static void scores(const problem *pb, int32_t r, int32_t h, int32_t b, int32_t lo, int32_t hi,
                   double *s) {
    int32_t G = pb->H_q / pb->H_kv;
    int32_t hk = h / G;
    const uint16_t *qv = pb->q + ((int64_t)r * pb->H_q + h) * pb->d;
    for (int32_t j = lo; j < hi; ++j) {
        const uint16_t *kr = kv_row(pb->k, pb->table, pb->max_pages, b, j, hk, pb->H_kv, pb->page,
                                    pb->d);
        double acc = 0.0;
        for (int32_t i = 0; i < pb->d; ++i) acc += bf16_to_double(qv[i]) * bf16_to_double(kr[i]);
        s[j - lo] = pb->scale * acc;
    }
}

/* Unnormalised partial (m, l, o) of (token r, head h) over keys [lo, hi) clipped to
 * the visible keys. An empty range gives m = -inf, l = 0, o = 0. */
static void partial_one(const problem *pb, int32_t r, int32_t h, int32_t lo, int32_t hi,
                        double *s, double *m_out, double *l_out, double *o_out) {
    int32_t b, t;
    locate(pb, r, &b, &t);
    int32_t n = visible_keys(pb, b, t);
    if (hi > n) hi = n;
    if (lo < 0) lo = 0;
    for (int32_t i = 0; i < pb->d; ++i) o_out[i] = 0.0;
    if (hi <= lo) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    scores(pb, r, h, b, lo, hi, s);
    double M = -INFINITY;
    for (int32_t j = 0; j < hi - lo; ++j)
        if (s[j] > M) M = s[j];
    double Z = 0.0;
    int32_t hk = h / (pb->H_q / pb->H_kv);
    for (int32_t j = lo; j < hi; ++j) {
        double p = exp(s[j - lo] - M);
        Z += p;
        const uint16_t *vr = kv_row(pb->v, pb->table, pb->max_pages, b, j, hk, pb->H_kv, pb->page,
                                    pb->d);
        for (int32_t i = 0; i < pb->d; ++i) o_out[i] += p * bf16_to_double(vr[i]);
    }
    *m_out = M;
    *l_out = Z;
}

static int32_t max_keys(const problem *pb) {
    int32_t mx = 1;
    for (int32_t b = 0; b < pb->B; ++b)
        if (pb->P + pb->S[b] > mx) mx = pb->P + pb->S[b];
    return mx;
}

/* Full attention for the listed tokens (all tokens when rows == NULL).
 * out [n][H_q][d], lse [n][H_q]. Returns 0, -1 on a bad token index. */
int oracle_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                const int32_t *table, int32_t max_pages, int32_t P, const int32_t *S,
                const int32_t *T, int32_t B, int32_t H_q, int32_t H_kv, int32_t d, int32_t page,
                double scale, int causal, const int32_t *rows, int32_t n_rows, double *out,
                double *lse) {
    problem pb = {q, k_pool, v_pool, table, max_pages, P, S, T, B, H_q, H_kv, d, page, scale,
                  causal};
    int32_t R = 0;
    for (int32_t b = 0; b < B; ++b) R += T[b];
    if (rows == NULL) n_rows = R;
    for (int32_t i = 0; i < n_rows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= R)) return -1;
    int32_t nk = max_keys(&pb);
    int64_t n_tasks = (int64_t)n_rows * H_q;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)nk);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < n_tasks; ++task) {
            int32_t i = (int32_t)(task / H_q), h = (int32_t)(task % H_q);
            int32_t r = rows ? rows[i] : i;
            double m, l;
            partial_one(&pb, r, h, 0, nk, s, &m, &l, o);
            double *dst = out + ((int64_t)i * H_q + h) * d;
            if (l > 0.0) {
                for (int32_t c = 0; c < d; ++c) dst[c] = o[c] / l;
                lse[(int64_t)i * H_q + h] = m + log(l);
            } else { /* no visible key: cannot happen for a valid problem */
                for (int32_t c = 0; c < d; ++c) dst[c] = NAN;
                lse[(int64_t)i * H_q + h] = NAN;
#pragma omp atomic write
                bad = 1;
            }
        }
        free(s);
        free(o);
    }
    return bad ? -2 : 0;
}

/* Partial state over keys [lo, hi) of each token's branch (natural-log domain).
 * m, l [n][H_q]; o [n][H_q][d] unnormalised. */
int oracle_attn_partial(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        const int32_t *table, int32_t max_pages, int32_t P, const int32_t *S,
                        const int32_t *T, int32_t B, int32_t H_q, int32_t H_kv, int32_t d,
                        int32_t page, double scale, int causal, const int32_t *rows,
                        int32_t n_rows, int32_t lo, int32_t hi, double *m, double *l, double *o) {
    problem pb = {q, k_pool, v_pool, table, max_pages, P, S, T, B, H_q, H_kv, d, page, scale,
                  causal};
    int32_t R = 0;
    for (int32_t b = 0; b < B; ++b) R += T[b];
    if (rows == NULL) n_rows = R;
    int32_t nk = hi - lo > 1 ? hi - lo : 1;
    int64_t n_tasks = (int64_t)n_rows * H_q;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)nk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < n_tasks; ++task) {
            int32_t i = (int32_t)(task / H_q), h = (int32_t)(task % H_q);
            int32_t r = rows ? rows[i] : i;
            partial_one(&pb, r, h, lo, hi, s, m + task, l + task, o + task * d);
        }
        free(s);
    }
    return 0;
}

/* Fold n_parts partial states per output, in the given order, with the pairwise
 * merge; then normalise. parts_m/l [n_parts][n], parts_o [n_parts][n][d].
 * Writes out [n][d] = o / l and lse [n] = m + ln l. */
void oracle_merge(const double *parts_m, const double *parts_l, const double *parts_o,
                  int32_t n_parts, int64_t n, int32_t d, double *out, double *lse) {
    for (int64_t i = 0; i < n; ++i) {
        double m = -INFINITY, l = 0.0;
        double *acc = out + i * d;
        for (int32_t c = 0; c < d; ++c) acc[c] = 0.0;
        for (int32_t p = 0; p < n_parts; ++p) {
            double mb = parts_m[(int64_t)p * n + i], lb = parts_l[(int64_t)p * n + i];
            const double *ob = parts_o + ((int64_t)p * n + i) * d;
            double mn = m > mb ? m : mb;
            if (mn == -INFINITY) continue; /* both empty: state stays empty */
            double sa = exp(m - mn), sb = exp(mb - mn);
            l = l * sa + lb * sb;
            for (int32_t c = 0; c < d; ++c) acc[c] = acc[c] * sa + ob[c] * sb;
            m = mn;
        }
        for (int32_t c = 0; c < d; ++c) acc[c] /= l;
        lse[i] = m + log(l);
    }
}

/* Fork when the prefix may end inside a page: the whole prefix pages are
 * shared; a partially filled last prefix page is given to each branch as its
 * own copy (a fresh page from the free list, filled by oracle_copy_pages),
 * followed by the branch's suffix pages; pages are taken in order, branch 0
 * first. cow[b] = {shared partial page, branch's copy} when the prefix ends
 * inside a page. Returns the number of free pages used, or -1. */
int oracle_fork_cow(const int32_t *prefix_pages, int32_t prefix_len, int32_t num_branches,
                    const int32_t *suffix_lens, int32_t page_size, const int32_t *free_pages,
                    int32_t n_free, int32_t *table, int32_t max_pages, int32_t *cow) {
    int32_t n_full = prefix_len / page_size;
    int32_t partial = (prefix_len % page_size) != 0;
    int32_t used = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        int32_t need = (prefix_len + suffix_lens[b] + page_size - 1) / page_size;
        if (need < n_full + partial) need = n_full + partial;
        if (need > max_pages) return -1;
        int32_t *row = table + (int64_t)b * max_pages;
        for (int32_t i = 0; i < max_pages; ++i) row[i] = -1;
        for (int32_t i = 0; i < n_full; ++i) row[i] = prefix_pages[i];
        for (int32_t i = n_full; i < need; ++i) {
            if (used >= n_free) return -1;
            row[i] = free_pages[used++];
        }
        if (partial) {
            cow[2 * b] = prefix_pages[n_full];
            cow[2 * b + 1] = row[n_full];
        }
    }
    return used;
}

/* Copy token slots [0, rows) of page pairs[i][0] to page pairs[i][1] (every
 * KV head, both pools). */
void oracle_copy_pages(uint16_t *k_pool, uint16_t *v_pool, const int32_t *pairs, int32_t n_pairs,
                       int32_t rows, int32_t H_kv, int32_t page, int32_t d) {
    for (int32_t i = 0; i < n_pairs; ++i)
        for (int32_t h = 0; h < H_kv; ++h)
            for (int32_t s = 0; s < rows; ++s) {
                int64_t src = (((int64_t)pairs[2 * i] * H_kv + h) * page + s) * (int64_t)d;
                int64_t dst = (((int64_t)pairs[2 * i + 1] * H_kv + h) * page + s) * (int64_t)d;
                for (int32_t c = 0; c < d; ++c) {
                    k_pool[dst + c] = k_pool[src + c];
                    v_pool[dst + c] = v_pool[src + c];
                }
            }
}

/* Grow branch page tables for new tokens: branch b's context goes from
 * prefix_len + suffix_lens[b] to prefix_len + suffix_lens[b] + add_lens[b]
 * tokens, logical position j living in table entry j / page ("AHBM Agentic
 * Runtime Architecture" section 3.1: shared prefix pages, then the branch's
 * private pages). The entries it now needs beyond its current
 * ceil((prefix_len + suffix_lens[b]) / page) come from free_pages in order
 * (branch 0 first). A prefix ending inside a page needs no special case: its
 * last page is already held (privately, after copy-on-write). Returns the
 * number of free pages used, or -1 when the free list or a table row is too
 * short. */
int oracle_extend(int32_t *table, int32_t num_branches, int32_t max_pages, int32_t prefix_len,
                  const int32_t *suffix_lens, const int32_t *add_lens, int32_t page_size,
                  const int32_t *free_pages, int32_t n_free) {
    int32_t used = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        int64_t len0 = (int64_t)prefix_len + suffix_lens[b];
        int64_t len1 = len0 + add_lens[b];
        int64_t have = (len0 + page_size - 1) / page_size;
        int64_t need = (len1 + page_size - 1) / page_size;
        if (need > max_pages) return -1;
        for (int64_t i = have; i < need; ++i) {
            if (used >= n_free) return -1;
            table[(int64_t)b * max_pages + i] = free_pages[used++];
        }
    }
    return used;
}

/* Write new K/V rows into the paged pool (the cache write that precedes
 * attention: ADR-0060 section 0.5.1, precondition P3). Row r = token t of
 * branch b (rows grouped by branch) goes to logical position
 * prefix_len + suffix_lens[b] + t of branch b, for every KV head.
 * k_new/v_new [R][H_kv][d]; pools [num_pages][H_kv][page][d]. */
void oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                      uint16_t *v_pool, const int32_t *table, int32_t max_pages,
                      int32_t prefix_len, const int32_t *suffix_lens, const int32_t *add_lens,
                      int32_t num_branches, int32_t H_kv, int32_t d, int32_t page) {
    int32_t r = 0;
    for (int32_t b = 0; b < num_branches; ++b) {
        for (int32_t t = 0; t < add_lens[b]; ++t, ++r) {
            int32_t j = prefix_len + suffix_lens[b] + t;
            int32_t phys = table[(int64_t)b * max_pages + j / page];
            for (int32_t h = 0; h < H_kv; ++h) {
                int64_t dst = (((int64_t)phys * H_kv + h) * page + (j % page)) * (int64_t)d;
                int64_t src = ((int64_t)r * H_kv + h) * (int64_t)d;
                for (int32_t i = 0; i < d; ++i) {
                    k_pool[dst + i] = k_new[src + i];
                    v_pool[dst + i] = v_new[src + i];
                }
            }
        }
    }
}

/* Number of visible (token, query head, key) triples: the attention work.
 * Each triple costs 2 d multiply-adds (q.k and p.v), i.e. 4 d flops. */
int64_t oracle_count_pairs(int32_t P, const int32_t *S, const int32_t *T, int32_t B, int32_t H_q,
                           int causal) {
    int64_t total = 0;
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t t = 0; t < T[b]; ++t) {
            int64_t n = (int64_t)P + S[b];
            if (causal) {
                int64_t pos = (int64_t)P + S[b] - T[b] + t;
                if (pos + 1 < n) n = pos + 1;
            }
            total += n;
        }
    }
    return total * H_q;
}
