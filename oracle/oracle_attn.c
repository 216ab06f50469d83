/*
 * oracle_attn.c -- plain, slow, fp64 CPU oracle for exact causal grouped-query
 * softmax attention over paged K/V.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA path and must never be called by it.
 *
 * What it computes (one output row per (b, q head h, query row i)):
 *
 *   kv head       g  = h / (Hq / Hkv)                       contiguous GQA groups
 *   visible keys  n  = L_b - q_len + i + 1                   queries are the suffix of K/V
 *   key t < n     k_t = k_pages[page_table[b][t / P]][g][t % P][:]   (same for v)
 *   s_t = scale * sum_d q[d] * k_t[d]
 *   o   = sum_t exp(s_t - M) v_t / sum_t exp(s_t - M),   M = max_t s_t
 *   lse = M + log(sum_t exp(s_t - M))
 *
 * Sources (page title, section):
 *  - CFR-Atlas README, "Core contract": folded attention over exact pages must
 *    equal full-KV attention; oracle_attn below is that full-KV definition and
 *    oracle_folded is the page-by-page online-softmax fold that the same
 *    README describes in its opening paragraph and in the "Attention" row of
 *    its responsibility table.
 *  - CFR-Atlas README, "Minimal integration": pages hold row-major K[token][dim]
 *    and V[token][dim] per (layer, K/V head, token range).
 *  - CPUAttn README, "Parallel example": with kv_cache=True the queries are the
 *    suffix of K/V, so query row i sits at position SKV - SQ + i; decode is the
 *    same pattern with one query row ("Operator model").
 *  - CPUAttn README, "Operator model": split-K needs a structured merge;
 *    oracle_state + oracle_merge state that merge.
 *  - ferrox-core crate index, "attention" module: the vanilla causal GQA path
 *    is the correctness baseline.
 *
 * Score and mask variants (ferrox-core crate index: causal_gqa_attention_windowed,
 * _softcap and _sinks; readings of their names, since the index gives no formula):
 *   window W > 0   row i sees only keys pos - W < t <= pos (the W most recent);
 *   softcap c > 0  s_t = c * tanh(scale * <q, k_t> / c);
 *   sinks          one extra logit sink[h] per q head joins the denominator with no
 *                  value row: l += exp(sink[h] - M), M = max(M, sink[h]).
 * W = 0, c = 0 and sinks == NULL give plain attention.
 *
 * Ragged query counts (chunked prefill): with q_lens != NULL sequence b has
 * q_lens[b] <= q_len query rows, the last q_lens[b] positions of its K/V; rows
 * i >= q_lens[b] are padding (output 0, lse NaN).
 *
 * oracle_kv_append is the write before all of this: the new tokens' K and V rows
 * of each sequence go to the page slots of positions seq_lens[b] .. (CFR-Atlas
 * README, "Minimal integration": row-major K[token][dim] per (layer, kv head,
 * range); ferrox-core "cache" module: a KV cache growable one position at a time).
 *
 * All inputs are fp32 arrays holding the exact stored values (bf16 inputs are
 * widened exactly by the caller); all arithmetic is fp64.
 *
 * Return codes: 0 ok, 1 bad argument (shape, GQA ratio), 2 a row has no
 * visible key or its context exceeds the page table, 3 a page id is out of
 * range, 4 out of memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const float *q, *k, *v;
    const int32_t *table, *lens;
    int B, Hq, Hkv, D, P, max_pages, num_pages, q_len;
    double scale;
    int window;          /* 0: none */
    double softcap;      /* 0: none */
    const float *sinks;  /* [Hq] or NULL */
    const int32_t *q_lens; /* [B] query rows per sequence (<= q_len) or NULL */
} problem;

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Query rows of sequence b: q_lens[b] when given (ragged), else q_len. */
static int rows_of(const problem *p, int b) { return p->q_lens ? p->q_lens[b] : p->q_len; }

static int check_problem(const problem *p) {
    if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->P <= 0 ||
        p->max_pages <= 0 || p->num_pages <= 0 || p->q_len <= 0)
        return 1;
    if (p->Hq % p->Hkv != 0) return 1;
    if (p->window < 0 || p->softcap < 0.0) return 1;
    return 0;
}

/* First key row (b, i) may see: the window's lower end, or 0. */
static int64_t first_key(const problem *p, int b, int i) {
    int64_t pos = (int64_t)p->lens[b] - rows_of(p, b) + i;
    if (p->window <= 0) return 0;
    int64_t lo = pos - p->window + 1;
    return lo > 0 ? lo : 0;
}

/* Split a flat row index r = (b * Hq + h) * q_len + i into its parts. */
static void row_parts(const problem *p, int64_t r, int *b, int *h, int *i) {
    *i = (int)(r % p->q_len);
    *h = (int)((r / p->q_len) % p->Hq);
    *b = (int)(r / ((int64_t)p->q_len * p->Hq));
}

/* Number of keys row (b, i) may see, or -1 if the row is invalid. */
static int64_t visible_keys(const problem *p, int b, int i) {
    int64_t L = p->lens[b];
    if (L > (int64_t)p->max_pages * p->P) return -1;
    int64_t n = L - rows_of(p, b) + i + 1;
    return n >= 1 ? n : -1;
}

/* Address of key/value row t of sequence b, kv head g; NULL if the page id is bad. */
static const float *kv_row(const problem *p, const float *pool, int b, int g, int64_t t) {
    int32_t page = p->table[(int64_t)b * p->max_pages + t / p->P];
    if (page < 0 || page >= p->num_pages) return NULL;
    return pool + (((int64_t)page * p->Hkv + g) * p->P + t % p->P) * p->D;
}

static double score(const problem *p, const float *qrow, const float *krow) {
    double acc = 0.0;
    for (int d = 0; d < p->D; ++d) acc += (double)qrow[d] * (double)krow[d];
    double s = p->scale * acc;
    if (p->softcap > 0.0) s = p->softcap * tanh(s / p->softcap);
    return s;
}

/*
 * Full-KV attention, the plain definition.  rows == NULL computes every row into
 * out[(b*Hq+h)*q_len+i][D]; otherwise rows[0..n_rows) lists flat row indices and
 * out[j][D] receives row rows[j].  lse (may be NULL) gets one value per row.
 */
int oracle_attn(const float *q, const float *k_pages, const float *v_pages,
                const int32_t *page_table, const int32_t *seq_lens,
                int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                int q_len, double scale, int window, double softcap, const float *sinks,
                const int32_t *q_lens, const int64_t *rows, int64_t n_rows, double *out,
                double *lse) {
    problem p = {q, k_pages, v_pages, page_table, seq_lens, B, Hq, Hkv, D, P,
                 max_pages, num_pages, q_len, scale, window, softcap, sinks, q_lens};
    if (check_problem(&p)) return 1;
    int64_t total = rows ? n_rows : (int64_t)B * Hq * q_len;
    int G = Hq / Hkv;
    int err = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < total; ++j) {
        int64_t r = rows ? rows[j] : j;
        int b, h, i;
        if (r < 0 || r >= (int64_t)B * Hq * q_len) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        row_parts(&p, r, &b, &h, &i);
        int g = h / G;
        if (q_lens && (q_lens[b] < 0 || q_lens[b] > q_len)) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        if (i >= rows_of(&p, b)) { /* padding row of a ragged batch: not a query */
            for (int d = 0; d < D; ++d) out[j * D + d] = 0.0;
            if (lse) lse[j] = NAN;
            continue;
        }
        int64_t n = visible_keys(&p, b, i);
        if (n < 0) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        const float *qrow = q + r * D;
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = 4;
            continue;
        }
        const int64_t lo = first_key(&p, b, i);
        /* scores of the visible keys lo..n-1 and their maximum (with the sink) */
        double M = -INFINITY;
        int bad = 0;
        for (int64_t t = lo; t < n; ++t) {
            const float *krow = kv_row(&p, k_pages, b, g, t);
            if (!krow) { bad = 1; break; }
            s[t] = score(&p, qrow, krow);
            if (s[t] > M) M = s[t];
        }
        if (bad) {
            free(s);
#pragma omp atomic write
            err = 3;
            continue;
        }
        if (sinks && (double)sinks[h] > M) M = (double)sinks[h];
        /* softmax weights and the weighted sum of value rows */
        double l = 0.0;
        double *o = out + j * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t t = lo; t < n; ++t) {
            double w = exp(s[t] - M);
            l += w;
            const float *vrow = kv_row(&p, v_pages, b, g, t);
            for (int d = 0; d < D; ++d) o[d] += w * (double)vrow[d];
        }
        if (sinks) l += exp((double)sinks[h] - M); /* the sink has no value row */
        for (int d = 0; d < D; ++d) o[d] /= l;
        if (lse) lse[j] = M + log(l);
        free(s);
    }
    return err;
}

/*
 * The page-by-page fold: each page's visible keys update the running state
 *   m' = max(m, max_t s_t),  c = exp(m - m'),
 *   l' = c l + sum_t exp(s_t - m'),  acc' = c acc + sum_t exp(s_t - m') v_t
 * in logical page order; the sink, if any, is folded last as a key with no
 * value; o = acc / l at the end.  Same argument convention as oracle_attn.
 * Used only to check the fold against the full-KV definition.
 */
int oracle_folded(const float *q, const float *k_pages, const float *v_pages,
                  const int32_t *page_table, const int32_t *seq_lens,
                  int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                  int q_len, double scale, int window, double softcap, const float *sinks,
                  const int32_t *q_lens, const int64_t *rows, int64_t n_rows, double *out,
                  double *lse) {
    problem p = {q, k_pages, v_pages, page_table, seq_lens, B, Hq, Hkv, D, P,
                 max_pages, num_pages, q_len, scale, window, softcap, sinks, q_lens};
    if (check_problem(&p)) return 1;
    int64_t total = rows ? n_rows : (int64_t)B * Hq * q_len;
    int G = Hq / Hkv;
    int err = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < total; ++j) {
        int64_t r = rows ? rows[j] : j;
        int b, h, i;
        if (r < 0 || r >= (int64_t)B * Hq * q_len) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        row_parts(&p, r, &b, &h, &i);
        int g = h / G;
        if (q_lens && (q_lens[b] < 0 || q_lens[b] > q_len)) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        if (i >= rows_of(&p, b)) {
            for (int d = 0; d < D; ++d) out[j * D + d] = 0.0;
            if (lse) lse[j] = NAN;
            continue;
        }
        int64_t n = visible_keys(&p, b, i);
        if (n < 0) {
#pragma omp atomic write
            err = 2;
            continue;
        }
        const float *qrow = q + r * D;
        double *acc = out + j * D;
        double *s = (double *)malloc((size_t)P * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = 4;
            continue;
        }
        const int64_t lo = first_key(&p, b, i);
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        double m = -INFINITY, l = 0.0;
        int bad = 0;
        for (int64_t pg = lo / P; pg * P < n && !bad; ++pg) {
            int64_t t0 = pg * P > lo ? pg * P : lo;
            int64_t t1 = pg * P + P < n ? pg * P + P : n;
            double m_page = -INFINITY;
            for (int64_t t = t0; t < t1; ++t) {
                const float *krow = kv_row(&p, k_pages, b, g, t);
                if (!krow) { bad = 1; break; }
                s[t - t0] = score(&p, qrow, krow);
                if (s[t - t0] > m_page) m_page = s[t - t0];
            }
            if (bad) break;
            double m_new = m_page > m ? m_page : m;
            double c = exp(m - m_new); /* exp(-inf) = 0 on the first page */
            l *= c;
            for (int d = 0; d < D; ++d) acc[d] *= c;
            for (int64_t t = t0; t < t1; ++t) {
                double w = exp(s[t - t0] - m_new);
                const float *vrow = kv_row(&p, v_pages, b, g, t);
                l += w;
                for (int d = 0; d < D; ++d) acc[d] += w * (double)vrow[d];
            }
            m = m_new;
        }
        free(s);
        if (bad) {
#pragma omp atomic write
            err = 3;
            continue;
        }
        if (sinks) {
            double sk = (double)sinks[h];
            double m_new = sk > m ? sk : m;
            double cs = exp(m - m_new);
            for (int d = 0; d < D; ++d) acc[d] *= cs;
            l = l * cs + exp(sk - m_new);
            m = m_new;
        }
        for (int d = 0; d < D; ++d) acc[d] /= l;
        if (lse) lse[j] = m + log(l);
    }
    return err;
}

/*
 * Unnormalised softmax state of one row over the visible keys in
 * [t_begin, t_end): m = max s_t, l = sum exp(s_t - m), acc = sum exp(s_t - m) v_t.
 * Window and softcap apply; the sink does not (it is one more state: m = sink,
 * l = 1, acc = 0).  An empty range gives m = -inf, l = 0, acc = 0.  One row per
 * call (flat index r).
 */
int oracle_state(const float *q, const float *k_pages, const float *v_pages,
                 const int32_t *page_table, const int32_t *seq_lens,
                 int B, int Hq, int Hkv, int D, int P, int max_pages, int num_pages,
                 int q_len, double scale, int window, double softcap, int64_t r,
                 int64_t t_begin, int64_t t_end, double *m_out, double *l_out, double *acc) {
    problem p = {q, k_pages, v_pages, page_table, seq_lens, B, Hq, Hkv, D, P,
                 max_pages, num_pages, q_len, scale, window, softcap, NULL, NULL};
    if (check_problem(&p)) return 1;
    if (r < 0 || r >= (int64_t)B * Hq * q_len) return 1;
    int b, h, i;
    row_parts(&p, r, &b, &h, &i);
    int g = h / (Hq / Hkv);
    int64_t n = visible_keys(&p, b, i);
    if (n < 0) return 2;
    int64_t lo = first_key(&p, b, i);
    if (t_begin < lo) t_begin = lo;
    if (t_end > n) t_end = n;
    const float *qrow = q + r * D;
    double m = -INFINITY;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const float *krow = kv_row(&p, k_pages, b, g, t);
        if (!krow) return 3;
        double s = score(&p, qrow, krow);
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int64_t t = t_begin; t < t_end; ++t) {
        double w = exp(score(&p, qrow, kv_row(&p, k_pages, b, g, t)) - m);
        const float *vrow = kv_row(&p, v_pages, b, g, t);
        l += w;
        for (int d = 0; d < D; ++d) acc[d] += w * (double)vrow[d];
    }
    *m_out = m;
    *l_out = l;
    return 0;
}

/*
 * Structured merge of S partial states of one row:
 *   M = max_s m_s,  l = sum_s exp(m_s - M) l_s,  o = sum_s exp(m_s - M) acc_s / l,
 *   lse = M + log(l).  States with l_s == 0 (empty ranges) contribute nothing.
 */
int oracle_merge(int S, int D, const double *m, const double *l, const double *acc,
                 double *out, double *lse) {
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (l[s] > 0.0 && m[s] > M) M = m[s];
    if (M == -INFINITY) return 2;
    double L = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int s = 0; s < S; ++s) {
        if (l[s] <= 0.0) continue;
        double w = exp(m[s] - M);
        L += w * l[s];
        for (int d = 0; d < D; ++d) out[d] += w * acc[(int64_t)s * D + d];
    }
    for (int d = 0; d < D; ++d) out[d] /= L;
    if (lse) *lse = M + log(L);
    return 0;
}

/*
 * Append: for each sequence b, kv head g and new token j < n_new[b] (n_new == NULL:
 * all max_new), write k_new[b][g][j][:] (and v_new) to the page slot of position
 * t = seq_lens[b] + j:  pools[page_table[b][t / P]][g][t % P][:].  Pools are
 * float32 here.  Returns 3 for a page id outside the pool, 2 for a position past
 * the page table.
 */
int oracle_kv_append(const float *k_new, const float *v_new, float *k_pages, float *v_pages,
                     const int32_t *page_table, const int32_t *seq_lens, const int32_t *n_new,
                     int B, int Hkv, int max_new, int D, int P, int max_pages, int num_pages) {
    for (int b = 0; b < B; ++b) {
        int cnt = n_new ? n_new[b] : max_new;
        if (cnt < 0 || cnt > max_new) return 1;
        for (int j = 0; j < cnt; ++j) {
            int64_t t = (int64_t)seq_lens[b] + j;
            if (t >= (int64_t)max_pages * P) return 2;
            int32_t page = page_table[(int64_t)b * max_pages + t / P];
            if (page < 0 || page >= num_pages) return 3;
            for (int g = 0; g < Hkv; ++g) {
                const int64_t src = (((int64_t)b * Hkv + g) * max_new + j) * D;
                const int64_t dst = (((int64_t)page * Hkv + g) * P + t % P) * D;
                for (int d = 0; d < D; ++d) {
                    k_pages[dst + d] = k_new[src + d];
                    v_pages[dst + d] = v_new[src + d];
                }
            }
        }
    }
    return 0;
}
