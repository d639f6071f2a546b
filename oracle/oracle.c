/*
 * oracle.c -- plain, slow, double-precision CPU oracle for softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or constant with the
 * CUDA kernels.
 *
 * What it computes (all arithmetic in IEEE double, no fast-math):
 *
 *   x_ij = scale * sum_c q[i,c] * k[j,c]        over visible keys j
 *   O[i] = sum_j exp(x_ij - m_i) v[j] / l_i,    m_i = max_j x_ij,
 *   l_i  = sum_j exp(x_ij - m_i),               LSE_i = m_i + ln l_i
 *
 * "visible" is j in [0, N) for full attention and j in [0, i] for causal
 * attention (a key after the query is masked, "Online Softmax: Tiling Across
 * a Reduction", section on causal attention).  Inputs are bf16 bit patterns;
 * the oracle widens each one to double exactly, so it sees precisely the
 * values the GPU sees.
 *
 * Two independent routes are provided:
 *
 *  - oracle_attention_three_pass: the safe softmax of the infra-guide page
 *    "5.2 CUDA Online Softmax", section 1.1 (max pass, exp-sum pass,
 *    normalise pass), applied to one row of scores at a time, as the
 *    double-precision host reference of "LLM kernels 3: attention and
 *    online softmax" (section "Two paths, one head, one reference") does.
 *
 *  - oracle_attention_online: the running (max, sum, accumulator) update,
 *    key tile by key tile: m_new = max(m_old, tile max), every carried
 *    quantity scaled by exp(m_old - m_new), division by the sum once at the
 *    end ("Online softmax, and the register that can't move", section
 *    "Online softmax"; "LLM kernels 3", section "Softmax needs the whole
 *    row, and does not").  A tile of 1 is the scalar recurrence of the
 *    infra-guide page, section 2.1.
 *
 *  - oracle_attention_backward: gradients dQ, dK, dV of L = sum(O * dO),
 *    the scores recomputed from Q and K and normalised with the saved LSE
 *    ("Online Softmax: Tiling Across a Reduction", backward-pass section).
 *
 *  - oracle_attention_masked: the three-pass route over the keys a general
 *    mask leaves visible -- a window of keys around the query and, when
 *    document ids are given, only keys of the query's own document (the
 *    structured masks of "Online Softmax: Tiling Across a Reduction", causal
 *    section, last paragraph).  The predicate is applied key by key; nothing
 *    is skipped by blocks.
 *
 * The softmax-only functions follow the infra-guide page: three-pass safe
 * softmax (section 1.1), the online recurrence (sections 2.1-2.2) and the
 * associative (m, d) merge (section 4.1).
 *
 * `mutation` plants a known mistake in the online route so that the tests
 * can show their pins catch it (the two canonical bugs named in "LLM
 * kernels 3", Exercise/Check, and the update-order bug of its Pitfalls).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_MUT_NONE 0
#define ORACLE_MUT_NO_RESCALE 1      /* accumulator not scaled when the max moves */
#define ORACLE_MUT_NORMALISE_TILE 2  /* divide by the running sum per tile, not once at the end */
#define ORACLE_MUT_SUM_BEFORE_MAX 3  /* update the sum against the old max, then the max */

static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* score x_ij in double from bf16 rows */
static double score(const uint16_t* qrow, const uint16_t* krow, int64_t d, double scale) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
    return scale * acc;
}

/* number of keys query i may see */
static int64_t visible_keys(int64_t i, int64_t N, int causal) { return causal ? (i + 1 < N ? i + 1 : N) : N; }

/* ------------------------------------------------------------------------ */
/* Softmax of one vector.                                                    */
/* ------------------------------------------------------------------------ */

/* Safe softmax in three passes: max, sum of exp(x - max), normalise. */
void oracle_softmax_three_pass(const double* x, int64_t n, double* y) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) m = x[j] > m ? x[j] : m;          /* pass 1 */
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(x[j] - m);               /* pass 2 */
    for (int64_t j = 0; j < n; ++j) y[j] = exp(x[j] - m) / l;         /* pass 3 */
}

/* Online normaliser: one pass keeps (m, d); a second pass normalises. */
void oracle_softmax_online(const double* x, int64_t n, double* y, double* m_out, double* d_out) {
    double m = -INFINITY, d = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double m_new = x[j] > m ? x[j] : m;
        /* exp(-inf - finite) = 0 wipes the empty initial state; when both are
           -inf there is nothing to correct, so the factor is 1 (the NaN trap
           of the infra-guide page, section 4.3). */
        double corr = (m_new == -INFINITY) ? 1.0 : exp(m - m_new);
        double term = (m_new == -INFINITY) ? 0.0 : exp(x[j] - m_new);
        d = d * corr + term;
        m = m_new;
    }
    for (int64_t j = 0; j < n; ++j) y[j] = exp(x[j] - m) / d;
    if (m_out) *m_out = m;
    if (d_out) *d_out = d;
}

/* Merge two partial (m, d) results: the associative rule. */
void oracle_online_merge(double m1, double d1, double m2, double d2, double* m, double* d) {
    double mm = m1 > m2 ? m1 : m2;
    if (mm == -INFINITY) { /* both empty */
        *m = -INFINITY;
        *d = 0.0;
        return;
    }
    *m = mm;
    *d = d1 * exp(m1 - mm) + d2 * exp(m2 - mm);
}

/* ------------------------------------------------------------------------ */
/* Attention, one query row.                                                 */
/* ------------------------------------------------------------------------ */

/* Three-pass safe softmax over one row of scores, then the weighted sum of V. */
static void row_three_pass(const uint16_t* qrow, const uint16_t* kh, const uint16_t* vh, int64_t nvis, int64_t d,
                           double scale, double* xbuf, double* o, double* lse) {
    for (int64_t j = 0; j < nvis; ++j) xbuf[j] = score(qrow, kh + j * d, d, scale);
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) m = xbuf[j] > m ? xbuf[j] : m;
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) l += exp(xbuf[j] - m);
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double w = exp(xbuf[j] - m) / l;
        const uint16_t* vrow = vh + j * d;
        for (int64_t c = 0; c < d; ++c) o[c] += w * bf16_bits_to_double(vrow[c]);
    }
    *lse = m + log(l);
}

/*
 * Online state over keys [j0, j1) of one query row, processed in tiles of
 * `tile` keys: returns the running max m, the running sum l (against m) and
 * the unnormalised accumulator acc (against m).  Keys past `jvis` (exclusive)
 * are masked.
 */
void oracle_row_online_state(const uint16_t* qrow, const uint16_t* kh, const uint16_t* vh, int64_t d, int64_t j0,
                             int64_t j1, int64_t jvis, int64_t tile, double scale, int mutation, double* m_out,
                             double* l_out, double* acc) {
    double m = -INFINITY, l = 0.0;
    for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
    if (tile < 1) tile = 1;
    double* contrib = (double*)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
    if (j1 > jvis) j1 = jvis;
    for (int64_t t0 = j0; t0 < j1; t0 += tile) {
        int64_t t1 = t0 + tile < j1 ? t0 + tile : j1;
        /* tile maximum */
        double tmax = -INFINITY;
        for (int64_t j = t0; j < t1; ++j) {
            double x = score(qrow, kh + j * d, d, scale);
            tmax = x > tmax ? x : tmax;
        }
        if (mutation == ORACLE_MUT_SUM_BEFORE_MAX) {
            /* wrong order: add the tile against the OLD max, then move the max */
            for (int64_t j = t0; j < t1; ++j) {
                double e = exp(score(qrow, kh + j * d, d, scale) - m);
                l += e;
                const uint16_t* vrow = vh + j * d;
                for (int64_t c = 0; c < d; ++c) acc[c] += e * bf16_bits_to_double(vrow[c]);
            }
            m = tmax > m ? tmax : m;
            continue;
        }
        double m_new = tmax > m ? tmax : m;
        /* correction factor; the empty state (m = -inf) is wiped by exp(-inf) = 0 */
        double alpha = (m_new == -INFINITY) ? 1.0 : exp(m - m_new);
        double tsum = 0.0;
        for (int64_t c = 0; c < d; ++c) contrib[c] = 0.0;
        for (int64_t j = t0; j < t1; ++j) {
            double e = (m_new == -INFINITY) ? 0.0 : exp(score(qrow, kh + j * d, d, scale) - m_new);
            tsum += e;
            const uint16_t* vrow = vh + j * d;
            for (int64_t c = 0; c < d; ++c) contrib[c] += e * bf16_bits_to_double(vrow[c]);
        }
        double l_new = l * alpha + tsum;
        for (int64_t c = 0; c < d; ++c) {
            double carried = (mutation == ORACLE_MUT_NO_RESCALE) ? acc[c] : acc[c] * alpha;
            if (mutation == ORACLE_MUT_NORMALISE_TILE)
                acc[c] = carried + contrib[c] / l_new; /* per-tile normalisation, no final division */
            else
                acc[c] = carried + contrib[c];
        }
        l = l_new;
        m = m_new;
    }
    free(contrib);
    *m_out = m;
    *l_out = l;
}

/* Merge two partial attention states (m, l, acc[d]); associative. */
void oracle_state_merge(double m1, double l1, const double* acc1, double m2, double l2, const double* acc2, int64_t d,
                        double* m, double* l, double* acc) {
    double mm = m1 > m2 ? m1 : m2;
    if (mm == -INFINITY) {
        *m = -INFINITY;
        *l = 0.0;
        for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
        return;
    }
    double a1 = exp(m1 - mm), a2 = exp(m2 - mm);
    *m = mm;
    *l = l1 * a1 + l2 * a2;
    for (int64_t c = 0; c < d; ++c) acc[c] = acc1[c] * a1 + acc2[c] * a2;
}

/*
 * Is key j visible to query i of batch b?  window_left < 0 / window_right < 0
 * mean unbounded on that side; doc (int32 [B][N]) may be NULL.
 */
static int key_visible(int64_t b, int64_t i, int64_t j, int64_t N, int64_t window_left, int64_t window_right,
                       const int32_t* doc) {
    if (window_left >= 0 && j < i - window_left) return 0;
    if (window_right >= 0 && j > i + window_right) return 0;
    if (doc && doc[b * N + i] != doc[b * N + j]) return 0;
    return 1;
}

/* Three-pass safe softmax over the visible keys of one row, then the weighted
   sum of V.  No visible key: o = 0, lse = -inf. */
static void row_three_pass_masked(const uint16_t* qrow, const uint16_t* kh, const uint16_t* vh, int64_t b, int64_t i,
                                  int64_t N, int64_t d, double scale, int64_t wl, int64_t wr, const int32_t* doc,
                                  double* xbuf, double* o, double* lse) {
    for (int64_t j = 0; j < N; ++j)
        xbuf[j] = key_visible(b, i, j, N, wl, wr, doc) ? score(qrow, kh + j * d, d, scale) : -INFINITY;
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) m = xbuf[j] > m ? xbuf[j] : m;
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) l += exp(xbuf[j] - m);
    for (int64_t j = 0; j < N; ++j) {
        if (xbuf[j] == -INFINITY) continue;
        double w = exp(xbuf[j] - m) / l;
        const uint16_t* vrow = vh + j * d;
        for (int64_t c = 0; c < d; ++c) o[c] += w * bf16_bits_to_double(vrow[c]);
    }
    *lse = m + log(l);
}

/* ------------------------------------------------------------------------ */
/* Batched drivers: [B][H][N][d] bf16 tensors, rows given as bh*N + i.       */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q, *k, *v;
    int64_t N, d;
    int causal;
    double scale;
    const int64_t* rows;
    int64_t n_rows;
    double *o, *lse;
    int route; /* 0 three-pass, 1 online, 2 three-pass under a general mask */
    int64_t tile;
    int mutation;
    int64_t H, window_left, window_right;  /* route 2 */
    const int32_t* doc;                     /* route 2: int32 [B][N] or NULL */
    int64_t next; /* shared work counter */
    pthread_mutex_t lock;
} job_t;

static int64_t take(job_t* jb) {
    pthread_mutex_lock(&jb->lock);
    int64_t r = jb->next++;
    pthread_mutex_unlock(&jb->lock);
    return r;
}

static void* worker(void* arg) {
    job_t* jb = (job_t*)arg;
    double* xbuf = (double*)malloc((size_t)(jb->N > 0 ? jb->N : 1) * sizeof(double));
    for (;;) {
        int64_t r = take(jb);
        if (r >= jb->n_rows) break;
        int64_t flat = jb->rows[r];
        int64_t bh = flat / jb->N, i = flat % jb->N;
        const uint16_t* qrow = jb->q + flat * jb->d;
        const uint16_t* kh = jb->k + bh * jb->N * jb->d;
        const uint16_t* vh = jb->v + bh * jb->N * jb->d;
        int64_t nvis = visible_keys(i, jb->N, jb->causal);
        double* o = jb->o + r * jb->d;
        if (jb->route == 0) {
            row_three_pass(qrow, kh, vh, nvis, jb->d, jb->scale, xbuf, o, jb->lse + r);
        } else if (jb->route == 2) {
            row_three_pass_masked(qrow, kh, vh, bh / jb->H, i, jb->N, jb->d, jb->scale, jb->window_left,
                                  jb->window_right, jb->doc, xbuf, o, jb->lse + r);
        } else {
            double m, l;
            oracle_row_online_state(qrow, kh, vh, jb->d, 0, nvis, nvis, jb->tile, jb->scale, jb->mutation, &m, &l, o);
            if (jb->mutation == ORACLE_MUT_NORMALISE_TILE) {
                /* already "normalised" tile by tile: no final division */
            } else {
                for (int64_t c = 0; c < jb->d; ++c) o[c] /= l;
            }
            jb->lse[r] = m + log(l);
        }
    }
    free(xbuf);
    return NULL;
}

static int run(job_t* jb, int n_threads) {
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > jb->n_rows) n_threads = jb->n_rows > 0 ? (int)jb->n_rows : 1;
    jb->next = 0;
    pthread_mutex_init(&jb->lock, NULL);
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < n_threads; ++t)
        if (pthread_create(&th[t], NULL, worker, jb) == 0) ++started;
    if (started == 0) worker(jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&jb->lock);
    return started > 0 ? started : 1;
}

/* Returns the number of threads used (>= 1), or a negative value on bad input. */
int oracle_attention_three_pass(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B, int64_t H,
                                int64_t N, int64_t d, int causal, double scale, const int64_t* rows, int64_t n_rows,
                                double* o, double* lse, int n_threads) {
    if (!q || !k || !v || !rows || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -2;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.N = N; jb.d = d; jb.causal = causal; jb.scale = scale;
    jb.rows = rows; jb.n_rows = n_rows; jb.o = o; jb.lse = lse; jb.route = 0;
    return run(&jb, n_threads);
}

int oracle_attention_online(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B, int64_t H, int64_t N,
                            int64_t d, int causal, double scale, int64_t tile, int mutation, const int64_t* rows,
                            int64_t n_rows, double* o, double* lse, int n_threads) {
    if (!q || !k || !v || !rows || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -2;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.N = N; jb.d = d; jb.causal = causal; jb.scale = scale;
    jb.rows = rows; jb.n_rows = n_rows; jb.o = o; jb.lse = lse; jb.route = 1;
    jb.tile = tile; jb.mutation = mutation;
    return run(&jb, n_threads);
}

/* Three-pass attention under a window and/or document mask (see key_visible). */
int oracle_attention_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B, int64_t H, int64_t N,
                            int64_t d, double scale, int64_t window_left, int64_t window_right, const int32_t* doc,
                            const int64_t* rows, int64_t n_rows, double* o, double* lse, int n_threads) {
    if (!q || !k || !v || !rows || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -2;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.N = N; jb.d = d; jb.causal = 0; jb.scale = scale;
    jb.rows = rows; jb.n_rows = n_rows; jb.o = o; jb.lse = lse; jb.route = 2;
    jb.H = H; jb.window_left = window_left; jb.window_right = window_right; jb.doc = doc;
    return run(&jb, n_threads);
}

/* ------------------------------------------------------------------------ */
/* Backward pass: gradients of L = sum(O * dO) through O = softmax(S) V,     */
/* S = scale Q K^T, with the scores recomputed from Q and K and normalised   */
/* by the saved per-row statistic LSE (the recomputation of "Online Softmax: */
/* Tiling Across a Reduction", backward-pass section).  For visible pairs:  */
/*   P_ij = exp(S_ij - LSE_i),  D_i = sum_c dO_ic O_ic,                       */
/*   dV_j = sum_i P_ij dO_i,    dS_ij = P_ij (dO_i . v_j - D_i),              */
/*   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i.            */
/* mag_* hold the same sums over absolute values of every term (the         */
/* conditioning of each element, used for error bounds).                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q, *k, *v;
    const double *o, *dout, *lse;
    int64_t N, d;
    int causal;
    double scale;
    const int64_t *q_rows, *k_rows;
    int64_t n_q, n_k;
    double *dq, *dk, *dv, *mdq, *mdk, *mdv;
    int64_t next;
    pthread_mutex_t lock;
} bwd_job_t;

static double row_D(const double* dout_row, const double* o_row, int64_t d) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += dout_row[c] * o_row[c];
    return acc;
}

static double dot_bd(const double* x, const uint16_t* y, int64_t d) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += x[c] * bf16_bits_to_double(y[c]);
    return acc;
}

/* one query row: dQ_i */
static void bwd_query_row(const bwd_job_t* jb, int64_t flat, double* dq, double* mdq) {
    const int64_t N = jb->N, d = jb->d;
    const int64_t bh = flat / N, i = flat % N;
    const uint16_t* qrow = jb->q + flat * d;
    const uint16_t* kh = jb->k + bh * N * d;
    const uint16_t* vh = jb->v + bh * N * d;
    const double* dor = jb->dout + flat * d;
    const double Di = row_D(dor, jb->o + flat * d, d);
    const double Li = jb->lse[flat];
    for (int64_t c = 0; c < d; ++c) dq[c] = mdq[c] = 0.0;
    const int64_t nvis = visible_keys(i, N, jb->causal);
    for (int64_t j = 0; j < nvis; ++j) {
        const double p = exp(score(qrow, kh + j * d, d, jb->scale) - Li);
        const double ds = p * (dot_bd(dor, vh + j * d, d) - Di);
        for (int64_t c = 0; c < d; ++c) {
            const double kc = bf16_bits_to_double(kh[j * d + c]);
            dq[c] += jb->scale * ds * kc;
            mdq[c] += jb->scale * fabs(ds) * fabs(kc);
        }
    }
}

/* one key row: dK_j and dV_j */
static void bwd_key_row(const bwd_job_t* jb, int64_t flat, double* dk, double* dv, double* mdk, double* mdv) {
    const int64_t N = jb->N, d = jb->d;
    const int64_t bh = flat / N, j = flat % N;
    const uint16_t* krow = jb->k + flat * d;
    const uint16_t* vrow = jb->v + flat * d;
    for (int64_t c = 0; c < d; ++c) dk[c] = dv[c] = mdk[c] = mdv[c] = 0.0;
    for (int64_t i = jb->causal ? j : 0; i < N; ++i) {
        const int64_t qf = bh * N + i;
        const uint16_t* qrow = jb->q + qf * d;
        const double* dor = jb->dout + qf * d;
        const double p = exp(score(qrow, krow, d, jb->scale) - jb->lse[qf]);
        const double ds = p * (dot_bd(dor, vrow, d) - row_D(dor, jb->o + qf * d, d));
        for (int64_t c = 0; c < d; ++c) {
            const double qc = bf16_bits_to_double(qrow[c]);
            dv[c] += p * dor[c];
            mdv[c] += p * fabs(dor[c]);
            dk[c] += jb->scale * ds * qc;
            mdk[c] += jb->scale * fabs(ds) * fabs(qc);
        }
    }
}

static void* bwd_worker(void* arg) {
    bwd_job_t* jb = (bwd_job_t*)arg;
    for (;;) {
        pthread_mutex_lock(&jb->lock);
        int64_t r = jb->next++;
        pthread_mutex_unlock(&jb->lock);
        if (r >= jb->n_q + jb->n_k) break;
        if (r < jb->n_q) {
            bwd_query_row(jb, jb->q_rows[r], jb->dq + r * jb->d, jb->mdq + r * jb->d);
        } else {
            const int64_t s = r - jb->n_q;
            bwd_key_row(jb, jb->k_rows[s], jb->dk + s * jb->d, jb->dv + s * jb->d, jb->mdk + s * jb->d,
                        jb->mdv + s * jb->d);
        }
    }
    return NULL;
}

/* Returns the number of threads used, or a negative value on bad input. */
int oracle_attention_backward(const uint16_t* q, const uint16_t* k, const uint16_t* v, const double* o,
                              const double* dout, const double* lse, int64_t B, int64_t H, int64_t N, int64_t d,
                              int causal, double scale, const int64_t* q_rows, int64_t n_q, const int64_t* k_rows,
                              int64_t n_k, double* dq, double* dk, double* dv, double* mag_dq, double* mag_dk,
                              double* mag_dv, int n_threads) {
    if (!q || !k || !v || !o || !dout || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    if ((n_q > 0 && (!q_rows || !dq || !mag_dq)) || (n_k > 0 && (!k_rows || !dk || !dv || !mag_dk || !mag_dv)))
        return -1;
    for (int64_t r = 0; r < n_q; ++r)
        if (q_rows[r] < 0 || q_rows[r] >= B * H * N) return -2;
    for (int64_t r = 0; r < n_k; ++r)
        if (k_rows[r] < 0 || k_rows[r] >= B * H * N) return -2;
    bwd_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.o = o; jb.dout = dout; jb.lse = lse;
    jb.N = N; jb.d = d; jb.causal = causal; jb.scale = scale;
    jb.q_rows = q_rows; jb.k_rows = k_rows; jb.n_q = n_q; jb.n_k = n_k;
    jb.dq = dq; jb.dk = dk; jb.dv = dv; jb.mdq = mag_dq; jb.mdk = mag_dk; jb.mdv = mag_dv;
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    if (n_threads > 256) n_threads = 256;
    const int64_t work = n_q + n_k;
    if ((int64_t)n_threads > work) n_threads = work > 0 ? (int)work : 1;
    pthread_mutex_init(&jb.lock, NULL);
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < n_threads; ++t)
        if (pthread_create(&th[t], NULL, bwd_worker, &jb) == 0) ++started;
    if (started == 0) bwd_worker(&jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&jb.lock);
    return started > 0 ? started : 1;
}
