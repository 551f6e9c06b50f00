/*
 * lizard_oracle.c -- plain, slow, fp64 CPU oracle for the Lizard-attention operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header, table
 * or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (page title, then the section the fact comes from):
 *   [P1] "Lizard: An Efficient Linearization Framework for Large Language Models"
 *        (arXiv 2507.09025, HTML) -- Preliminaries (linear attention, recurrent form),
 *        Method (parallel GLA with the cumulative gate matrix C; hardware-aware
 *        reparameterisation), Experiments setup (window w and m meta tokens).
 *   [P2] papernotes.org note "Lizard: An Efficient Linearization Framework for Large
 *        Language Models" -- section "方法详解 / 关键设计": the GLA recurrence
 *        h_i = gamma_i (.) h_{i-1} + phi(k_i) v_i^T, y_i = phi(q_i)^T h_i, and the Anchor
 *        Window formula softmax([q_i^T T ; q_i^T k_{i-W:i}]) [V_T ; v_{i-W:i}];
 *        section "整体框架": the two branch outputs are summed with a weight.
 *
 * Readings taken where the pages are silent:
 *   - the window holds W keys including the query's own token: j in [max(0,i-W+1), i];
 *   - meta keys/values are per head, shared over the batch, always visible;
 *   - softmax logits are scale * <q, key> (scale passed in, normally 1/sqrt(dk));
 *   - y = y_gla + alpha * y_win; no normaliser, no output gate;
 *   - gamma_i scales the rows (key dimension) of h; h starts at h0 (zero if absent).
 *
 * Every function walks the definition token by token in fp64.  No chunking, no
 * blocking, no reordering beyond the plain loops.  Work is spread over host threads
 * by independent (batch, head) units only; each unit's arithmetic is serial.
 *
 * Layouts: row-major [B,H,L,d] for per-token tensors, [H,M,d] for meta tensors,
 * [B,H,dk,dv] for states.  All arrays are double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_NOMEM 2

/* ------------------------------------------------------------------------- */
/* Thread fan-out over independent units.                                     */
/* ------------------------------------------------------------------------- */
typedef void (*unit_fn)(long unit, void *ctx);

typedef struct {
    unit_fn fn;
    void *ctx;
    long n;
    long next;
} unit_pool;

static void *unit_worker(void *arg) {
    unit_pool *p = (unit_pool *)arg;
    for (;;) {
        long u = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
        if (u >= p->n) break;
        p->fn(u, p->ctx);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Runs fn(u) for u in [0, n); returns the number of threads actually used. */
static int run_units(long n, int nthreads, unit_fn fn, void *ctx) {
    unit_pool p = {fn, ctx, n, 0};
    int t = resolve_threads(nthreads);
    if (t > n) t = (int)n;
    if (t <= 1) {
        unit_worker(&p);
        return 1;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)t);
    int started = 0;
    if (th) {
        for (int i = 0; i < t - 1; ++i) { /* the calling thread is the t-th worker */
            if (pthread_create(&th[started], NULL, unit_worker, &p) == 0) ++started;
        }
    }
    unit_worker(&p); /* the calling thread takes part too */
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return started + 1;
}

static int g_last_threads = 1;
int oracle_last_threads(void) { return g_last_threads; }

/* ------------------------------------------------------------------------- */
/* GLA branch, one head.  [P2 关键设计: GLA recurrence]                         */
/*   for i = 0..L-1:  h[k,:] = exp(log_gamma_i[k]) * h[k,:] + phi_k_i[k] * v_i   */
/*                    y_i[:] = sum_k phi_q_i[k] * h[k,:]                         */
/* hs (nullable) receives every state: hs[0] = h0, hs[i+1] = state after i.   */
/* ------------------------------------------------------------------------- */
static void gla_fwd_head(int L, int dk, int dv, const double *pq, const double *pk,
                         const double *v, const double *lg, const double *h0, double *y,
                         double *h_final, double *h, double *hs) {
    const size_t hsz = (size_t)dk * dv;
    if (h0) memcpy(h, h0, hsz * sizeof(double));
    else memset(h, 0, hsz * sizeof(double));
    if (hs) memcpy(hs, h, hsz * sizeof(double));
    for (int i = 0; i < L; ++i) {
        const double *pk_i = pk + (size_t)i * dk;
        const double *pq_i = pq + (size_t)i * dk;
        const double *lg_i = lg + (size_t)i * dk;
        const double *v_i = v + (size_t)i * dv;
        for (int k = 0; k < dk; ++k) {
            const double g = exp(lg_i[k]);
            const double a = pk_i[k];
            double *row = h + (size_t)k * dv;
            for (int c = 0; c < dv; ++c) row[c] = g * row[c] + a * v_i[c];
        }
        double *y_i = y + (size_t)i * dv;
        for (int c = 0; c < dv; ++c) y_i[c] = 0.0;
        for (int k = 0; k < dk; ++k) {
            const double a = pq_i[k];
            const double *row = h + (size_t)k * dv;
            for (int c = 0; c < dv; ++c) y_i[c] += a * row[c];
        }
        if (hs) memcpy(hs + (size_t)(i + 1) * hsz, h, hsz * sizeof(double));
    }
    if (h_final) memcpy(h_final, h, hsz * sizeof(double));
}

/* ------------------------------------------------------------------------- */
/* Anchor-window branch, one head.  [P2 关键设计: Anchor Window Attention]      */
/* Key set of query i: the M meta keys, then tokens j in [max(0,i-W+1), i].    */
/* Logits scale*<q_i,key>, max-subtracted softmax, y_i = sum p * value.        */
/* ------------------------------------------------------------------------- */
static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* Fills z (logits) and returns the number of keys; keys are ordered meta first. */
static int window_logits(int i, int d, int M, int W, double scale, const double *q,
                         const double *k, const double *mk, double *z) {
    const double *q_i = q + (size_t)i * d;
    int n = 0;
    for (int m = 0; m < M; ++m) z[n++] = scale * dot(q_i, mk + (size_t)m * d, d);
    int j0 = i - W + 1;
    if (j0 < 0) j0 = 0;
    for (int j = j0; j <= i; ++j) z[n++] = scale * dot(q_i, k + (size_t)j * d, d);
    return n;
}

/* Turns logits into probabilities in place. */
static void softmax_inplace(double *z, int n) {
    double zmax = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (z[j] > zmax) zmax = z[j];
    double sum = 0.0;
    for (int j = 0; j < n; ++j) {
        z[j] = exp(z[j] - zmax);
        sum += z[j];
    }
    for (int j = 0; j < n; ++j) z[j] /= sum;
}

static void window_fwd_head(int L, int d, int dv, int M, int W, double scale,
                            const double *q, const double *k, const double *v,
                            const double *mk, const double *mv, double *y, double *z) {
    for (int i = 0; i < L; ++i) {
        const int n = window_logits(i, d, M, W, scale, q, k, mk, z);
        softmax_inplace(z, n);
        double *y_i = y + (size_t)i * dv;
        for (int c = 0; c < dv; ++c) y_i[c] = 0.0;
        int j0 = i - W + 1;
        if (j0 < 0) j0 = 0;
        for (int m = 0; m < M; ++m)
            for (int c = 0; c < dv; ++c) y_i[c] += z[m] * mv[(size_t)m * dv + c];
        for (int j = j0; j <= i; ++j) {
            const double p = z[M + (j - j0)];
            for (int c = 0; c < dv; ++c) y_i[c] += p * v[(size_t)j * dv + c];
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Forward over all (b, h): y = y_gla + alpha * y_win.                         */
/* ------------------------------------------------------------------------- */
typedef struct {
    int B, H, L, dk, dv, M, W;
    double alpha, scale;
    const double *pq, *pk, *v, *lg, *q, *k, *mk, *mv, *h0;
    double *y, *y_gla, *y_win, *h_final;
    int failed;
} fwd_ctx;

static void fwd_unit(long u, void *vctx) {
    fwd_ctx *c = (fwd_ctx *)vctx;
    const int hh = (int)(u % c->H);
    const size_t tok_k = (size_t)u * c->L * c->dk;
    const size_t tok_v = (size_t)u * c->L * c->dv;
    const size_t hsz = (size_t)c->dk * c->dv;
    double *h = (double *)malloc(hsz * sizeof(double));
    double *yg = (double *)malloc((size_t)c->L * c->dv * sizeof(double));
    double *yw = (double *)malloc((size_t)c->L * c->dv * sizeof(double));
    double *z = (double *)malloc((size_t)(c->M + c->W + 1) * sizeof(double));
    if (!h || !yg || !yw || !z) {
        __atomic_store_n(&c->failed, 1, __ATOMIC_RELAXED);
        free(h); free(yg); free(yw); free(z);
        return;
    }
    gla_fwd_head(c->L, c->dk, c->dv, c->pq + tok_k, c->pk + tok_k, c->v + tok_v, c->lg + tok_k,
                 c->h0 ? c->h0 + (size_t)u * hsz : NULL, yg,
                 c->h_final ? c->h_final + (size_t)u * hsz : NULL, h, NULL);
    window_fwd_head(c->L, c->dk, c->dv, c->M, c->W, c->scale, c->q + tok_k, c->k + tok_k,
                    c->v + tok_v, c->mk + (size_t)hh * c->M * c->dk,
                    c->mv + (size_t)hh * c->M * c->dv, yw, z);
    for (size_t e = 0; e < (size_t)c->L * c->dv; ++e) {
        c->y[tok_v + e] = yg[e] + c->alpha * yw[e];
        if (c->y_gla) c->y_gla[tok_v + e] = yg[e];
        if (c->y_win) c->y_win[tok_v + e] = yw[e];
    }
    free(h); free(yg); free(yw); free(z);
}

static int dims_ok(int B, int H, int L, int dk, int dv, int M, int W) {
    return B >= 1 && H >= 1 && L >= 0 && dk >= 1 && dv >= 1 && M >= 0 && W >= 1;
}

/* Forward.  y_gla, y_win, h0 and h_final are nullable. */
int oracle_fwd(int B, int H, int L, int dk, int dv, int M, int W, double alpha, double scale,
               const double *phi_q, const double *phi_k, const double *v,
               const double *log_gamma, const double *q, const double *k,
               const double *meta_k, const double *meta_v, const double *h0, double *y,
               double *y_gla, double *y_win, double *h_final, int nthreads) {
    if (!dims_ok(B, H, L, dk, dv, M, W)) return OR_ERR_ARG;
    if (!phi_q || !phi_k || !v || !log_gamma || !q || !k || !y) return OR_ERR_ARG;
    if (M > 0 && (!meta_k || !meta_v)) return OR_ERR_ARG;
    fwd_ctx c = {B, H, L, dk, dv, M, W, alpha, scale, phi_q, phi_k, v, log_gamma, q, k,
                 meta_k, meta_v, h0, y, y_gla, y_win, h_final, 0};
    g_last_threads = run_units((long)B * H, nthreads, fwd_unit, &c);
    return c.failed ? OR_ERR_NOMEM : OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Backward: hand-written reverse-mode adjoint of the two loops above.         */
/* ------------------------------------------------------------------------- */
/*
 * GLA adjoint, one head.  With hs[i+1] the state after token i (hs[0] = h0) and
 * dh the adjoint of the state after the token being visited, for i = L-1..0:
 *   dh        += phi_q_i dy_i^T                 (from y_i = phi_q_i^T h_i)
 *   dphi_q_i   = h_i dy_i
 *   dphi_k_i   = dh v_i                         (from h_i += phi_k_i v_i^T)
 *   dv_i      += dh^T phi_k_i
 *   dlogg_i[k] = exp(lg_i[k]) * sum_c dh[k,c] h_{i-1}[k,c]
 *   dh[k,:]   *= exp(lg_i[k])                   (through h_i = gamma_i (.) h_{i-1})
 * After the loop dh is the adjoint of h0.
 */
static void gla_bwd_head(int L, int dk, int dv, const double *pq, const double *pk,
                         const double *v, const double *lg, const double *hs,
                         const double *dy, double *dpq, double *dpk, double *dvv,
                         double *dlg, double *dh, double *dh0) {
    const size_t hsz = (size_t)dk * dv;
    memset(dh, 0, hsz * sizeof(double));
    for (int i = L - 1; i >= 0; --i) {
        const double *pq_i = pq + (size_t)i * dk;
        const double *pk_i = pk + (size_t)i * dk;
        const double *lg_i = lg + (size_t)i * dk;
        const double *v_i = v + (size_t)i * dv;
        const double *dy_i = dy + (size_t)i * dv;
        const double *h_i = hs + (size_t)(i + 1) * hsz;
        const double *h_prev = hs + (size_t)i * hsz;
        for (int kk = 0; kk < dk; ++kk) {
            double *row = dh + (size_t)kk * dv;
            for (int c = 0; c < dv; ++c) row[c] += pq_i[kk] * dy_i[c];
        }
        for (int kk = 0; kk < dk; ++kk)
            dpq[(size_t)i * dk + kk] = dot(h_i + (size_t)kk * dv, dy_i, dv);
        for (int kk = 0; kk < dk; ++kk)
            dpk[(size_t)i * dk + kk] = dot(dh + (size_t)kk * dv, v_i, dv);
        for (int c = 0; c < dv; ++c) {
            double s = 0.0;
            for (int kk = 0; kk < dk; ++kk) s += dh[(size_t)kk * dv + c] * pk_i[kk];
            dvv[(size_t)i * dv + c] += s;
        }
        for (int kk = 0; kk < dk; ++kk) {
            const double g = exp(lg_i[kk]);
            dlg[(size_t)i * dk + kk] = g * dot(dh + (size_t)kk * dv, h_prev + (size_t)kk * dv, dv);
            double *row = dh + (size_t)kk * dv;
            for (int c = 0; c < dv; ++c) row[c] *= g;
        }
    }
    if (dh0) memcpy(dh0, dh, hsz * sizeof(double));
}

/*
 * Window adjoint, one head, textbook softmax backward.  dyw_i = alpha * dy_i;
 * dp_j = <dyw_i, value_j>; D = sum_j p_j dp_j; ds_j = p_j (dp_j - D);
 * dq_i += scale sum_j ds_j key_j; dkey_j += scale ds_j q_i; dvalue_j += p_j dyw_i.
 * Meta-key/value adjoints accumulate into dmk, dmv (this head's, this batch's).
 */
static void window_bwd_head(int L, int d, int dv, int M, int W, double scale, double alpha,
                            const double *q, const double *k, const double *v,
                            const double *mk, const double *mv, const double *dy,
                            double *dq, double *dkk, double *dvv, double *dmk,
                            double *dmv, double *z, double *dp, double *dyw) {
    for (int i = 0; i < L; ++i) {
        const int n = window_logits(i, d, M, W, scale, q, k, mk, z);
        softmax_inplace(z, n);
        int j0 = i - W + 1;
        if (j0 < 0) j0 = 0;
        for (int c = 0; c < dv; ++c) dyw[c] = alpha * dy[(size_t)i * dv + c];
        double D = 0.0;
        for (int m = 0; m < M; ++m) {
            dp[m] = dot(dyw, mv + (size_t)m * dv, dv);
            D += z[m] * dp[m];
        }
        for (int j = j0; j <= i; ++j) {
            const int s = M + (j - j0);
            dp[s] = dot(dyw, v + (size_t)j * dv, dv);
            D += z[s] * dp[s];
        }
        const double *q_i = q + (size_t)i * d;
        double *dq_i = dq + (size_t)i * d;
        for (int m = 0; m < M; ++m) {
            const double ds = z[m] * (dp[m] - D);
            for (int e = 0; e < d; ++e) {
                dq_i[e] += scale * ds * mk[(size_t)m * d + e];
                dmk[(size_t)m * d + e] += scale * ds * q_i[e];
            }
            for (int c = 0; c < dv; ++c) dmv[(size_t)m * dv + c] += z[m] * dyw[c];
        }
        for (int j = j0; j <= i; ++j) {
            const int s = M + (j - j0);
            const double ds = z[s] * (dp[s] - D);
            for (int e = 0; e < d; ++e) {
                dq_i[e] += scale * ds * k[(size_t)j * d + e];
                dkk[(size_t)j * d + e] += scale * ds * q_i[e];
            }
            for (int c = 0; c < dv; ++c) dvv[(size_t)j * dv + c] += z[s] * dyw[c];
        }
    }
}

typedef struct {
    int B, H, L, dk, dv, M, W;
    double alpha, scale;
    const double *pq, *pk, *v, *lg, *q, *k, *mk, *mv, *h0, *dy;
    double *dpq, *dpk, *dvv, *dlg, *dq, *dk_, *dmk_part, *dmv_part, *dh0;
    int failed;
} bwd_ctx;

static void bwd_unit(long u, void *vctx) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const int hh = (int)(u % c->H);
    const size_t tok_k = (size_t)u * c->L * c->dk;
    const size_t tok_v = (size_t)u * c->L * c->dv;
    const size_t hsz = (size_t)c->dk * c->dv;
    double *hs = (double *)malloc((size_t)(c->L + 1) * hsz * sizeof(double));
    double *h = (double *)malloc(hsz * sizeof(double));
    double *dh = (double *)malloc(hsz * sizeof(double));
    double *yg = (double *)malloc(((size_t)c->L * c->dv + 1) * sizeof(double));
    double *z = (double *)malloc((size_t)(c->M + c->W + 1) * sizeof(double));
    double *dp = (double *)malloc((size_t)(c->M + c->W + 1) * sizeof(double));
    double *dyw = (double *)malloc((size_t)c->dv * sizeof(double));
    if (!hs || !h || !dh || !yg || !z || !dp || !dyw) {
        __atomic_store_n(&c->failed, 1, __ATOMIC_RELAXED);
        free(hs); free(h); free(dh); free(yg); free(z); free(dp); free(dyw);
        return;
    }
    /* Forward states, then the two adjoints. */
    gla_fwd_head(c->L, c->dk, c->dv, c->pq + tok_k, c->pk + tok_k, c->v + tok_v, c->lg + tok_k,
                 c->h0 ? c->h0 + (size_t)u * hsz : NULL, yg, NULL, h, hs);
    memset(c->dvv + tok_v, 0, (size_t)c->L * c->dv * sizeof(double));
    memset(c->dq + tok_k, 0, (size_t)c->L * c->dk * sizeof(double));
    memset(c->dk_ + tok_k, 0, (size_t)c->L * c->dk * sizeof(double));
    gla_bwd_head(c->L, c->dk, c->dv, c->pq + tok_k, c->pk + tok_k, c->v + tok_v, c->lg + tok_k,
                 hs, c->dy + tok_v, c->dpq + tok_k, c->dpk + tok_k, c->dvv + tok_v,
                 c->dlg + tok_k, dh, c->dh0 ? c->dh0 + (size_t)u * hsz : NULL);
    double *dmk = c->dmk_part + (size_t)u * c->M * c->dk;
    double *dmv = c->dmv_part + (size_t)u * c->M * c->dv;
    memset(dmk, 0, (size_t)c->M * c->dk * sizeof(double));
    memset(dmv, 0, (size_t)c->M * c->dv * sizeof(double));
    window_bwd_head(c->L, c->dk, c->dv, c->M, c->W, c->scale, c->alpha, c->q + tok_k,
                    c->k + tok_k, c->v + tok_v, c->mk + (size_t)hh * c->M * c->dk,
                    c->mv + (size_t)hh * c->M * c->dv, c->dy + tok_v, c->dq + tok_k,
                    c->dk_ + tok_k, c->dvv + tok_v, dmk, dmv, z, dp, dyw);
    free(hs); free(h); free(dh); free(yg); free(z); free(dp); free(dyw);
}

/*
 * Backward.  Outputs: d_phi_q, d_phi_k, d_log_gamma, d_q, d_k [B,H,L,dk];
 * d_v [B,H,L,dv] (GLA + window); d_meta_k [H,M,dk], d_meta_v [H,M,dv] (summed over
 * batch and tokens, batch order 0..B-1); d_h0 [B,H,dk,dv] nullable.
 * Memory: one head keeps all L+1 states, (L+1)*dk*dv doubles per running thread.
 */
int oracle_bwd(int B, int H, int L, int dk, int dv, int M, int W, double alpha, double scale,
               const double *phi_q, const double *phi_k, const double *v,
               const double *log_gamma, const double *q, const double *k,
               const double *meta_k, const double *meta_v, const double *h0,
               const double *dy, double *d_phi_q, double *d_phi_k, double *d_v,
               double *d_log_gamma, double *d_q, double *d_k, double *d_meta_k,
               double *d_meta_v, double *d_h0, int nthreads) {
    if (!dims_ok(B, H, L, dk, dv, M, W)) return OR_ERR_ARG;
    if (!phi_q || !phi_k || !v || !log_gamma || !q || !k || !dy) return OR_ERR_ARG;
    if (!d_phi_q || !d_phi_k || !d_v || !d_log_gamma || !d_q || !d_k) return OR_ERR_ARG;
    if (M > 0 && (!meta_k || !meta_v || !d_meta_k || !d_meta_v)) return OR_ERR_ARG;
    const long units = (long)B * H;
    double *dmk_part = (double *)malloc(((size_t)units * M * dk + 1) * sizeof(double));
    double *dmv_part = (double *)malloc(((size_t)units * M * dv + 1) * sizeof(double));
    if (!dmk_part || !dmv_part) {
        free(dmk_part); free(dmv_part);
        return OR_ERR_NOMEM;
    }
    bwd_ctx c = {B, H, L, dk, dv, M, W, alpha, scale, phi_q, phi_k, v, log_gamma, q, k,
                 meta_k, meta_v, h0, dy, d_phi_q, d_phi_k, d_v, d_log_gamma, d_q, d_k,
                 dmk_part, dmv_part, d_h0, 0};
    g_last_threads = run_units(units, nthreads, bwd_unit, &c);
    if (M > 0) {
        memset(d_meta_k, 0, (size_t)H * M * dk * sizeof(double));
        memset(d_meta_v, 0, (size_t)H * M * dv * sizeof(double));
        for (int b = 0; b < B; ++b)
            for (int hh = 0; hh < H; ++hh) {
                const long u = (long)b * H + hh;
                for (size_t e = 0; e < (size_t)M * dk; ++e)
                    d_meta_k[(size_t)hh * M * dk + e] += dmk_part[(size_t)u * M * dk + e];
                for (size_t e = 0; e < (size_t)M * dv; ++e)
                    d_meta_v[(size_t)hh * M * dv + e] += dmv_part[(size_t)u * M * dv + e];
            }
    }
    free(dmk_part);
    free(dmv_part);
    return c.failed ? OR_ERR_NOMEM : OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Decode: one token per sequence, in place on (h, rings, pos).                */
/* [P1 Preliminaries: recurrent form]; [P2 关键设计: both branches]            */
/* Ring slot of absolute position t is t mod W; the window of position p holds  */
/* the tokens t in [max(0, p-W+1), p].                                          */
/* ------------------------------------------------------------------------- */
typedef struct {
    int N, H, dk, dv, M, W;
    double alpha, scale;
    const double *pq, *pk, *v, *lg, *q, *k, *mk, *mv;
    double *h, *kr, *vr, *y;
    const int64_t *pos;
    int failed;
} dec_ctx;

static void dec_unit(long u, void *vctx) {
    dec_ctx *c = (dec_ctx *)vctx;
    const int n = (int)(u / c->H);
    const int hh = (int)(u % c->H);
    const int64_t p = c->pos[n];
    const int dk = c->dk, dv = c->dv, W = c->W, M = c->M;
    const double *pq = c->pq + (size_t)u * dk, *pk = c->pk + (size_t)u * dk;
    const double *lg = c->lg + (size_t)u * dk, *q = c->q + (size_t)u * dk;
    const double *kn = c->k + (size_t)u * dk, *vn = c->v + (size_t)u * dv;
    double *h = c->h + (size_t)u * dk * dv;
    double *kr = c->kr + (size_t)u * W * dk, *vr = c->vr + (size_t)u * W * dv;
    double *y = c->y + (size_t)u * dv;
    double *z = (double *)malloc((size_t)(M + W + 1) * sizeof(double));
    if (!z) {
        __atomic_store_n(&c->failed, 1, __ATOMIC_RELAXED);
        return;
    }
    /* GLA: h = gamma (.) h + phi_k v^T ; y_gla = phi_q^T h */
    for (int kk = 0; kk < dk; ++kk) {
        const double g = exp(lg[kk]);
        for (int e = 0; e < dv; ++e)
            h[(size_t)kk * dv + e] = g * h[(size_t)kk * dv + e] + pk[kk] * vn[e];
    }
    for (int e = 0; e < dv; ++e) {
        double s = 0.0;
        for (int kk = 0; kk < dk; ++kk) s += pq[kk] * h[(size_t)kk * dv + e];
        y[e] = s;
    }
    /* Window: write the new token, then attend over meta + the last W tokens. */
    const int slot = (int)(p % W);
    memcpy(kr + (size_t)slot * dk, kn, (size_t)dk * sizeof(double));
    memcpy(vr + (size_t)slot * dv, vn, (size_t)dv * sizeof(double));
    int64_t t0 = p - W + 1;
    if (t0 < 0) t0 = 0;
    int cnt = 0;
    for (int m = 0; m < M; ++m) z[cnt++] = c->scale * dot(q, c->mk + ((size_t)hh * M + m) * dk, dk);
    for (int64_t t = t0; t <= p; ++t)
        z[cnt++] = c->scale * dot(q, kr + (size_t)(t % W) * dk, dk);
    softmax_inplace(z, cnt);
    for (int e = 0; e < dv; ++e) {
        double s = 0.0;
        for (int m = 0; m < M; ++m) s += z[m] * c->mv[((size_t)hh * M + m) * dv + e];
        int idx = M;
        for (int64_t t = t0; t <= p; ++t) s += z[idx++] * vr[(size_t)(t % W) * dv + e];
        y[e] += c->alpha * s;
    }
    free(z);
}

int oracle_decode_step(int N, int H, int dk, int dv, int M, int W, double alpha, double scale,
                       const double *phi_q, const double *phi_k, const double *v,
                       const double *log_gamma, const double *q, const double *k,
                       const double *meta_k, const double *meta_v, double *h,
                       double *k_ring, double *v_ring, int64_t *pos, double *y, int nthreads) {
    if (N < 1 || H < 1 || dk < 1 || dv < 1 || M < 0 || W < 1) return OR_ERR_ARG;
    if (!phi_q || !phi_k || !v || !log_gamma || !q || !k || !h || !k_ring || !v_ring ||
        !pos || !y)
        return OR_ERR_ARG;
    if (M > 0 && (!meta_k || !meta_v)) return OR_ERR_ARG;
    for (int n = 0; n < N; ++n)
        if (pos[n] < 0) return OR_ERR_ARG;
    dec_ctx c = {N, H, dk, dv, M, W, alpha, scale, phi_q, phi_k, v, log_gamma, q, k,
                 meta_k, meta_v, h, k_ring, v_ring, y, pos, 0};
    g_last_threads = run_units((long)N * H, nthreads, dec_unit, &c);
    for (int n = 0; n < N; ++n) pos[n] += 1;
    return c.failed ? OR_ERR_NOMEM : OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Chunk-local inclusive cumulative sum of log gamma.                          */
/* [P1 Method: cumulative gate products, taken in log space]                   */
/* b_t = sum_{s = chunk start .. t} lg_s;  Gamma_c = b at the chunk's last token */
/* ------------------------------------------------------------------------- */
int oracle_chunk_cumsum(int units, int L, int dk, int chunk, const double *log_gamma,
                        double *b, double *gamma_chunk) {
    if (units < 1 || L < 0 || dk < 1 || chunk < 1 || !log_gamma || !b) return OR_ERR_ARG;
    const int nchunks = (L + chunk - 1) / chunk;
    for (int u = 0; u < units; ++u) {
        const double *lg = log_gamma + (size_t)u * L * dk;
        double *bu = b + (size_t)u * L * dk;
        for (int kk = 0; kk < dk; ++kk) {
            double run = 0.0;
            for (int t = 0; t < L; ++t) {
                if (t % chunk == 0) run = 0.0;
                run += lg[(size_t)t * dk + kk];
                bu[(size_t)t * dk + kk] = run;
                const int last = (t % chunk == chunk - 1) || (t == L - 1);
                if (last && gamma_chunk)
                    gamma_chunk[((size_t)u * nchunks + t / chunk) * dk + kk] = run;
            }
        }
    }
    return OR_OK;
}
