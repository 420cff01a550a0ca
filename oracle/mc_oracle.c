/*
 * mc_oracle.c -- plain fp64 CPU oracle for the Memory Caching (MC) forward pass
 * over a linear matrix-valued memory, and for its gradient (the backward pass).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path.  It is deliberately slow and literal: one token at a time, in the
 * order the method is written, in double precision.
 *
 * Pages cited (the text of the method):
 *   [MC-zh]  "記憶體快取：具備成長型記憶力的循環神經網路" (Memory Caching: RNNs
 *            with growing memory, zh-Hant translation, news.neo-ai.one/article/2518)
 *   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (ja translation of the
 *            same paper, news.neo-ai.one/ja/article/2519)
 *   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
 *            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
 *
 * What is computed, per (batch, head), tokens t = 0..L-1 (0-based here):
 *   segments of constant length C; segment n = [nC, min(nC+C, L))       [MC-ja §3, eq. 4b]
 *   update rule f(M; k, v) = M + v k^T, memory restarts at each segment  [MC-ja §3, eq. 4b]
 *   cached state of segment n: M^(n) = sum_{t in n} v_t k_t^T            [MC-ja §3, after eq. 4b]
 *   online state at t (segment s, start t0): M_t^(s) = sum_{j=t0..t} v_j k_j^T
 *       (the read comes after the update, so token t is included)        [MC-ja §3, eq. 4b-5]
 *   pooled segment summary: mean of the segment's keys                  [MC-ja §3.1, eq. 10]
 *       (the current segment is pooled over the keys seen so far, t0..t)
 *   scores r_{t,i} = <u_t, pool_i>, i = 0..s                             [MC-ja §3.1, eq. 10]
 *   Residual: y_t = M_t^(s) q_t + sum_{i<s} M^(i) q_t                    [MC-ja §3.1, eq. 7]
 *   GRM:      gamma_t = softmax_i(r_{t,0..s}),
 *             y_t = gamma_{t,s} M_t^(s) q_t + sum_{i<s} gamma_{t,i} M^(i) q_t
 *                                                                        [MC-ja §3.1, eq. 9-10]
 *   Soup:     M*_t = gamma_{t,s} M_t^(s) + sum_{i<s} gamma_{t,i} M^(i),  y_t = M*_t q_t
 *                                                                        [MC-sum §3.3]
 *   SSC:      R_t = the topk largest r_{t,i}, i<s (all of them when s <= topk),
 *             gamma_t = softmax over {r_{t,i} : i in R_t} and r_{t,s},
 *             y_t = gamma_{t,s} M_t^(s) q_t + sum_{i in R_t} gamma_{t,i} M^(i) q_t
 *                                                                        [MC-sum §3.4]
 *   Mean:     memory caching added to a model after training: the memories
 *             are averaged with no learned weights,
 *             y_t = (M_t^(s) q_t + sum_{i<s} M^(i) q_t) / (s + 1)
 *                          [MC-ja, variants appendix after eq. 35, post-training MC]
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - phi = identity and no 1/Z normaliser (unnormalised linear attention, [MC-ja §2]);
 *   - the pooled summary pools keys (the gate needs a vector in the key space);
 *   - softmax has no temperature; the last segment may be shorter than C;
 *   - SSC ranks on the scores rounded to fp32 (the precision the router is
 *     specified in), equal fp32 scores going to the lower segment index;
 *   - Mean averages the online memory together with the cached ones, each with
 *     weight 1 / (s + 1).
 *
 * Sliding-window linear attention with c = 2 under memory caching (SWLA, the
 * second memory family the pages cache) replaces the update rule by
 *   M_t^(s) = alpha_t M_{t-1}^(s) + beta_t v_{t-1} k_{t-1}^T + lambda_t v_t k_t^T
 *                                                                        [MC-ja §3.1, SWLA eq. 28]
 * with per-token scalars alpha, beta, lambda; the read and the aggregation are
 * unchanged ([MC-ja §3.1, eq. 29]; GRM and Soup coincide for this linear memory).
 * Reading: the memory restarts at each segment, so at a segment's first token the
 * beta term (which would reach back into the previous segment) is absent.
 *
 * All arrays are dense, row-major, [BH][L][d] for q,k,v,u,y and [BH][N][d][d]
 * for the states, state[a][b] = sum v[a] k[b] (row = value dim, column = key dim);
 * alpha, beta, lambda are [BH][L].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_RESIDUAL = 0, OR_GRM = 1, OR_SOUP = 2, OR_SSC = 3, OR_MEAN = 4 };

enum {
    OR_OK = 0,
    OR_ERR_ARG = -1,
    OR_ERR_NOMEM = -2,
};

typedef struct {
    const double *q, *k, *v, *u;
    int L, d, C, mode, topk;
    const uint8_t *seg_mask; /* optional: compute y only for segments with mask != 0 */
    const int32_t *given_sel; /* optional: SSC selections to use instead of ranking */
    double *y;
    double *states;
    int32_t *sel; /* optional [L][topk], rank order, -1 padded */
    double *gap;  /* optional [L] */
    const double *alpha, *beta, *lam; /* SWLA scalars [L]; all NULL = plain linear memory */
    const double *dy;                 /* backward: upstream gradient of y [L][d] */
    double *dq, *dk, *dv, *du;        /* backward: gradients [L][d], written */
    const int32_t *seg_off;           /* optional: segment n = [seg_off[n], seg_off[n+1]), nseg of them */
    int nseg;
} head_job;

/* Segments: constant length C (the last one may be shorter), or the given boundaries. */
static int num_seg(const head_job *J) { return J->seg_off ? J->nseg : (J->L + J->C - 1) / J->C; }
static int seg_lo(const head_job *J, int n) { return J->seg_off ? J->seg_off[n] : n * J->C; }
static int seg_hi(const head_job *J, int n)
{
    if (J->seg_off) return J->seg_off[n + 1];
    return (n + 1) * J->C < J->L ? (n + 1) * J->C : J->L;
}
static int seg_of(const head_job *J, int t)
{
    if (!J->seg_off) return t / J->C;
    int n = 0;
    while (J->seg_off[n + 1] <= t) ++n;
    return n;
}

/*
 * One step of the segment memory at token t (segment start t0):
 *   plain: M += v_t k_t^T                                       [MC-ja §3, eq. 4b]
 *   SWLA:  M = alpha_t M + beta_t v_{t-1} k_{t-1}^T + lambda_t v_t k_t^T, no beta
 *          term at t = t0                                       [MC-ja §3.1, eq. 28]
 */
static void memory_step(const head_job *J, double *M, int t, int t0)
{
    const int d = J->d;
    const double *kt = J->k + (size_t)t * d, *vt = J->v + (size_t)t * d;
    if (!J->alpha) {
        for (int a = 0; a < d; ++a)
            for (int b = 0; b < d; ++b) M[(size_t)a * d + b] += vt[a] * kt[b];
        return;
    }
    const double al = J->alpha[t], be = t > t0 ? J->beta[t] : 0.0, la = J->lam[t];
    const double *kp = t > t0 ? J->k + (size_t)(t - 1) * d : kt, *vp = t > t0 ? J->v + (size_t)(t - 1) * d : vt;
    for (int a = 0; a < d; ++a)
        for (int b = 0; b < d; ++b)
            M[(size_t)a * d + b] = al * M[(size_t)a * d + b] + be * vp[a] * kp[b] + la * vt[a] * kt[b];
}

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += a[i] * b[i];
    return s;
}

/* out += w * (M x), M is d x d row-major. */
static void add_matvec(double *out, double w, const double *M, const double *x, int d)
{
    for (int a = 0; a < d; ++a) out[a] += w * dot(M + (size_t)a * d, x, d);
}

/* softmax over n entries in place, max subtracted first */
static void softmax(double *r, int n)
{
    double m = r[0];
    for (int i = 1; i < n; ++i)
        if (r[i] > m) m = r[i];
    double z = 0.0;
    for (int i = 0; i < n; ++i) {
        r[i] = exp(r[i] - m);
        z += r[i];
    }
    for (int i = 0; i < n; ++i) r[i] /= z;
}

/*
 * SSC router for one token: pick the topk largest of r[0..ncached-1] ranked in
 * fp32, equal fp32 values going to the lower index.  Writes the chosen indices in
 * rank order into idx (count returned) and the fp64 distance between the last
 * chosen and the best unchosen score into *gap (INFINITY if nothing is left out).
 */
static int ssc_rank(const double *r, int ncached, int topk, int *idx, uint8_t *taken, double *gap)
{
    int want = ncached < topk ? ncached : topk;
    memset(taken, 0, (size_t)(ncached > 0 ? ncached : 1));
    for (int c = 0; c < want; ++c) {
        int best = -1;
        float bv = 0.f;
        for (int i = 0; i < ncached; ++i) {
            if (taken[i]) continue;
            float fi = (float)r[i];
            if (best < 0 || fi > bv) { /* strict: ties keep the lower index */
                best = i;
                bv = fi;
            }
        }
        taken[best] = 1;
        idx[c] = best;
    }
    *gap = INFINITY;
    if (want > 0 && want < ncached) {
        int best = -1;
        float bv = 0.f;
        for (int i = 0; i < ncached; ++i) {
            if (taken[i]) continue;
            float fi = (float)r[i];
            if (best < 0 || fi > bv) {
                best = i;
                bv = fi;
            }
        }
        *gap = fabs(r[idx[want - 1]] - r[best]);
    }
    return want;
}

/* State form, literal: eq. 4b per token, eq. 7/9/10 or the Soup / SSC formulas per token. */
static int head_forward(const head_job *J)
{
    const int d = J->d;
    const int N = num_seg(J);
    const size_t dd = (size_t)d * d;

    double *kbar = calloc((size_t)N * d, sizeof(double));
    double *Mon = malloc(dd * sizeof(double));
    double *Mstar = malloc(dd * sizeof(double));
    double *ksum = malloc((size_t)d * sizeof(double));
    double *r = malloc((size_t)(N + 1) * sizeof(double));
    double *g = malloc((size_t)(N + 1) * sizeof(double));
    int *idx = malloc((size_t)(N + 1) * sizeof(int));
    uint8_t *taken = malloc((size_t)(N + 1));
    if (!kbar || !Mon || !Mstar || !ksum || !r || !g || !idx || !taken) {
        free(kbar); free(Mon); free(Mstar); free(ksum); free(r); free(g); free(idx); free(taken);
        return OR_ERR_NOMEM;
    }

    /* Step 1: compress every segment with f(M;k,v) = M + v k^T from a zero memory and
     * cache its last state; pool the segment's keys. */
    memset(J->states, 0, (size_t)N * dd * sizeof(double));
    for (int n = 0; n < N; ++n) {
        double *M = J->states + (size_t)n * dd;
        int t0 = seg_lo(J, n), t1 = seg_hi(J, n);
        for (int t = t0; t < t1; ++t) {
            const double *kt = J->k + (size_t)t * d;
            memory_step(J, M, t, t0);
            for (int b = 0; b < d; ++b) kbar[(size_t)n * d + b] += kt[b];
        }
        for (int b = 0; b < d; ++b) kbar[(size_t)n * d + b] /= (double)(t1 - t0);
    }

    /* Step 2: per token, the online memory after its update, the scores, the aggregation. */
    for (int s = 0; s < N; ++s) {
        int t0 = seg_lo(J, s), t1 = seg_hi(J, s);
        int want_y = J->seg_mask == NULL || J->seg_mask[s] != 0;
        memset(Mon, 0, dd * sizeof(double));
        memset(ksum, 0, (size_t)d * sizeof(double));
        for (int t = t0; t < t1; ++t) {
            const double *qt = J->q + (size_t)t * d, *kt = J->k + (size_t)t * d;
            const double *ut = J->u + (size_t)t * d;
            memory_step(J, Mon, t, t0);
            for (int b = 0; b < d; ++b) ksum[b] += kt[b];
            if (!want_y) continue;

            double *yt = J->y + (size_t)t * d;
            memset(yt, 0, (size_t)d * sizeof(double));
            double cnt = (double)(t - t0 + 1);

            if (J->mode == OR_RESIDUAL) {
                add_matvec(yt, 1.0, Mon, qt, d);
                for (int i = 0; i < s; ++i) add_matvec(yt, 1.0, J->states + (size_t)i * dd, qt, d);
                continue;
            }
            if (J->mode == OR_MEAN) { /* the average of the s + 1 memories, read at q_t */
                const double w = 1.0 / (double)(s + 1);
                add_matvec(yt, w, Mon, qt, d);
                for (int i = 0; i < s; ++i) add_matvec(yt, w, J->states + (size_t)i * dd, qt, d);
                continue;
            }

            for (int i = 0; i < s; ++i) r[i] = dot(ut, kbar + (size_t)i * d, d);
            r[s] = dot(ut, ksum, d) / cnt;

            if (J->mode == OR_GRM || J->mode == OR_SOUP) {
                memcpy(g, r, (size_t)(s + 1) * sizeof(double));
                softmax(g, s + 1);
                if (J->mode == OR_GRM) {
                    add_matvec(yt, g[s], Mon, qt, d);
                    for (int i = 0; i < s; ++i) add_matvec(yt, g[i], J->states + (size_t)i * dd, qt, d);
                } else {
                    /* Memory Soup: average the memories' parameters first, then read once. */
                    for (size_t e = 0; e < dd; ++e) Mstar[e] = g[s] * Mon[e];
                    for (int i = 0; i < s; ++i) {
                        const double *Mi = J->states + (size_t)i * dd;
                        for (size_t e = 0; e < dd; ++e) Mstar[e] += g[i] * Mi[e];
                    }
                    add_matvec(yt, 1.0, Mstar, qt, d);
                }
                continue;
            }

            /* SSC */
            int nsel;
            double gp = INFINITY;
            if (J->given_sel) {
                const int32_t *gs = J->given_sel + (size_t)t * J->topk;
                nsel = 0;
                for (int c = 0; c < J->topk; ++c)
                    if (gs[c] >= 0) idx[nsel++] = gs[c];
            } else {
                nsel = ssc_rank(r, s, J->topk, idx, taken, &gp);
            }
            if (J->sel) {
                int32_t *so = J->sel + (size_t)t * J->topk;
                for (int c = 0; c < J->topk; ++c) so[c] = c < nsel ? idx[c] : -1;
            }
            if (J->gap) J->gap[t] = gp;
            for (int c = 0; c < nsel; ++c) g[c] = r[idx[c]];
            g[nsel] = r[s];
            softmax(g, nsel + 1);
            add_matvec(yt, g[nsel], Mon, qt, d);
            for (int c = 0; c < nsel; ++c) add_matvec(yt, g[c], J->states + (size_t)idx[c] * dd, qt, d);
        }
    }
    free(kbar); free(Mon); free(Mstar); free(ksum); free(r); free(g); free(idx); free(taken);
    return OR_OK;
}

/*
 * Weight of token j's outer product v_j k_j^T in a segment memory read at step t
 * (j <= t, both in the same segment, which starts at t0): 1 for the plain update;
 * for SWLA, unrolling eq. 28, lambda_j prod_{i=j+1..t} alpha_i plus (when j < t)
 * beta_{j+1} prod_{i=j+2..t} alpha_i.
 */
static double token_weight(const head_job *J, int j, int t)
{
    if (!J->alpha) return 1.0;
    double a_lam = J->lam[j], a_beta = j < t ? J->beta[j + 1] : 0.0;
    for (int i = j + 1; i <= t; ++i) a_lam *= J->alpha[i];
    for (int i = j + 2; i <= t; ++i) a_beta *= J->alpha[i];
    return a_lam + a_beta;
}

/*
 * Token-level twin (tiny inputs only): never forms a memory matrix.  For each
 * token it recomputes every pooled key from the raw keys, the gates, and then
 * y_t = sum_{j<=t} w_{t,seg(j)} v_j (k_j . q_t), the same sum regrouped by token
 * ([MC-sum §2.2]: N = L turns MC into direct access to every past token).
 */
static int head_bruteforce(const head_job *J)
{
    const int L = J->L, d = J->d;
    const int N = num_seg(J);
    double *w = malloc((size_t)(N + 1) * sizeof(double));
    double *r = malloc((size_t)(N + 1) * sizeof(double));
    double *pool = malloc((size_t)d * sizeof(double));
    int *order = malloc((size_t)(N + 1) * sizeof(int));
    if (!w || !r || !pool || !order) {
        free(w); free(r); free(pool); free(order);
        return OR_ERR_NOMEM;
    }
    for (int t = 0; t < L; ++t) {
        const int s = seg_of(J, t);
        const double *qt = J->q + (size_t)t * d, *ut = J->u + (size_t)t * d;
        /* pooled keys: segments i < s over their whole span, segment s from its start to t */
        for (int i = 0; i <= s; ++i) {
            int a0 = seg_lo(J, i), a1 = (i < s) ? seg_hi(J, i) : t + 1;
            memset(pool, 0, (size_t)d * sizeof(double));
            for (int j = a0; j < a1; ++j)
                for (int b = 0; b < d; ++b) pool[b] += J->k[(size_t)j * d + b];
            double acc = 0.0;
            for (int b = 0; b < d; ++b) acc += ut[b] * (pool[b] / (double)(a1 - a0));
            r[i] = acc;
        }
        for (int i = 0; i <= s; ++i) w[i] = 0.0;
        if (J->mode == OR_RESIDUAL) {
            for (int i = 0; i <= s; ++i) w[i] = 1.0;
        } else if (J->mode == OR_MEAN) {
            for (int i = 0; i <= s; ++i) w[i] = 1.0 / (double)(s + 1);
        } else if (J->mode == OR_GRM || J->mode == OR_SOUP) {
            double m = r[0];
            for (int i = 1; i <= s; ++i) m = r[i] > m ? r[i] : m;
            double z = 0.0;
            for (int i = 0; i <= s; ++i) z += exp(r[i] - m);
            for (int i = 0; i <= s; ++i) w[i] = exp(r[i] - m) / z;
        } else {
            /* SSC: sort cached indices by fp32 score descending, index ascending on ties */
            for (int i = 0; i < s; ++i) order[i] = i;
            for (int a = 1; a < s; ++a) { /* insertion sort, stable */
                int x = order[a], b = a - 1;
                while (b >= 0 && (float)r[order[b]] < (float)r[x]) {
                    order[b + 1] = order[b];
                    --b;
                }
                order[b + 1] = x;
            }
            int nsel = s < J->topk ? s : J->topk;
            double m = r[s];
            for (int c = 0; c < nsel; ++c) m = r[order[c]] > m ? r[order[c]] : m;
            double z = exp(r[s] - m);
            for (int c = 0; c < nsel; ++c) z += exp(r[order[c]] - m);
            for (int c = 0; c < nsel; ++c) w[order[c]] = exp(r[order[c]] - m) / z;
            w[s] = exp(r[s] - m) / z;
        }
        double *yt = J->y + (size_t)t * d;
        memset(yt, 0, (size_t)d * sizeof(double));
        for (int j = 0; j <= t; ++j) {
            const int sj = seg_of(J, j);
            double wj = w[sj];
            if (wj == 0.0) continue;
            /* a cached segment is read at its last token, the current one at t */
            const int seg_end = seg_hi(J, sj) - 1;
            wj *= token_weight(J, j, sj == s ? t : seg_end);
            double kq = dot(J->k + (size_t)j * d, qt, d);
            const double *vj = J->v + (size_t)j * d;
            for (int a = 0; a < d; ++a) yt[a] += wj * kq * vj[a];
        }
    }
    free(w); free(r); free(pool); free(order);
    return OR_OK;
}

/*
 * Gradient of the forward pass (plain linear memory) for an upstream gradient dy
 * of y: the chain rule taken through the forward's own steps, token by token.
 * With the aggregation y_t = g_on o_on + sum_c g_c o_c over the memories that take
 * part (o = M q_t, the online memory M_t^(s) and the selected cached M^(i)):
 *   dg = dy_t . o                                          (gate of each memory)
 *   softmax:  dr = g (dg - sum g dg)      (GRM / Soup / SSC over the selected set;
 *             the selection itself is piecewise constant and passes no gradient)
 *   scores:   r_i = <u_t, kbar_i>, r_on = <u_t, ksum_t> / cnt
 *             -> du_t, and d kbar_i += dr_i u_t, d k_j += dr_on u_t / cnt (j = t0..t)
 *   reads:    dq_t = sum g M^T dy_t;  a read of M = sum_j v_j k_j^T with weight g passes
 *             d v_j += g (k_j . q_t) dy_t,  d k_j += g (v_j . dy_t) q_t
 * Residual (g = 1) and Mean (g = 1 / (s + 1)) have constant gates.  Soup is the same
 * function as GRM for a linear memory (the parameter average read at q_t is the
 * gated sum of the reads), so it takes the same derivative.  A cached memory's
 * contributions are gathered per segment, G_i = sum_t g_{t,i} dy_t q_t^T, and
 * spread over its tokens at the end (d v_j += G_i k_j, d k_j += G_i^T v_j), with the
 * pooled key's gradient d kbar_i / |segment i|.
 */
static int head_backward(const head_job *J)
{
    const int L = J->L, d = J->d;
    const int N = num_seg(J);
    const size_t dd = (size_t)d * d;
    const int gated = J->mode == OR_GRM || J->mode == OR_SOUP || J->mode == OR_SSC;

    double *kbar = calloc((size_t)N * d, sizeof(double));
    double *Mon = malloc(dd * sizeof(double));
    double *ksum = malloc((size_t)d * sizeof(double));
    double *r = malloc((size_t)(N + 1) * sizeof(double));
    double *g = malloc((size_t)(N + 1) * sizeof(double));
    double *dg = malloc((size_t)(N + 1) * sizeof(double));
    double *o = malloc((size_t)d * sizeof(double));
    double *G = calloc((size_t)N * dd, sizeof(double));
    double *dkbar = calloc((size_t)N * d, sizeof(double));
    double *states = calloc((size_t)N * dd, sizeof(double));
    int *idx = malloc((size_t)(N + 1) * sizeof(int));
    uint8_t *taken = malloc((size_t)(N + 1));
    if (!kbar || !Mon || !ksum || !r || !g || !dg || !o || !G || !dkbar || !states || !idx || !taken) {
        free(kbar); free(Mon); free(ksum); free(r); free(g); free(dg); free(o); free(G); free(dkbar);
        free(states); free(idx); free(taken);
        return OR_ERR_NOMEM;
    }
    memset(J->dq, 0, (size_t)L * d * sizeof(double));
    memset(J->dk, 0, (size_t)L * d * sizeof(double));
    memset(J->dv, 0, (size_t)L * d * sizeof(double));
    memset(J->du, 0, (size_t)L * d * sizeof(double));

    /* the forward's cached states and pooled keys */
    for (int n = 0; n < N; ++n) {
        double *M = states + (size_t)n * dd;
        int t0 = seg_lo(J, n), t1 = seg_hi(J, n);
        for (int t = t0; t < t1; ++t) {
            memory_step(J, M, t, t0);
            for (int b = 0; b < d; ++b) kbar[(size_t)n * d + b] += J->k[(size_t)t * d + b];
        }
        for (int b = 0; b < d; ++b) kbar[(size_t)n * d + b] /= (double)(t1 - t0);
    }

    for (int s = 0; s < N; ++s) {
        int t0 = seg_lo(J, s), t1 = seg_hi(J, s);
        memset(Mon, 0, dd * sizeof(double));
        memset(ksum, 0, (size_t)d * sizeof(double));
        for (int t = t0; t < t1; ++t) {
            const double *qt = J->q + (size_t)t * d, *kt = J->k + (size_t)t * d;
            const double *ut = J->u + (size_t)t * d, *dyt = J->dy + (size_t)t * d;
            memory_step(J, Mon, t, t0);
            for (int b = 0; b < d; ++b) ksum[b] += kt[b];
            const double cnt = (double)(t - t0 + 1);

            /* the memories that take part (idx[0..nsel)) and their gates g[0..nsel], online last */
            int nsel = 0;
            if (gated) {
                for (int i = 0; i < s; ++i) r[i] = dot(ut, kbar + (size_t)i * d, d);
                r[s] = dot(ut, ksum, d) / cnt;
            }
            if (J->mode == OR_SSC && J->given_sel) { /* the forward evaluated on a given selection */
                const int32_t *gs = J->given_sel + (size_t)t * J->topk;
                for (int c = 0; c < J->topk; ++c)
                    if (gs[c] >= 0) idx[nsel++] = gs[c];
            } else if (J->mode == OR_SSC) {
                double gp;
                nsel = ssc_rank(r, s, J->topk, idx, taken, &gp);
            } else {
                for (int i = 0; i < s; ++i) idx[nsel++] = i;
            }
            if (gated) {
                for (int c = 0; c < nsel; ++c) g[c] = r[idx[c]];
                g[nsel] = r[s];
                softmax(g, nsel + 1);
            } else {
                const double w = J->mode == OR_MEAN ? 1.0 / (double)(s + 1) : 1.0;
                for (int c = 0; c <= nsel; ++c) g[c] = w;
            }

            /* gate gradients dg = dy_t . (M q_t) */
            for (int c = 0; c <= nsel; ++c) {
                const double *M = c < nsel ? states + (size_t)idx[c] * dd : Mon;
                memset(o, 0, (size_t)d * sizeof(double));
                add_matvec(o, 1.0, M, qt, d);
                dg[c] = dot(dyt, o, d);
            }
            if (gated) { /* softmax, then the scores */
                double sgd = 0.0;
                for (int c = 0; c <= nsel; ++c) sgd += g[c] * dg[c];
                double *dut = J->du + (size_t)t * d;
                for (int c = 0; c <= nsel; ++c) {
                    const double dr = g[c] * (dg[c] - sgd);
                    if (c < nsel) {
                        const double *kb = kbar + (size_t)idx[c] * d;
                        double *dkb = dkbar + (size_t)idx[c] * d;
                        for (int b = 0; b < d; ++b) {
                            dut[b] += dr * kb[b];
                            dkb[b] += dr * ut[b];
                        }
                    } else {
                        for (int b = 0; b < d; ++b) dut[b] += dr * ksum[b] / cnt;
                        for (int j = t0; j <= t; ++j)
                            for (int b = 0; b < d; ++b) J->dk[(size_t)j * d + b] += dr * ut[b] / cnt;
                    }
                }
            }

            /* the reads: dq_t, the online memory's tokens, and G of the cached memories */
            double *dqt = J->dq + (size_t)t * d;
            for (int c = 0; c <= nsel; ++c) {
                const double *M = c < nsel ? states + (size_t)idx[c] * dd : Mon;
                for (int a = 0; a < d; ++a)
                    for (int b = 0; b < d; ++b) dqt[b] += g[c] * M[(size_t)a * d + b] * dyt[a];
            }
            for (int c = 0; c < nsel; ++c) {
                double *Gi = G + (size_t)idx[c] * dd;
                for (int a = 0; a < d; ++a)
                    for (int b = 0; b < d; ++b) Gi[(size_t)a * d + b] += g[c] * dyt[a] * qt[b];
            }
            const double gon = g[nsel];
            for (int j = t0; j <= t; ++j) {
                const double *kj = J->k + (size_t)j * d, *vj = J->v + (size_t)j * d;
                const double kq = dot(kj, qt, d), vdy = dot(vj, dyt, d);
                for (int b = 0; b < d; ++b) {
                    J->dv[(size_t)j * d + b] += gon * kq * dyt[b];
                    J->dk[(size_t)j * d + b] += gon * vdy * qt[b];
                }
            }
        }
    }

    /* spread each cached memory's gradient over its segment's tokens */
    for (int n = 0; n < N; ++n) {
        const double *Gn = G + (size_t)n * dd;
        int t0 = seg_lo(J, n), t1 = seg_hi(J, n);
        for (int j = t0; j < t1; ++j) {
            const double *kj = J->k + (size_t)j * d, *vj = J->v + (size_t)j * d;
            double *dvj = J->dv + (size_t)j * d, *dkj = J->dk + (size_t)j * d;
            for (int a = 0; a < d; ++a)
                for (int b = 0; b < d; ++b) {
                    dvj[a] += Gn[(size_t)a * d + b] * kj[b];
                    dkj[b] += Gn[(size_t)a * d + b] * vj[a];
                }
            for (int b = 0; b < d; ++b) dkj[b] += dkbar[(size_t)n * d + b] / (double)(t1 - t0);
        }
    }
    free(kbar); free(Mon); free(ksum); free(r); free(g); free(dg); free(o); free(G); free(dkbar);
    free(states); free(idx); free(taken);
    return OR_OK;
}

/* ---- threading over (batch, head) ---- */

typedef struct {
    head_job base;
    int BH;
    int brute; /* 0 state form, 1 token-level twin, 2 backward */
    int next;  /* shared work counter */
    int status;
    pthread_mutex_t mu;
} pool_ctx;

static void *worker(void *arg)
{
    pool_ctx *P = (pool_ctx *)arg;
    const int L = P->base.L, d = P->base.d;
    const int N = num_seg(&P->base);
    const size_t Ld = (size_t)L * d, Ndd = (size_t)N * d * d;
    for (;;) {
        pthread_mutex_lock(&P->mu);
        int h = P->next++;
        pthread_mutex_unlock(&P->mu);
        if (h >= P->BH) break;
        head_job J = P->base;
        J.q += h * Ld; J.k += h * Ld; J.v += h * Ld; J.u += h * Ld;
        if (J.alpha) {
            J.alpha += (size_t)h * L; J.beta += (size_t)h * L; J.lam += (size_t)h * L;
        }
        if (J.y) J.y += h * Ld;
        if (J.states) J.states += h * Ndd;
        if (J.sel) J.sel += (size_t)h * L * J.topk;
        if (J.gap) J.gap += (size_t)h * L;
        if (J.given_sel) J.given_sel += (size_t)h * L * J.topk;
        if (J.dy) {
            J.dy += h * Ld; J.dq += h * Ld; J.dk += h * Ld; J.dv += h * Ld; J.du += h * Ld;
        }
        int st = P->brute == 2 ? head_backward(&J) : P->brute ? head_bruteforce(&J) : head_forward(&J);
        if (st != OR_OK) {
            pthread_mutex_lock(&P->mu);
            P->status = st;
            pthread_mutex_unlock(&P->mu);
        }
    }
    return NULL;
}

static int run_pool(pool_ctx *P, int nthreads)
{
    if (nthreads <= 0) {
        long nc = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = nc > 0 ? (int)nc : 1;
    }
    if (nthreads > P->BH) nthreads = P->BH;
    if (nthreads < 1) nthreads = 1;
    pthread_mutex_init(&P->mu, NULL);
    P->next = 0;
    P->status = OR_OK;
    pthread_t *th = malloc((size_t)nthreads * sizeof(pthread_t));
    if (!th) return OR_ERR_NOMEM;
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, worker, P) == 0) ++started;
    if (started == 0) worker(P);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&P->mu);
    return P->status;
}

static int check_args(int BH, int L, int d, int C, int mode, int topk)
{
    if (BH <= 0 || L <= 0 || d <= 0 || C <= 0) return OR_ERR_ARG;
    if (mode < OR_RESIDUAL || mode > OR_MEAN) return OR_ERR_ARG;
    if (mode == OR_SSC && topk < 0) return OR_ERR_ARG;
    return OR_OK;
}

/*
 * Full MC forward in state form.  y [BH][L][d] and states [BH][N][d][d] are
 * written.  For SSC, sel [BH][L][topk] (rank order, -1 padded) and gap [BH][L]
 * are written when non-NULL; given_sel (same layout), when non-NULL, replaces the
 * router's choice.  seg_mask [N] (may be NULL) restricts which segments' outputs
 * are computed (states are always computed in full).  nthreads <= 0: all cores.
 */
int mc_oracle_forward(const double *q, const double *k, const double *v, const double *u,
                      int BH, int L, int d, int C, int mode, int topk,
                      const uint8_t *seg_mask, const int32_t *given_sel,
                      double *y, double *states, int32_t *sel, double *gap, int nthreads)
{
    int st = check_args(BH, L, d, C, mode, topk);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y || !states) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, C, mode, mode == OR_SSC ? topk : 0,
                        seg_mask, mode == OR_SSC ? given_sel : NULL, y, states,
                        mode == OR_SSC ? sel : NULL, mode == OR_SSC ? gap : NULL, NULL, NULL, NULL,
                        NULL, NULL, NULL, NULL, NULL, NULL, 0};
    P.BH = BH;
    P.brute = 0;
    return run_pool(&P, nthreads);
}

/* The same forward with the SWLA (c = 2) update rule; alpha, beta, lam are [BH][L]. */
int mc_oracle_forward_swla(const double *q, const double *k, const double *v, const double *u,
                           const double *alpha, const double *beta, const double *lam,
                           int BH, int L, int d, int C, int mode, int topk,
                           const uint8_t *seg_mask, const int32_t *given_sel,
                           double *y, double *states, int32_t *sel, double *gap, int nthreads)
{
    int st = check_args(BH, L, d, C, mode, topk);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y || !states || !alpha || !beta || !lam) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, C, mode, mode == OR_SSC ? topk : 0,
                        seg_mask, mode == OR_SSC ? given_sel : NULL, y, states,
                        mode == OR_SSC ? sel : NULL, mode == OR_SSC ? gap : NULL, alpha, beta, lam,
                        NULL, NULL, NULL, NULL, NULL, NULL, 0};
    P.BH = BH;
    P.brute = 0;
    return run_pool(&P, nthreads);
}

/* Token-level twin: y only, O(L^2 d) per head, no memory matrices formed. */
int mc_oracle_bruteforce(const double *q, const double *k, const double *v, const double *u,
                         int BH, int L, int d, int C, int mode, int topk, double *y, int nthreads)
{
    int st = check_args(BH, L, d, C, mode, topk);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, C, mode, mode == OR_SSC ? topk : 0,
                        NULL, NULL, y, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0};
    P.BH = BH;
    P.brute = 1;
    return run_pool(&P, nthreads);
}

/* Token-level twin of the SWLA forward (y only). */
int mc_oracle_bruteforce_swla(const double *q, const double *k, const double *v, const double *u,
                              const double *alpha, const double *beta, const double *lam,
                              int BH, int L, int d, int C, int mode, int topk, double *y, int nthreads)
{
    int st = check_args(BH, L, d, C, mode, topk);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y || !alpha || !beta || !lam) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, C, mode, mode == OR_SSC ? topk : 0,
                        NULL, NULL, y, NULL, NULL, NULL, alpha, beta, lam, NULL, NULL, NULL, NULL, NULL, NULL, 0};
    P.BH = BH;
    P.brute = 1;
    return run_pool(&P, nthreads);
}

/*
 * Gradients of the forward (plain linear memory) for the upstream gradient dy:
 * dq, dk, dv, du [BH][L][d] are written (du is zero for Residual and Mean).
 * given_sel ([BH][L][topk], -1 padded; may be NULL) replaces the SSC router's
 * choice, as in mc_oracle_forward: the gradient is then that of the forward
 * evaluated on the given selection (the selection itself passes no gradient).
 */
int mc_oracle_backward(const double *q, const double *k, const double *v, const double *u, const double *dy,
                       int BH, int L, int d, int C, int mode, int topk, const int32_t *given_sel,
                       double *dq, double *dk, double *dv, double *du, int nthreads)
{
    int st = check_args(BH, L, d, C, mode, topk);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !dy || !dq || !dk || !dv || !du) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, C, mode, mode == OR_SSC ? topk : 0,
                        NULL, mode == OR_SSC ? given_sel : NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                        dy, dq, dk, dv, du, NULL, 0};
    P.BH = BH;
    P.brute = 2;
    return run_pool(&P, nthreads);
}

static int check_segments(int L, const int32_t *seg_off, int nseg)
{
    if (!seg_off || nseg <= 0 || seg_off[0] != 0 || seg_off[nseg] != L) return OR_ERR_ARG;
    for (int n = 0; n < nseg; ++n)
        if (seg_off[n + 1] <= seg_off[n]) return OR_ERR_ARG;
    return OR_OK;
}

/*
 * The forward with given segment boundaries: segment n is tokens
 * [seg_off[n], seg_off[n+1]) (seg_off[0] = 0, strictly increasing, seg_off[nseg] = L),
 * the same for every (batch, head).  Everything else as mc_oracle_forward; states
 * is [BH][nseg][d][d].
 */
int mc_oracle_forward_segments(const double *q, const double *k, const double *v, const double *u,
                               int BH, int L, int d, const int32_t *seg_off, int nseg, int mode, int topk,
                               const int32_t *given_sel, double *y, double *states, int32_t *sel, double *gap,
                               int nthreads)
{
    int st = check_args(BH, L, d, 1, mode, topk);
    if (st == OR_OK) st = check_segments(L, seg_off, nseg);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y || !states) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, 1, mode, mode == OR_SSC ? topk : 0,
                        NULL, mode == OR_SSC ? given_sel : NULL, y, states,
                        mode == OR_SSC ? sel : NULL, mode == OR_SSC ? gap : NULL, NULL, NULL, NULL,
                        NULL, NULL, NULL, NULL, NULL, seg_off, nseg};
    P.BH = BH;
    P.brute = 0;
    return run_pool(&P, nthreads);
}

/* Token-level twin with given segment boundaries (y only). */
int mc_oracle_bruteforce_segments(const double *q, const double *k, const double *v, const double *u,
                                  int BH, int L, int d, const int32_t *seg_off, int nseg, int mode, int topk,
                                  double *y, int nthreads)
{
    int st = check_args(BH, L, d, 1, mode, topk);
    if (st == OR_OK) st = check_segments(L, seg_off, nseg);
    if (st != OR_OK) return st;
    if (!q || !k || !v || !u || !y) return OR_ERR_ARG;
    pool_ctx P;
    memset(&P, 0, sizeof(P));
    P.base = (head_job){q, k, v, u, L, d, 1, mode, mode == OR_SSC ? topk : 0,
                        NULL, NULL, y, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                        seg_off, nseg};
    P.BH = BH;
    P.brute = 1;
    return run_pool(&P, nthreads);
}
