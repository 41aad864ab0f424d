/*
 * kvc_oracle.c -- plain fp64 CPU oracle for the budgeted-KV decode step and
 * the LaProx prefill scorer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA library against a
 * slow, obviously correct restatement of the method.  It shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Inputs are bf16 bit patterns (uint16) exactly as the GPU received them;
 * every value is widened to double before any arithmetic.  All arithmetic
 * is double precision, in the order the method states it, with no blocking
 * or fusion.
 *
 * Sources (web pages; section / equation / algorithm named per function):
 *   [MomentKV]  "MOMENTKV: Closing the Directional Gap in KV Cache Eviction
 *               for Long-Context Inference" (arXiv 2606.01563)
 *   [InertiaKV] "Key factors of KV cache eviction in aggressive decoding:
 *               temporal aggregation and rank preservation" (InertiaKV,
 *               arXiv 2609.03515)
 *   [KeepKV]    "KeepKV: lossless KV cache compression with electoral votes
 *               and zero-perturbation merging" (reading notes on arXiv
 *               2504.09936)
 *   [LaProx]    "Reformulating KV Cache Eviction Problem for Long-Context
 *               LLM Inference" (NeurIPS 2026 notes, arXiv 2605.07234)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* helpers                                                             */
/* ------------------------------------------------------------------ */

/* bf16 -> double: the bf16 bit pattern is the top half of an IEEE float. */
static double bfd(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* decode-step session                                                 */
/* ------------------------------------------------------------------ */

/*
 * One session holds U independent units (sequence, layer, KV head).  Each
 * unit keeps its cache as a list of slots ordered by token position, and the
 * eviction-set moment statistics as the four raw running sums the MomentKV
 * page defines (count n_e, key sum s_k, value sum s_v, outer-product sum
 * S = sum v k^T) [MomentKV sec 4.1 "efficient statistics update"; App. A.1].
 */
typedef struct {
    int U, G, d, cap;
    int *n;           /* slots present per unit                           */
    int32_t *pos;     /* [U][cap] token position of each slot              */
    int32_t *vote;    /* [U][cap] integer vote p_i (KeepKV eq 6)           */
    double *util;     /* [U][cap] aggregated utility m(i)                  */
    uint8_t *scored;  /* [U][cap] 0 = never scored (protected)             */
    uint16_t *k, *v;  /* [U][cap][d] bf16 bits                             */
    double *ne;       /* [U]      eviction count n_e (vote-weighted)       */
    double *sk, *sv;  /* [U][d]   s_k, s_v                                 */
    double *S;        /* [U][d][d] S[a][b] = sum v_a k_b                   */
} ocl_session;

void *ocl_create(int U, int G, int d, int cap)
{
    ocl_session *s = (ocl_session *)calloc(1, sizeof *s);
    if (!s) return NULL;
    s->U = U; s->G = G; s->d = d; s->cap = cap;
    size_t uc = (size_t)U * cap;
    s->n = (int *)calloc((size_t)U, sizeof(int));
    s->pos = (int32_t *)calloc(uc, sizeof(int32_t));
    s->vote = (int32_t *)calloc(uc, sizeof(int32_t));
    s->util = (double *)calloc(uc, sizeof(double));
    s->scored = (uint8_t *)calloc(uc, 1);
    s->k = (uint16_t *)calloc(uc * d, sizeof(uint16_t));
    s->v = (uint16_t *)calloc(uc * d, sizeof(uint16_t));
    s->ne = (double *)calloc((size_t)U, sizeof(double));
    s->sk = (double *)calloc((size_t)U * d, sizeof(double));
    s->sv = (double *)calloc((size_t)U * d, sizeof(double));
    s->S = (double *)calloc((size_t)U * d * d, sizeof(double));
    if (!s->n || !s->pos || !s->vote || !s->util || !s->scored || !s->k ||
        !s->v || !s->ne || !s->sk || !s->sv || !s->S) {
        free(s->n); free(s->pos); free(s->vote); free(s->util);
        free(s->scored); free(s->k); free(s->v); free(s->ne); free(s->sk);
        free(s->sv); free(s->S); free(s);
        return NULL;
    }
    return s;
}

void ocl_destroy(void *h)
{
    ocl_session *s = (ocl_session *)h;
    if (!s) return;
    free(s->n); free(s->pos); free(s->vote); free(s->util); free(s->scored);
    free(s->k); free(s->v); free(s->ne); free(s->sk); free(s->sv); free(s->S);
    free(s);
}

/*
 * Load the prefill cache of unit u: n slots, positions pos[0..n), optional
 * votes (NULL = all 1).  All slots start unscored; the moment statistics
 * start at zero at the start of each generation [MomentKV sec A4 setup].
 * Returns 0, or -1 if n exceeds the capacity.
 */
int ocl_load(void *h, int u, int n, const uint16_t *k, const uint16_t *v,
             const int32_t *vote, const int32_t *pos)
{
    ocl_session *s = (ocl_session *)h;
    int d = s->d;
    if (u < 0 || u >= s->U || n < 0 || n > s->cap) return -1;
    size_t base = (size_t)u * s->cap;
    for (int i = 0; i < n; i++) {
        s->pos[base + i] = pos[i];
        s->vote[base + i] = vote ? vote[i] : 1;
        s->util[base + i] = 0.0;
        s->scored[base + i] = 0;
        memcpy(&s->k[(base + i) * d], &k[(size_t)i * d], d * sizeof(uint16_t));
        memcpy(&s->v[(base + i) * d], &v[(size_t)i * d], d * sizeof(uint16_t));
    }
    s->n[u] = n;
    s->ne[u] = 0.0;
    memset(&s->sk[(size_t)u * d], 0, d * sizeof(double));
    memset(&s->sv[(size_t)u * d], 0, d * sizeof(double));
    memset(&s->S[(size_t)u * d * d], 0, (size_t)d * d * sizeof(double));
    return 0;
}

/*
 * Append the new token of this decode step to every unit: its key and value,
 * vote 1, position new_pos, not yet scored.  [MomentKV Algorithm 1: the
 * new pair joins the retained set before eviction; KeepKV Algorithm 1,
 * decoding stage: a new pair enters with vote 1].  Returns -1 if a unit is
 * full.
 */
int ocl_append(void *h, const uint16_t *knew, const uint16_t *vnew,
               int32_t new_pos)
{
    ocl_session *s = (ocl_session *)h;
    int d = s->d;
    for (int u = 0; u < s->U; u++)
        if (s->n[u] >= s->cap) return -1;
    for (int u = 0; u < s->U; u++) {
        size_t i = (size_t)u * s->cap + s->n[u];
        s->pos[i] = new_pos;
        s->vote[i] = 1;
        s->util[i] = 0.0;
        s->scored[i] = 0;
        memcpy(&s->k[i * d], &knew[(size_t)u * d], d * sizeof(uint16_t));
        memcpy(&s->v[i * d], &vnew[(size_t)u * d], d * sizeof(uint16_t));
        s->n[u] += 1;
    }
    return 0;
}

/*
 * Vote-weighted single-query attention over all slots present, for each of
 * the G query heads that share the unit's KV head.
 *
 *   logit  x_hi = q_h . k_i / sqrt(d) + ln p_i
 *          [MomentKV sec 2 notation s_i = q^T k_i / sqrt(d); KeepKV eq 6 /
 *           eq 23 vote weighting, written as the logit bias ln p_i of the
 *           KeepKV "integration" item 2]
 *   lse_h  = log sum_i exp(x_hi)                  (max-shifted)
 *   a_hi   = exp(x_hi - lse_h)                    (attention probability)
 *   f_h    = sum_i a_hi v_i                       [MomentKV sec 2; KeepKV eq 1]
 *   probs_i = (1/G) sum_h a_hi   head-mean score  [InertiaKV sec 3.1 eq 1,
 *                                 mean taken over the query heads of the
 *                                 KV group]
 *
 * Outputs: lse [U][G], f [U][G][d], probs [U][cap] (slot order; entries past
 * n[u] untouched).  Any output pointer may be NULL.
 */
/* One unit of ocl_attend; lse [G], f [G][d] and probs [n] are the unit's
 * own rows (any may be NULL). */
static void attend_unit(ocl_session *s, int u, const uint16_t *q, double *lse, double *f,
                        double *probs)
{
    int G = s->G, d = s->d, cap = s->cap;
    double rsd = 1.0 / sqrt((double)d);
    {
        int n = s->n[u];
        size_t base = (size_t)u * cap;
        double *x = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        double *ps = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
        for (int hh = 0; hh < G; hh++) {
            const uint16_t *qh = &q[((size_t)u * G + hh) * d];
            double mx = -INFINITY;
            for (int i = 0; i < n; i++) {
                const uint16_t *ki = &s->k[(base + i) * d];
                double dot = 0.0;
                for (int a = 0; a < d; a++) dot += bfd(qh[a]) * bfd(ki[a]);
                x[i] = dot * rsd + log((double)s->vote[base + i]);
                if (x[i] > mx) mx = x[i];
            }
            double z = 0.0;
            for (int i = 0; i < n; i++) z += exp(x[i] - mx);
            double l = mx + log(z);
            if (lse) lse[hh] = l;
            if (f) {
                double *fh = &f[(size_t)hh * d];
                for (int a = 0; a < d; a++) fh[a] = 0.0;
                for (int i = 0; i < n; i++) {
                    double ai = exp(x[i] - l);
                    const uint16_t *vi = &s->v[(base + i) * d];
                    for (int a = 0; a < d; a++) fh[a] += ai * bfd(vi[a]);
                }
            }
            for (int i = 0; i < n; i++) ps[i] += exp(x[i] - l);
        }
        if (probs)
            for (int i = 0; i < n; i++) probs[i] = ps[i] / (double)G;
        free(x);
        free(ps);
    }
}

void ocl_attend(void *h, const uint16_t *q, double *lse, double *f,
                double *probs)
{
    ocl_session *s = (ocl_session *)h;
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < s->U; u++)
        attend_unit(s, u, q, lse ? &lse[(size_t)u * s->G] : NULL,
                    f ? &f[(size_t)u * s->G * s->d] : NULL,
                    probs ? &probs[(size_t)u * s->cap] : NULL);
}

/*
 * Temporal utility aggregation on a refresh step [InertiaKV sec 3.1 eqs 2-4]:
 *   single      m = s
 *   cumulative  m = m_prev + s
 *   EMA         m = alpha * m_prev + (1 - alpha) * s
 * A slot seen for the first time takes m = s under every rule (reading of a
 * step the surviving InertiaKV text leaves open; it equals the KeepKV
 * bias-corrected EMA at its first observation, eq 14).
 * probs is [U][cap] in slot order.
 */
void ocl_update_util(void *h, const double *probs, int rule, double alpha)
{
    ocl_session *s = (ocl_session *)h;
    for (int u = 0; u < s->U; u++) {
        size_t base = (size_t)u * s->cap;
        for (int i = 0; i < s->n[u]; i++) {
            double sc = probs[base + i];
            double *m = &s->util[base + i];
            if (!s->scored[base + i]) {
                *m = sc;
                s->scored[base + i] = 1;
            } else if (rule == 0) {
                *m = sc;
            } else if (rule == 1) {
                *m = *m + sc;
            } else {
                *m = alpha * (*m) + (1.0 - alpha) * sc;
            }
        }
    }
}

/*
 * The layer-chained EMA of InertiaKV's evaluated implementation [InertiaKV
 * sec 1 and sec 3.1, last paragraph: compression runs at several layers and
 * one running EMA state is updated after each of them, so that alpha weighs
 * both the persistence across decode steps and the influence of consecutive
 * layers; sec 3.1 eq 1: s_t(i) is the mean over all H query heads].  Units
 * are grouped by sequence: unit u = (b NL + l) Hkv + g, and every unit of a
 * sequence holds the same positions in the same slot order (one retained set
 * per sequence).  On a refresh step, for every slot i of sequence b, for
 * l = 0 .. NL - 1 in order:
 *   s_l(i) = (1/Hkv) sum_g probs[(b NL + l) Hkv + g][i]   (the layer's mean
 *            over its H = Hkv G query heads: probs are group means already)
 *   m(i)   = s_l(i) at the first observation, else alpha m(i) + (1-alpha) s_l(i).
 * The result is stored as the utility of slot i in every unit of the
 * sequence (so a per-unit selection picks the same slots everywhere).
 * Returns 0, or -1 if U is not a multiple of NL Hkv or the sequence's units
 * differ in length.
 */
int ocl_update_util_chained(void *h, const double *probs, int NL, int Hkv, double alpha)
{
    ocl_session *s = (ocl_session *)h;
    int per = NL * Hkv;
    if (NL < 1 || Hkv < 1 || s->U % per != 0) return -1;
    for (int b = 0; b < s->U / per; b++) {
        int u0 = b * per, n = s->n[u0];
        for (int q = 1; q < per; q++)
            if (s->n[u0 + q] != n) return -1;
        for (int i = 0; i < n; i++) {
            size_t i0 = (size_t)u0 * s->cap + i;
            double m = s->util[i0];
            int seen = s->scored[i0];
            for (int l = 0; l < NL; l++) {
                double sl = 0.0;
                for (int g = 0; g < Hkv; g++)
                    sl += probs[(size_t)(u0 + l * Hkv + g) * s->cap + i];
                sl /= (double)Hkv;
                if (!seen) { m = sl; seen = 1; }
                else m = alpha * m + (1.0 - alpha) * sl;
            }
            for (int q = 0; q < per; q++) {
                size_t iq = (size_t)(u0 + q) * s->cap + i;
                s->util[iq] = m;
                s->scored[iq] = 1;
            }
        }
    }
    return 0;
}

/*
 * Moment-informed eviction scores [MomentKV sec 4.2, "moment residual" and
 * "moment-aware eviction score"; Algorithm 1, phase 1]: for every live slot
 *   r_i = v_i - v_bar - S_tilde (k_i - k_bar) / (n_e sqrt(d))
 *   (v_bar = s_v / n_e, k_bar = s_k / n_e, S_tilde = S - s_v s_k^T / n_e;
 *    r_i = v_i while n_e = 0, as the algorithm sets v_bar, S_tilde to 0)
 *   score_i = alpha_i ||r_i||_2,
 * alpha_i being the slot's attention weight, given in probs [U][cap] (the
 * head-mean of the vote-weighted probabilities, as ocl_attend writes it).
 * Output: out [U][cap] (entries past n[u] untouched).
 */
/* One unit of ocl_mi_scores; probs and out are the unit's rows [n]. */
static void mi_unit(ocl_session *s, int u, const double *probs, double *out)
{
    int d = s->d;
    double rsd = 1.0 / sqrt((double)d);
    {
        size_t base = (size_t)u * s->cap;
        double ne = s->ne[u];
        const double *sk = &s->sk[(size_t)u * d], *sv = &s->sv[(size_t)u * d];
        const double *S = &s->S[(size_t)u * d * d];
        double *dk = (double *)malloc((size_t)d * sizeof(double));
        for (int i = 0; i < s->n[u]; i++) {
            const uint16_t *ki = &s->k[(base + i) * d], *vi = &s->v[(base + i) * d];
            double rr = 0.0;
            if (ne > 0.0) {
                for (int b = 0; b < d; b++) dk[b] = bfd(ki[b]) - sk[b] / ne;
                for (int a = 0; a < d; a++) {
                    double t = 0.0;
                    for (int b = 0; b < d; b++)
                        t += (S[(size_t)a * d + b] - sv[a] * sk[b] / ne) * dk[b];
                    double r = bfd(vi[a]) - sv[a] / ne - t / ne * rsd;
                    rr += r * r;
                }
            } else {
                for (int a = 0; a < d; a++) rr += bfd(vi[a]) * bfd(vi[a]);
            }
            out[i] = probs[i] * sqrt(rr);
        }
        free(dk);
    }
}

void ocl_mi_scores(void *h, const double *probs, double *out)
{
    ocl_session *s = (ocl_session *)h;
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < s->U; u++)
        mi_unit(s, u, &probs[(size_t)u * s->cap], &out[(size_t)u * s->cap]);
}

/*
 * Set the utilities of unit u's first n slots and mark them scored (a
 * utility carried over from the prefill, e.g. KeepKV's windowed EMA
 * initialization).  Returns 0, or -1 if n exceeds the slots present.
 */
int ocl_set_util(void *h, int u, int n, const double *util)
{
    ocl_session *s = (ocl_session *)h;
    if (u < 0 || u >= s->U || n < 0 || n > s->n[u]) return -1;
    size_t base = (size_t)u * s->cap;
    for (int i = 0; i < n; i++) {
        s->util[base + i] = util[i];
        s->scored[base + i] = 1;
    }
    return 0;
}

/* Export the slot table (positions, votes, utilities, scored flags). */
void ocl_get_slots(void *h, int32_t *n, int32_t *pos, int32_t *vote,
                   double *util, uint8_t *scored)
{
    ocl_session *s = (ocl_session *)h;
    size_t uc = (size_t)s->U * s->cap;
    for (int u = 0; u < s->U; u++) n[u] = s->n[u];
    if (pos) memcpy(pos, s->pos, uc * sizeof(int32_t));
    if (vote) memcpy(vote, s->vote, uc * sizeof(int32_t));
    if (util) memcpy(util, s->util, uc * sizeof(double));
    if (scored) memcpy(scored, s->scored, uc);
}

typedef struct { double m; int32_t pos; } ocl_key;

static int key_cmp(const void *a, const void *b)
{
    const ocl_key *x = (const ocl_key *)a, *y = (const ocl_key *)b;
    if (x->m < y->m) return -1;
    if (x->m > y->m) return 1;
    return (x->pos < y->pos) ? -1 : (x->pos > y->pos);
}

/*
 * Proposed victims of one eviction round: while a unit holds more than L
 * slots, the lowest-utility slots go [InertiaKV sec 3.1 "evict the token
 * with the lowest m_t(i)"; MomentKV Algorithm 1 phase 1 argmin loop].
 * k = n - L victims are the first k scored slots in (m ascending, position
 * ascending) order; unscored slots are never candidates.  Writes victim
 * positions in that order to victims [U][kmax], their count to nvict [U],
 * and the k-th (largest evicted) utility to thr [U] (0 when k = 0).
 * Lu [U] (or NULL): a budget per unit in place of L.
 * Returns 0, or -1 if some unit has fewer than k scored slots or k > kmax.
 */
int ocl_select(void *h, int L, int kmax, int32_t *victims, int32_t *nvict,
               double *thr, const int32_t *Lu)
{
    ocl_session *s = (ocl_session *)h;
    int rc = 0;
    for (int u = 0; u < s->U; u++) {
        size_t base = (size_t)u * s->cap;
        int n = s->n[u], Lb = Lu ? Lu[u] : L;
        int k = n > Lb ? n - Lb : 0;
        nvict[u] = 0;
        if (thr) thr[u] = 0.0;
        if (k == 0) continue;
        ocl_key *keys = (ocl_key *)malloc((size_t)n * sizeof(ocl_key));
        int ns = 0;
        for (int i = 0; i < n; i++)
            if (s->scored[base + i]) {
                keys[ns].m = s->util[base + i];
                keys[ns].pos = s->pos[base + i];
                ns++;
            }
        if (ns < k || k > kmax) { free(keys); rc = -1; continue; }
        qsort(keys, (size_t)ns, sizeof(ocl_key), key_cmp);
        for (int j = 0; j < k; j++) victims[(size_t)u * kmax + j] = keys[j].pos;
        nvict[u] = k;
        if (thr) thr[u] = keys[k - 1].m;
        free(keys);
    }
    return rc;
}

/*
 * Evict the given positions.  Each evicted token is folded into the raw
 * eviction-set sums with its vote as weight (a slot with vote p stands for
 * p identical tokens, KeepKV eq 6 "equivalent to p duplicated pairs"):
 *   n_e += p,  s_k += p k,  s_v += p v,  S += p v k^T
 * [MomentKV Algorithm 1, eviction phase; App. A.1 update by plain
 * addition], then the slot is removed, keeping the rest in position order.
 * Returns 0, or -1 if a position is not present.
 */
static int evict_unit(ocl_session *s, int u, const int32_t *victims, int nv)
{
    int d = s->d, rc = 0;
    {
        size_t base = (size_t)u * s->cap;
        int n = s->n[u];
        uint8_t *gone = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
        for (int j = 0; j < nv; j++) {
            int32_t p = victims[j];
            int i = 0;
            while (i < n && (s->pos[base + i] != p || gone[i])) i++;
            if (i == n) { rc = -1; continue; }
            gone[i] = 1;
            double w = (double)s->vote[base + i];
            const uint16_t *ki = &s->k[(base + i) * d];
            const uint16_t *vi = &s->v[(base + i) * d];
            double *sk = &s->sk[(size_t)u * d], *sv = &s->sv[(size_t)u * d];
            double *S = &s->S[(size_t)u * d * d];
            s->ne[u] += w;
            for (int a = 0; a < d; a++) {
                sk[a] += w * bfd(ki[a]);
                sv[a] += w * bfd(vi[a]);
            }
            for (int a = 0; a < d; a++)
                for (int b = 0; b < d; b++)
                    S[(size_t)a * d + b] += w * bfd(vi[a]) * bfd(ki[b]);
        }
        int w = 0;
        for (int i = 0; i < n; i++) {
            if (gone[i]) continue;
            if (w != i) {
                s->pos[base + w] = s->pos[base + i];
                s->vote[base + w] = s->vote[base + i];
                s->util[base + w] = s->util[base + i];
                s->scored[base + w] = s->scored[base + i];
                memmove(&s->k[(base + w) * d], &s->k[(base + i) * d], d * sizeof(uint16_t));
                memmove(&s->v[(base + w) * d], &s->v[(base + i) * d], d * sizeof(uint16_t));
            }
            w++;
        }
        s->n[u] = w;
        free(gone);
    }
    return rc;
}

int ocl_evict(void *h, const int32_t *victims, const int32_t *nvict, int kmax)
{
    ocl_session *s = (ocl_session *)h;
    int rc = 0;
    for (int u = 0; u < s->U; u++)
        if (evict_unit(s, u, &victims[(size_t)u * kmax], nvict[u]) != 0) rc = -1;
    return rc;
}

/*
 * Moment-aware eviction phase of one decode step [MomentKV Algorithm 1,
 * phase 1; sec 4.2 "moment residual" and "moment-aware eviction score"]:
 * while a unit holds more than L slots,
 *   - alpha = softmax over the slots still present (re-formed every round,
 *     so it renormalizes over R; for a GQA group the head mean of the G
 *     query heads' vote-weighted probabilities, as ocl_attend forms it),
 *   - k_bar, v_bar, S_tilde from the running sums as they stand (zero
 *     residual model while n_e = 0),
 *   - score(j) = alpha_j ||v_j - v_bar - S_tilde (k_j - k_bar)/(n_e sqrt d)||,
 *   - the slot with the lowest score goes (ties to the smaller position),
 *     folded into the sums with its vote as weight and removed,
 * so every round sees the moments and the softmax left by the previous one.
 * With one victim this is one scoring pass and one argmin.
 * forced [U][kmax] (positions, or NULL): when given, round r of unit u
 * removes forced[u][r] instead of its own argmin (the caller replays another
 * implementation's choices and checks each against best / used).
 * Outputs: victims [U][kmax] positions in eviction order, nvict [U],
 * best [U][kmax] the lowest score of each round, used [U][kmax] the score of
 * the slot removed in that round (NULL allowed), scores0 [U][cap] the scores
 * of the first round (slot order before the step's removals; NULL allowed).
 * Returns 0, or -1 if k > kmax or a forced position is not present.
 */
int ocl_mi_greedy(void *h, const uint16_t *q, int L, int kmax, const int32_t *forced,
                  int32_t *victims, int32_t *nvict, double *best, double *used,
                  double *scores0, const int32_t *Lu)
{
    ocl_session *s = (ocl_session *)h;
    int rc = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : rc)
    for (int u = 0; u < s->U; u++) {
        size_t base = (size_t)u * s->cap;
        int Lb = Lu ? Lu[u] : L;
        int k = s->n[u] > Lb ? s->n[u] - Lb : 0;
        nvict[u] = 0;
        if (k > kmax) { rc = -1; continue; }
        double *pr = (double *)malloc((size_t)s->cap * sizeof(double));
        double *sc = (double *)malloc((size_t)s->cap * sizeof(double));
        for (int r = 0; r < k; r++) {
            attend_unit(s, u, q, NULL, NULL, pr);
            mi_unit(s, u, pr, sc);
            int n = s->n[u], jb = 0;
            for (int i = 1; i < n; i++) {
                double a = sc[i], b = sc[jb];
                if (a < b || (a == b && s->pos[base + i] < s->pos[base + jb])) jb = i;
            }
            if (r == 0 && scores0)
                for (int i = 0; i < n; i++) scores0[base + i] = sc[i];
            int32_t vp = s->pos[base + jb];
            double vs = sc[jb];
            if (best) best[(size_t)u * kmax + r] = sc[jb];
            if (forced) {
                vp = forced[(size_t)u * kmax + r];
                int i = 0;
                while (i < n && s->pos[base + i] != vp) i++;
                if (i == n) { rc = -1; break; }
                vs = sc[i];
            }
            if (used) used[(size_t)u * kmax + r] = vs;
            for (int i = 0; i < n; i++) {          /* the slot's score as its utility */
                s->util[base + i] = sc[i];
                s->scored[base + i] = 1;
            }
            victims[(size_t)u * kmax + r] = vp;
            nvict[u] = r + 1;
            if (evict_unit(s, u, &vp, 1) != 0) { rc = -1; break; }
        }
        free(pr);
        free(sc);
    }
    return rc;
}

/*
 * Nearest bf16 of a double, ties to the even pattern (one rounding step:
 * the candidates around the float conversion are compared in double).
 */
static uint16_t dbf(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t a = (uint16_t)(u >> 16);          /* bf16 of f truncated toward 0 */
    uint16_t best = a;
    double bd = fabs(bfd(a) - x);
    for (int j = -1; j <= 1; j += 2) {
        if (j < 0 && (a & 0x7FFF) == 0) continue;
        uint16_t c = (uint16_t)(a + j);
        double cd = fabs(bfd(c) - x);
        if (cd < bd || (cd == bd && (c & 1) == 0)) { best = c; bd = cd; }
    }
    return best;
}

/*
 * KeepKV ZIP-merging of one victim per unit into its most similar retained
 * slot, instead of dropping it [KeepKV reading notes, "ZIP-Merging" eqs
 * 7-12; candidate choice by the cosine similarity of keys, the most recent
 * R tokens excluded ("why cosine similarity"); the epsilon guard of the
 * "numerical stability" item 2].
 *
 * victim[u]: position of the unit's victim, or -1 (unit untouched).
 * Candidates c: live slots other than the victim whose position is at most
 * new_pos - R (the last R positions of the sequence are excluded).  The
 * partner maximizes cos(k_e, k_c) = k_e . k_c / (|k_e| |k_c|) (0 when a norm
 * is 0), ties to the smaller position; force[u] >= 0 (optional) names the
 * partner's position instead (it must be a candidate).  No candidate: the
 * unit is left untouched, partner[u] = -1.
 *
 * Scores (reading for a GQA group): ln s_j = xbar_j = (1/G) sum_h q_h . k_j
 * / sqrt(d), the logit of the group's mean query, so that the page's
 * single-head formula applies unchanged (G = 1 gives it exactly).  With
 * weights w_j = p_j s_j (eq 8), lambda_j = w_j / (w_e + w_c):
 *   v_r = lambda_e v_e + lambda_c v_c                            (eq 10)
 *   xt  = lambda_e xbar_e + lambda_c xbar_c
 *   ell = ln((w_e + w_c) / (p_e + p_c))
 *   k_r = (lambda_e k_e + lambda_c k_c) ell / xt                 (eq 12,
 *         numerator and denominator divided by w_e + w_c)
 *   |xt| < eps: k_r = (k_e + k_c) / 2                            (guard)
 *   p_r = p_e + p_c                                              (eq 7)
 * Weights are formed after subtracting max(xbar_e, xbar_c).  The partner
 * slot takes k_r, v_r rounded to bf16, the vote p_r and (reading) the sum
 * of the two utilities, and keeps its position and scored flag; the
 * victim's slot is removed.  Outputs per unit (any may be NULL): partner
 * position, the largest candidate cosine and the partner's, the unrounded
 * k_r and v_r [U][d], the guard flag and xt.  Returns 0, or -1 if a victim or
 * a forced partner is not present / not a candidate.
 */
int ocl_zip_merge(void *h, const uint16_t *q, const int32_t *victim, int32_t new_pos,
                  int R, double eps, const int32_t *force, int32_t *partner,
                  double *cos_best, double *cos_used, double *kr, double *vr,
                  int32_t *guard, double *xt_out)
{
    ocl_session *s = (ocl_session *)h;
    int G = s->G, d = s->d, rc = 0;
    double rsd = 1.0 / sqrt((double)d);
    double *kre = (double *)malloc((size_t)d * sizeof(double));
    double *vre = (double *)malloc((size_t)d * sizeof(double));
    for (int u = 0; u < s->U; u++) {
        if (partner) partner[u] = -1;
        if (guard) guard[u] = 0;
        if (victim[u] < 0) continue;
        size_t base = (size_t)u * s->cap;
        int n = s->n[u], e = 0;
        while (e < n && s->pos[base + e] != victim[u]) e++;
        if (e == n) { rc = -1; continue; }
        const uint16_t *ke = &s->k[(base + e) * d];
        double nke = 0.0;
        for (int a = 0; a < d; a++) nke += bfd(ke[a]) * bfd(ke[a]);
        nke = sqrt(nke);
        int c = -1, cf = -1;
        double cb = -INFINITY, cu = 0.0;
        for (int i = 0; i < n; i++) {
            if (i == e || s->pos[base + i] > new_pos - R) continue;
            const uint16_t *ki = &s->k[(base + i) * d];
            double dot = 0.0, nki = 0.0;
            for (int a = 0; a < d; a++) {
                dot += bfd(ke[a]) * bfd(ki[a]);
                nki += bfd(ki[a]) * bfd(ki[a]);
            }
            nki = sqrt(nki);
            double cs = (nke > 0.0 && nki > 0.0) ? dot / (nke * nki) : 0.0;
            /* slots are in position order: the first maximum is the oldest */
            if (cs > cb) { cb = cs; c = i; }
            if (force && force[u] >= 0 && s->pos[base + i] == force[u]) { cf = i; cu = cs; }
        }
        if (c < 0) continue;
        if (force && force[u] >= 0) {
            if (cf < 0) { rc = -1; continue; }
            c = cf;
        } else {
            cu = cb;
        }
        if (cos_best) cos_best[u] = cb;
        if (cos_used) cos_used[u] = cu;
        const uint16_t *kc = &s->k[(base + c) * d];
        const uint16_t *ve = &s->v[(base + e) * d], *vc = &s->v[(base + c) * d];
        double xe = 0.0, xc = 0.0;
        for (int hh = 0; hh < G; hh++) {
            const uint16_t *qh = &q[((size_t)u * G + hh) * d];
            for (int a = 0; a < d; a++) {
                xe += bfd(qh[a]) * bfd(ke[a]);
                xc += bfd(qh[a]) * bfd(kc[a]);
            }
        }
        xe *= rsd / G;
        xc *= rsd / G;
        double pe = (double)s->vote[base + e], pc = (double)s->vote[base + c];
        double m = xe > xc ? xe : xc;
        double we = pe * exp(xe - m), wc = pc * exp(xc - m), W = we + wc;
        double le = we / W, lc = wc / W;
        double xt = le * xe + lc * xc;
        double ell = m + log(W / (pe + pc));
        int gd = fabs(xt) < eps;
        for (int a = 0; a < d; a++) {
            vre[a] = le * bfd(ve[a]) + lc * bfd(vc[a]);
            kre[a] = gd ? 0.5 * (bfd(ke[a]) + bfd(kc[a]))
                        : (le * bfd(ke[a]) + lc * bfd(kc[a])) * ell / xt;
        }
        if (kr) memcpy(&kr[(size_t)u * d], kre, d * sizeof(double));
        if (vr) memcpy(&vr[(size_t)u * d], vre, d * sizeof(double));
        if (guard) guard[u] = gd;
        if (xt_out) xt_out[u] = xt;
        if (partner) partner[u] = s->pos[base + c];
        uint16_t *kcw = &s->k[(base + c) * d], *vcw = &s->v[(base + c) * d];
        for (int a = 0; a < d; a++) {
            kcw[a] = dbf(kre[a]);
            vcw[a] = dbf(vre[a]);
        }
        s->vote[base + c] = s->vote[base + e] + s->vote[base + c];
        if (s->scored[base + c]) s->util[base + c] += s->util[base + e];
        /* remove the victim, keeping position order */
        for (int i = e; i + 1 < n; i++) {
            s->pos[base + i] = s->pos[base + i + 1];
            s->vote[base + i] = s->vote[base + i + 1];
            s->util[base + i] = s->util[base + i + 1];
            s->scored[base + i] = s->scored[base + i + 1];
            memmove(&s->k[(base + i) * d], &s->k[(base + i + 1) * d], d * sizeof(uint16_t));
            memmove(&s->v[(base + i) * d], &s->v[(base + i + 1) * d], d * sizeof(uint16_t));
        }
        s->n[u] = n - 1;
    }
    free(kre);
    free(vre);
    return rc;
}

/*
 * Overwrite the key and value of the slot holding position p in unit u
 * (test support: the parity driver lets the oracle adopt a row the GPU
 * rounded differently within one bf16 unit).  Returns 0, or -1 if absent.
 */
int ocl_set_row(void *h, int u, int32_t p, const uint16_t *k, const uint16_t *v)
{
    ocl_session *s = (ocl_session *)h;
    size_t base = (size_t)u * s->cap;
    for (int i = 0; i < s->n[u]; i++)
        if (s->pos[base + i] == p) {
            memcpy(&s->k[(base + i) * s->d], k, s->d * sizeof(uint16_t));
            memcpy(&s->v[(base + i) * s->d], v, s->d * sizeof(uint16_t));
            return 0;
        }
    return -1;
}

/*
 * Copy out the key and value rows of every live slot, in slot (position)
 * order: k, v [U][cap][d] bf16 bits.
 */
void ocl_get_rows(void *h, uint16_t *k, uint16_t *v)
{
    ocl_session *s = (ocl_session *)h;
    size_t rows = (size_t)s->U * s->cap * s->d;
    memcpy(k, s->k, rows * sizeof(uint16_t));
    memcpy(v, s->v, rows * sizeof(uint16_t));
}

/*
 * Moments in mean / covariance form, recovered from the raw sums
 * [MomentKV sec 4.1 and App. A.1: k_bar = s_k / n_e, v_bar = s_v / n_e,
 *  S_tilde = S - s_v s_k^T / n_e]; C = S_tilde / n_e (the population
 * value-key covariance, C[a][b] = cov(v_a, k_b)).  All zero when n_e = 0.
 */
void ocl_moments(void *h, double *n, double *mu_k, double *mu_v, double *C)
{
    ocl_session *s = (ocl_session *)h;
    int d = s->d;
    for (int u = 0; u < s->U; u++) {
        double ne = s->ne[u];
        const double *sk = &s->sk[(size_t)u * d], *sv = &s->sv[(size_t)u * d];
        const double *S = &s->S[(size_t)u * d * d];
        if (n) n[u] = ne;
        for (int a = 0; a < d; a++) {
            if (mu_k) mu_k[(size_t)u * d + a] = ne > 0 ? sk[a] / ne : 0.0;
            if (mu_v) mu_v[(size_t)u * d + a] = ne > 0 ? sv[a] / ne : 0.0;
        }
        if (C)
            for (int a = 0; a < d; a++)
                for (int b = 0; b < d; b++)
                    C[(size_t)u * d * d + (size_t)a * d + b] =
                        ne > 0 ? (S[(size_t)a * d + b] - sv[a] * sk[b] / ne) / ne : 0.0;
    }
}

/*
 * Output of the decode step after eviction [MomentKV Algorithm 1,
 * normalization-corrected inference phase]:
 *   f_R, Z_R  = attention over the retained slots, computed directly
 *               (logZ_R = log Z_R with vote weights)
 *   n_e = 0 or correction off:  o = f_R
 *   otherwise, from the raw sums:
 *     k_bar = s_k/n_e, v_bar = s_v/n_e, S_tilde = S - s_v s_k^T / n_e
 *     log Zhat_E = ln n_e + q . k_bar / sqrt(d)    Jensen lower bound
 *                                                 (sec 4.2 eq 10)
 *     fhat_E = v_bar + S_tilde q / (n_e sqrt(d))   first order (sec 4.1 eq 9)
 *            = v_bar                               zero order (sec A4,
 *                                                 Table 4 zero-order variant)
 *     w_R = Z_R / (Z_R + Zhat_E) evaluated as 1 / (1 + exp(log Zhat_E -
 *           log Z_R)), the log-domain form of App. C.2
 *     o = w_R f_R + (1 - w_R) fhat_E                (sec 4.2 eq 12)
 * correction: 0 off, 1 zero order, 2 first order.
 * Outputs: o, f_R [U][G][d]; logZ_R [U][G]  (f_R / logZ_R may be NULL).
 */
void ocl_output(void *h, const uint16_t *q, int correction, double *o,
                double *fR, double *logZR)
{
    ocl_session *s = (ocl_session *)h;
    int G = s->G, d = s->d;
    double rsd = 1.0 / sqrt((double)d);
    double *lse = (double *)malloc((size_t)s->U * G * sizeof(double));
    double *f = (double *)malloc((size_t)s->U * G * d * sizeof(double));
    ocl_attend(h, q, lse, f, NULL);
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < s->U; u++) {
        double ne = s->ne[u];
        const double *sk = &s->sk[(size_t)u * d], *sv = &s->sv[(size_t)u * d];
        const double *S = &s->S[(size_t)u * d * d];
        for (int hh = 0; hh < G; hh++) {
            size_t uh = (size_t)u * G + hh;
            const uint16_t *qh = &q[uh * d];
            const double *fr = &f[uh * d];
            double *oh = &o[uh * d];
            if (fR) memcpy(&fR[uh * d], fr, d * sizeof(double));
            if (logZR) logZR[uh] = lse[uh];
            if (ne <= 0.0 || correction == 0) {
                for (int a = 0; a < d; a++) oh[a] = fr[a];
                continue;
            }
            double qk = 0.0;
            for (int b = 0; b < d; b++) qk += bfd(qh[b]) * (sk[b] / ne);
            double logZE = log(ne) + qk * rsd;
            double wR = 1.0 / (1.0 + exp(logZE - lse[uh]));
            for (int a = 0; a < d; a++) {
                double fe = sv[a] / ne;
                if (correction == 2) {
                    double st = 0.0;
                    for (int b = 0; b < d; b++)
                        st += (S[(size_t)a * d + b] - sv[a] * sk[b] / ne) * bfd(qh[b]);
                    fe += st / (ne * sqrt((double)d));
                }
                oh[a] = wR * fr[a] + (1.0 - wR) * fe;
            }
        }
    }
    free(lse);
    free(f);
}

/* ------------------------------------------------------------------ */
/* LaProx prefill scorer                                               */
/* ------------------------------------------------------------------ */

/*
 * Per-group Gram matrix of the output projection.  The MHA output splits as
 * sum_h A^h (V^h W_O^h) [LaProx key design 1]; with the GQA group mean of
 * the attention standing in for every A^h of the group [LaProx
 * "training-free" paragraph], the group's product is A_bar (V_g W_g) with
 * W_g = sum over the group's query heads h of W_O^h, W_O^h being rows
 * [h d, (h+1) d) of W_O (a reading: the page is silent on GQA slicing).
 * Gram[l][g] = W_g W_g^T (d x d), so that ||v W_g||^2 = v^T Gram v.
 * Query head h belongs to KV group h / (Hq / Hkv).
 * W_O: [NL][Hq*d][D] bf16; Gram: [NL][Hkv][d][d] double.
 */
void ocl_prefill_gram(int NL, int Hq, int Hkv, int d, int D,
                      const uint16_t *W_O, double *Gram)
{
    int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int l = 0; l < NL; l++)
        for (int g = 0; g < Hkv; g++) {
            double *W = (double *)calloc((size_t)d * D, sizeof(double));
            for (int hh = g * G; hh < (g + 1) * G; hh++)
                for (int a = 0; a < d; a++) {
                    const uint16_t *row = &W_O[((size_t)l * Hq * d + (size_t)hh * d + a) * D];
                    for (int c = 0; c < D; c++) W[(size_t)a * D + c] += bfd(row[c]);
                }
            double *Gm = &Gram[((size_t)l * Hkv + g) * d * d];
            for (int a = 0; a < d; a++)
                for (int b = 0; b < d; b++) {
                    double acc = 0.0;
                    for (int c = 0; c < D; c++)
                        acc += W[(size_t)a * D + c] * W[(size_t)b * D + c];
                    Gm[(size_t)a * d + b] = acc;
                }
            free(W);
        }
}

/*
 * Column norm of the group-mean window attention [LaProx key design 1 and
 * the GQA group-mean paragraph; SnapKV-style observation window of w
 * queries, MomentKV sec A4]:
 *   window query j (0..w-1) sits at position N - w + j and sees keys
 *   0..N-w+j (causal);  A^h[j,i] = softmax_i(q_hj . k_i / sqrt(d));
 *   A_bar[j,i] = (1/G) sum_{h in group} A^h[j,i];   c_i = ||A_bar[:,i]||_2.
 * q_win: [NL][Hq][w][d]; K: [NL][Hkv][N][d]; c: [NL][Hkv][N].
 */
void ocl_prefill_colnorm(int NL, int Hq, int Hkv, int d, int N, int w,
                         const uint16_t *q_win, const uint16_t *K, double *c)
{
    int G = Hq / Hkv;
    double rsd = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int l = 0; l < NL; l++)
        for (int g = 0; g < Hkv; g++) {
            const uint16_t *Kg = &K[((size_t)l * Hkv + g) * N * d];
            double *Abar = (double *)calloc((size_t)w * N, sizeof(double));
            double *x = (double *)malloc((size_t)N * sizeof(double));
            for (int hh = g * G; hh < (g + 1) * G; hh++)
                for (int j = 0; j < w; j++) {
                    const uint16_t *qj = &q_win[(((size_t)l * Hq + hh) * w + j) * d];
                    int last = N - w + j;           /* last visible key */
                    double mx = -INFINITY;
                    for (int i = 0; i <= last; i++) {
                        double dot = 0.0;
                        for (int a = 0; a < d; a++)
                            dot += bfd(qj[a]) * bfd(Kg[(size_t)i * d + a]);
                        x[i] = dot * rsd;
                        if (x[i] > mx) mx = x[i];
                    }
                    double z = 0.0;
                    for (int i = 0; i <= last; i++) z += exp(x[i] - mx);
                    for (int i = 0; i <= last; i++)
                        Abar[(size_t)j * N + i] += exp(x[i] - mx) / z / (double)G;
                }
            double *cg = &c[((size_t)l * Hkv + g) * N];
            for (int i = 0; i < N; i++) {
                double ss = 0.0;
                for (int j = 0; j < w; j++)
                    ss += Abar[(size_t)j * N + i] * Abar[(size_t)j * N + i];
                cg[i] = sqrt(ss);
            }
            free(Abar);
            free(x);
        }
}

/*
 * Weighted column sum of the group-mean window attention: with the causal
 * window attention of the LaProx column norm (query j of w at position
 * N - w + j sees keys 0..N-w+j; A^h the row softmax of q K^T / sqrt(d);
 * A_bar the mean over the group's G query heads),
 *   S_i = sum_{j=0}^{w-1} roww[j] A_bar[j, i].
 * With roww = 1 this is SnapKV's attention accumulated over the observation
 * window [MomentKV sec A4 setup, "SnapKV prefill protocol"]; with the
 * weights below it is KeepKV's windowed EMA initialization.
 * q_win: [NL][Hq][w][d]; K: [NL][Hkv][N][d]; roww: [w]; S: [NL][Hkv][N].
 */
void ocl_prefill_window_colsum(int NL, int Hq, int Hkv, int d, int N, int w,
                               const double *roww, const uint16_t *q_win,
                               const uint16_t *K, double *S)
{
    int G = Hq / Hkv;
    double rsd = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int l = 0; l < NL; l++)
        for (int g = 0; g < Hkv; g++) {
            const uint16_t *Kg = &K[((size_t)l * Hkv + g) * N * d];
            double *Sg = &S[((size_t)l * Hkv + g) * N];
            double *x = (double *)malloc((size_t)N * sizeof(double));
            for (int i = 0; i < N; i++) Sg[i] = 0.0;
            for (int j = 0; j < w; j++) {
                double wj = roww[j];
                int last = N - w + j;
                for (int hh = g * G; hh < (g + 1) * G; hh++) {
                    const uint16_t *qj = &q_win[(((size_t)l * Hq + hh) * w + j) * d];
                    double mx = -INFINITY;
                    for (int i = 0; i <= last; i++) {
                        double dot = 0.0;
                        for (int a = 0; a < d; a++)
                            dot += bfd(qj[a]) * bfd(Kg[(size_t)i * d + a]);
                        x[i] = dot * rsd;
                        if (x[i] > mx) mx = x[i];
                    }
                    double z = 0.0;
                    for (int i = 0; i <= last; i++) z += exp(x[i] - mx);
                    for (int i = 0; i <= last; i++)
                        Sg[i] += wj * exp(x[i] - mx) / z / (double)G;
                }
            }
            free(x);
        }
}

/*
 * KeepKV's windowed EMA initialization of the utilities [KeepKV reading
 * notes, eq 15 at the end of the prefill: S = sum over the last window of
 * queries of (1 - alpha) alpha^(age) s^k]: the weighted column sum above
 * with roww[j] = (1 - alpha) alpha^(w-1-j), the last window query weighing
 * (1 - alpha).
 */
void ocl_prefill_ema_init(int NL, int Hq, int Hkv, int d, int N, int w, double alpha,
                          const uint16_t *q_win, const uint16_t *K, double *S)
{
    double *roww = (double *)malloc((size_t)(w > 0 ? w : 1) * sizeof(double));
    for (int j = 0; j < w; j++) roww[j] = (1.0 - alpha) * pow(alpha, (double)(w - 1 - j));
    ocl_prefill_window_colsum(NL, Hq, Hkv, d, N, w, roww, q_win, K, S);
    free(roww);
}

/*
 * SnapKV's scores under MomentKV's prefill protocol [MomentKV sec A4
 * setup: attention accumulated over the observation window, the first
 * token kept as the attention sink, adjacent tokens merged into blocks of
 * 4 before scoring]: acc is the accumulated window attention [NL][Hkv][N];
 * each block of `pool` consecutive positions [b pool, (b + 1) pool) takes
 * the mean of its tokens' acc and every token of the block that score; with
 * sink != 0 position 0 scores +infinity (always kept).  s: [NL][Hkv][N].
 */
void ocl_snapkv_scores(int NL, int Hkv, int N, int pool, int sink, const double *acc,
                       double *s)
{
    for (size_t u = 0; u < (size_t)NL * Hkv; u++) {
        const double *a = &acc[u * N];
        double *o = &s[u * N];
        for (int b0 = 0; b0 < N; b0 += pool) {
            int b1 = b0 + pool < N ? b0 + pool : N;
            double m = 0.0;
            for (int i = b0; i < b1; i++) m += a[i];
            m /= (double)(b1 - b0);
            for (int i = b0; i < b1; i++) o[i] = m;
        }
        if (sink && N > 0) o[0] = INFINITY;
    }
}

/*
 * Row norm of the projected values through the Gram matrix:
 *   r_i = ||v_i W_g||_2 = sqrt(max(0, v_i^T Gram v_i))  [LaProx key design 1,
 *   ||(V W_O)[i,:]||_2].  V: [NL][Hkv][N][d]; Gram: [NL][Hkv][d][d].
 */
void ocl_prefill_rownorm(int NL, int Hkv, int d, int N, const uint16_t *V,
                         const double *Gram, double *r)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int l = 0; l < NL; l++)
        for (int g = 0; g < Hkv; g++) {
            const double *Gm = &Gram[((size_t)l * Hkv + g) * d * d];
            const uint16_t *Vg = &V[((size_t)l * Hkv + g) * N * d];
            double *vd = (double *)malloc((size_t)d * sizeof(double));
            for (int i = 0; i < N; i++) {
                for (int a = 0; a < d; a++) vd[a] = bfd(Vg[(size_t)i * d + a]);
                double acc = 0.0;
                for (int a = 0; a < d; a++) {
                    double t = 0.0;
                    for (int b = 0; b < d; b++) t += Gm[(size_t)a * d + b] * vd[b];
                    acc += vd[a] * t;
                }
                r[((size_t)l * Hkv + g) * N + i] = sqrt(acc > 0.0 ? acc : 0.0);
            }
            free(vd);
        }
}

/*
 * Direct form ||v_i W_g||_2 for a list of token indices of one (l, g), as a
 * cross-check of the Gram route.  tokens: nt indices; out: nt values.
 */
void ocl_prefill_rownorm_direct(int Hq, int Hkv, int d, int D, int N, int l,
                                int g, const uint16_t *V, const uint16_t *W_O,
                                int nt, const int32_t *tokens, double *out)
{
    int G = Hq / Hkv;
    const uint16_t *Vg = &V[((size_t)l * Hkv + g) * N * d];
    for (int t = 0; t < nt; t++) {
        int i = tokens[t];
        double ss = 0.0;
        for (int c = 0; c < D; c++) {
            double acc = 0.0;
            for (int hh = g * G; hh < (g + 1) * G; hh++)
                for (int a = 0; a < d; a++)
                    acc += bfd(Vg[(size_t)i * d + a]) *
                           bfd(W_O[((size_t)l * Hq * d + (size_t)hh * d + a) * D + c]);
            ss += acc * acc;
        }
        out[t] = sqrt(ss);
    }
}

typedef struct { double s; int64_t flat; } ocl_skey;

static int skey_cmp(const void *a, const void *b)
{
    const ocl_skey *x = (const ocl_skey *)a, *y = (const ocl_skey *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->flat < y->flat) ? -1 : (x->flat > y->flat);
}

/*
 * Indicator, per-layer normalization and top-K selection [LaProx key
 * designs 1-3; the allocation ablation table of the experiments]:
 *   p_{l,g,i} = c_{l,g,i} * r_{l,g,i}
 *   s_{l,g,i} = p_{l,g,i} / sum_{g',i'} p_{l,g',i'}   (normalize != 0;
 *               the layer's heads and tokens flattened together)
 *   alloc 0 (LaProx: head- and layer-flatten): keep the B_total largest s
 *           over all (l, g, i);
 *   alloc 1 (head-flatten only): every layer keeps its B_total / NL largest
 *           s over its heads and tokens;
 *   alloc 2 (uniform per head): every (l, g) keeps its B_total / (NL Hkv)
 *           largest s.
 * Equal scores are kept in ascending flat index (l*Hkv + g)*N + i (a
 * reading; the page does not order ties).  B_total must be a multiple of the
 * number of segments (1, NL or NL*Hkv).
 * Outputs: s [NL][Hkv][N]; keep [NL][Hkv][N] (0/1); counts [NL][Hkv];
 * idx [B_total] kept flat indices in ascending order; thr [segments] = the
 * segment's smallest kept score.  Returns 0, or -1 if B_total or alloc is
 * out of range.
 */
int ocl_prefill_select(int NL, int Hkv, int N, const double *c,
                       const double *r, int normalize, int alloc, int64_t B_total,
                       double *s, uint8_t *keep, int32_t *counts, int64_t *idx,
                       double *thr)
{
    int64_t M = (int64_t)NL * Hkv * N;
    if (B_total < 0 || B_total > M || alloc < 0 || alloc > 2) return -1;
    int64_t nseg = alloc == 0 ? 1 : alloc == 1 ? NL : (int64_t)NL * Hkv;
    if (B_total % nseg != 0) return -1;
    int64_t seg = M / nseg, kseg = B_total / nseg;
    for (int l = 0; l < NL; l++) {
        double sum = 0.0;
        size_t lo = (size_t)l * Hkv * N, hi = lo + (size_t)Hkv * N;
        for (size_t j = lo; j < hi; j++) sum += c[j] * r[j];
        for (size_t j = lo; j < hi; j++)
            s[j] = normalize ? (sum > 0.0 ? c[j] * r[j] / sum : 0.0) : c[j] * r[j];
    }
    memset(keep, 0, (size_t)M);
    ocl_skey *keys = (ocl_skey *)malloc((size_t)seg * sizeof(ocl_skey));
    for (int64_t q = 0; q < nseg; q++) {
        for (int64_t j = 0; j < seg; j++) {
            keys[j].s = s[q * seg + j];
            keys[j].flat = q * seg + j;
        }
        qsort(keys, (size_t)seg, sizeof(ocl_skey), skey_cmp);
        for (int64_t j = 0; j < kseg; j++) keep[keys[j].flat] = 1;
        if (thr) thr[q] = kseg > 0 ? keys[kseg - 1].s : 0.0;
    }
    free(keys);
    int64_t w = 0;
    for (int l = 0; l < NL; l++)
        for (int g = 0; g < Hkv; g++) {
            int32_t cnt = 0;
            for (int i = 0; i < N; i++) {
                int64_t j = ((int64_t)l * Hkv + g) * N + i;
                if (keep[j]) { cnt++; if (idx) idx[w++] = j; }
            }
            counts[l * Hkv + g] = cnt;
        }
    return 0;
}
