/*
 * kvc.h -- C ABI of libkvc, the GB300 (sm_103a) budgeted-KV decode step and
 * LaProx prefill scorer.
 *
 * Method sources (web pages), cited per entry point:
 *   MomentKV  "MOMENTKV: Closing the Directional Gap in KV Cache Eviction for
 *             Long-Context Inference" (arXiv 2606.01563)
 *   InertiaKV "Key factors of KV cache eviction in aggressive decoding:
 *             temporal aggregation and rank preservation" (arXiv 2609.03515)
 *   KeepKV    "KeepKV: lossless KV cache compression with electoral votes and
 *             zero-perturbation merging" (reading notes, arXiv 2504.09936)
 *   LaProx    "Reformulating KV Cache Eviction Problem for Long-Context LLM
 *             Inference" (arXiv 2605.07234)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - A unit is one (sequence, layer, KV head); units are independent.  The
 *   unit index of sequence b, layer l, KV head g is u = (b*NL + l)*Hkv + g.
 *   G = query heads per KV head (GQA group); query head h of the unit is the
 *   group's h-th head.
 * - bf16 values are passed as uint16_t bit patterns.  Every pointer is a
 *   DEVICE pointer owned by the caller unless stated otherwise; the library
 *   allocates no device memory.  Scratch lives in a caller-allocated
 *   workspace whose size the *_workspace_size functions return.
 * - Every call is asynchronous on the CUDA stream passed as `stream`
 *   (a cudaStream_t; NULL = legacy default stream).  Only
 *   kvc_get_device_status blocks.
 * - Arguments are validated on the host before any launch; a failed check
 *   returns an error code, launches nothing and sets kvc_last_error().
 *   Conditions that only the device can see (a unit whose length does not
 *   fit the caller's bounds) set a status word in the workspace and leave
 *   that unit untouched; kvc_get_device_status reads and clears it.
 * - Errors never trap or abort on the device.
 * - Layouts (row-major, innermost last):
 *     q        [U][G][d]   bf16     query of the current step
 *     k_new    [U][d]      bf16     key of the token appended this step
 *     v_new    [U][d]      bf16
 *     K, V     [U][cap][d] bf16     slot i of unit u at (u*cap + i)*d
 *     votes    [U][cap]    int32    integer vote p_i >= 1, or NULL = all 1
 *     pos      [U][cap]    int32    token position of each slot
 *     util     [U][cap]    fp64     aggregated utility m(i); +inf = never
 *                                   scored (protected from eviction).  fp64
 *                                   keeps the order of utilities far below
 *                                   fp32's range (sharp attention)
 *     len      [U]         int32    slots in use (slots [0, len) are live)
 *     moments  n [U], mu_k [U][d], mu_v [U][d], C [U][d][d]   fp32
 *              C[a][b] = cov(v_a, k_b) over the evicted set (population)
 * - Supported shapes: d = 128, G in {1, 2, 4, 8}.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_VERSION 10100  /* major*10000 + minor*100 + patch */

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

typedef enum {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = 1,  /* a null pointer or a value out of range      */
    KVC_ERR_SHAPE = 2,        /* sizes inconsistent (e.g. len + 1 > cap)     */
    KVC_ERR_CUDA = 3,         /* a CUDA runtime call failed                  */
    KVC_ERR_TIMEOUT = 4,      /* a bounded device wait ran out               */
    KVC_ERR_UNSUPPORTED = 5,  /* shape outside the supported set             */
    KVC_ERR_WORKSPACE = 6     /* workspace missing, misaligned or too small  */
} kvc_status;

enum {
    KVC_RULE_SINGLE = 0,
    KVC_RULE_CUMULATIVE = 1,
    KVC_RULE_EMA = 2,
    KVC_RULE_MI = 3,
    KVC_RULE_EMA_CHAINED = 4   /* InertiaKV's layer-chained EMA: see
                                  kvc_params.chain_layers */
};
enum { KVC_CORR_OFF = 0, KVC_CORR_ZERO_ORDER = 1, KVC_CORR_FIRST_ORDER = 2 };
enum { KVC_ALLOC_GLOBAL = 0, KVC_ALLOC_LAYER = 1, KVC_ALLOC_HEAD = 2 };

/* Method parameters of a decode stream. */
typedef struct {
    int32_t U;               /* units                                        */
    int32_t G;               /* query heads per KV head (1, 2, 4, 8)         */
    int32_t d;               /* head dimension (128)                         */
    int32_t cap;             /* slot capacity per unit (row stride of K, V)  */
    int32_t L;               /* budget: slots kept per unit after a step     */
    int32_t rule;            /* KVC_RULE_*  (InertiaKV sec 3.1 eqs 2-4;
                                KVC_RULE_EMA_CHAINED: see chain_layers;
                                KVC_RULE_MI: MomentKV's moment-informed
                                score, every step, needs T = 1 and
                                merge = 0; see kvc_mi_scores and
                                kvc_mi_evict)                                */
    float alpha;             /* EMA coefficient, 0 <= alpha < 1              */
    int32_t refresh_period;  /* 0 <= T <= L: utilities refresh on step
                                t = 1 and whenever (t - 1) mod T == 0
                                (InertiaKV-Lazy; T = 1 is full refresh);
                                T = 0 refreshes on step 1 only (InertiaKV
                                Score-Free: the step-1 ranking is frozen)    */
    int32_t correction;      /* KVC_CORR_* (MomentKV sec 4.2 eq 12; the zero-
                                order variant of MomentKV Table 4)           */
    int32_t merge;           /* 0: victims are evicted; 1: a unit removing
                                one slot ZIP-merges its victim instead
                                (KeepKV; see kvc_zip_merge); needs votes     */
    int32_t merge_recent;    /* R >= 0: merge partners exclude the last R
                                token positions (KeepKV candidate choice)    */
    const int32_t *budget;   /* NULL, or a DEVICE array [U]: the budget of
                                each unit (1 <= budget[u] <= L; L is then
                                the largest), e.g. the variable per-head
                                budgets a prefill selection hands over
                                (LaProx key design 3, MomentKV's adaptive
                                per-head allocation; kvc_prefill_handoff).
                                A unit outside [1, L] records KVC_ERR_SHAPE
                                and is left untouched.  Wherever the other
                                entry points say L of a unit, they mean
                                budget[u].  The fused steady state runs when
                                max_len == L + 1 and every unit enters at
                                its own budget.                              */
    int32_t chain_layers;    /* KVC_RULE_EMA_CHAINED (InertiaKV sec 1 and sec
                                3.1, the evaluated implementation: one EMA
                                state updated after each layer): units are
                                grouped by sequence, NL = chain_layers layers
                                of Hkv = chain_heads KV heads (u = (b NL + l)
                                Hkv + g; U a multiple of NL Hkv), every unit
                                of a sequence holding the same positions in
                                the same slots.  On a refresh step each
                                slot's utility passes the layers in order,
                                m = alpha m + (1 - alpha) s_l (m = s_l at the
                                first observation), s_l the layer's mean
                                over its Hkv units' probabilities (all H
                                heads), and is stored in every unit; every
                                unit of the sequence evicts the same slots
                                (budget: the sequence's first unit's).  The
                                call sequence runs (no fused kernel).  Other
                                rules ignore both fields.                    */
    int32_t chain_heads;
} kvc_params;

/* Guard of the ZIP-merge key formula: below this |weighted mean logit| the
 * merged key is the plain mean of the two keys (KeepKV reading notes,
 * "numerical stability" item 2, which gives no value). */
#define KVC_ZIP_EPS 1e-3

/* The budgeted cache of every unit (device pointers, caller-owned). */
typedef struct {
    uint16_t *K;
    uint16_t *V;
    int32_t *votes;   /* NULL = every vote is 1 (no vote weighting)        */
    int32_t *pos;
    double *util;
    int32_t *len;
} kvc_cache;

/* Eviction-set moment statistics (device pointers, caller-owned; zero at the
 * start of each generation, MomentKV sec A4 setup). */
typedef struct {
    float *n;      /* [U]       vote-weighted count n_e                    */
    float *mu_k;   /* [U][d]    key mean k_bar                             */
    float *mu_v;   /* [U][d]    value mean v_bar                           */
    float *C;      /* [U][d][d] S_tilde / n_e, C[a][b] = cov(v_a, k_b)     */
} kvc_moments;

/* ------------------------------------------------------------------ */
/* library                                                             */
/* ------------------------------------------------------------------ */

/* KVC_VERSION of the loaded library. */
KVC_API int32_t kvc_version(void);

/* Message of the last failed call on this host thread ("" if none).  The
 * string is owned by the library and valid until the next call on the same
 * thread. */
KVC_API const char *kvc_last_error(void);

/* Static name of a status code. */
KVC_API const char *kvc_status_string(int32_t status);

/* ------------------------------------------------------------------ */
/* decode step                                                          */
/* ------------------------------------------------------------------ */

/* Bytes of workspace the decode entry points need for these parameters
 * (covers every decode call, including a step-1 pass over cap slots).  The
 * same workspace (device memory, 256-byte aligned) must be passed to every
 * call of one decode stream and left untouched between calls: it carries
 * per-step scratch and per-stream state. */
KVC_API size_t kvc_decode_workspace_size(const kvc_params *p);

/* Zero the workspace's persistent state and status word (enqueued on
 * `stream`).  Call once before the first step of a decode stream. */
KVC_API kvc_status kvc_decode_workspace_init(const kvc_params *p, void *ws,
                                     size_t ws_bytes, void *stream);

/* Read and clear the device status word of a workspace (blocks on `stream`).
 * *device_status receives KVC_OK or the first error a kernel recorded. */
KVC_API kvc_status kvc_get_device_status(void *ws, size_t ws_bytes, void *stream,
                                 int32_t *device_status);

/*
 * kvc_decode_attend -- append the step's token, then vote-weighted
 * single-query GQA attention over every slot of every unit.
 *
 * Defined by: MomentKV sec 2 (s_i = q^T k_i / sqrt(d), Z, alpha_i, f) and
 * Algorithm 1 (append before eviction); KeepKV eq 6 / eq 23 (votes, applied as the
 * logit bias ln p_i, KeepKV "integration" item 2); InertiaKV sec 3.1 eq 1
 * (head-mean probability s_t(i), averaged over the G query heads sharing the
 * KV head).
 *
 * For each unit u (n = len[u] on entry):
 *   slot n receives k_new[u], v_new[u], vote 1, position new_pos, utility
 *   +inf (unscored); len[u] becomes n + 1;
 *   x_hi = q_h . k_i / sqrt(d) + ln p_i, i in [0, n];
 *   lse[u][h]  = log sum_i exp(x_hi);
 *   f_all[u][h][:] = sum_i exp(x_hi - lse) v_i;
 *   probs[u][i] = (1/G) sum_h exp(x_hi - lse_h)   (only if probs != NULL).
 * t is the 1-based decode step (only recorded; it does not change the
 * arithmetic).  max_len >= n + 1 for every unit bounds the launch; a unit
 * with n + 1 > max_len or n + 1 > cap is skipped and sets the device status
 * KVC_ERR_SHAPE.
 * Outputs lse [U][G], f_all [U][G][d] fp32 (required), probs [U][cap] fp64
 * (optional; entries past len untouched).  Logits are fp32; the
 * probabilities are formed in fp64 so that values below fp32's range keep
 * their order.
 */
KVC_API kvc_status kvc_decode_attend(const kvc_params *p, int32_t t, int32_t new_pos,
                             int32_t max_len, const uint16_t *q,
                             const uint16_t *k_new, const uint16_t *v_new,
                             const kvc_cache *cache, float *lse, float *f_all,
                             double *probs, void *ws, size_t ws_bytes,
                             void *stream);

/*
 * kvc_aggregate_evict -- temporal utility update and lowest-utility victim
 * selection.
 *
 * Defined by: InertiaKV sec 3.1 eqs 2-4 (single m = s, cumulative
 * m = m + s, EMA m = alpha m + (1 - alpha) s) and "evict the lowest m_t(i)
 * while the cache exceeds the budget"; InertiaKV-Lazy periodic refresh;
 * MomentKV Algorithm 1 phase 1 (argmin loop).
 *
 * On a refresh step (t = 1, or (t - 1) mod T == 0 when T >= 1) every live
 * slot's utility is updated from probs (required then): an unscored slot
 * takes m = s, a scored one the rule.  On other steps utilities are left as they are.
 * Then k = len[u] - L victims (0 if len <= L) are chosen among scored slots:
 * the k smallest (m, pos) pairs, utility ascending, ties to the smaller
 * token position.  evict_idx[u][0..k) receives their slot indices in
 * ascending slot order, evict_pos (optional) their positions in the same
 * order, n_evict[u] = k.  A unit needing more than kmax victims, or with
 * fewer than k scored slots, gets n_evict = 0 and sets the device status
 * (KVC_ERR_SHAPE / KVC_ERR_INVALID_ARG).  Nothing is removed here.
 */
KVC_API kvc_status kvc_aggregate_evict(const kvc_params *p, int32_t t,
                               const double *probs, const kvc_cache *cache,
                               int32_t kmax, int32_t *evict_idx,
                               int32_t *evict_pos, int32_t *n_evict, void *ws,
                               size_t ws_bytes, void *stream);

/*
 * kvc_moment_update -- fold the evicted tokens into the eviction-set
 * moments, each weighted by its vote.
 *
 * Defined by: MomentKV sec 4.1 "efficient statistics update", Algorithm 1
 * eviction phase and App. A.1 (n_e, s_k, s_v, S updated by addition;
 * S_tilde = S - s_v s_k^T / n_e).  The library keeps the equivalent mean /
 * covariance form (n, mu_k, mu_v, C = S_tilde / n) and updates it with the
 * weighted pairwise merge of Chan, Golub and LeVeque (1979), the one-token
 * case being West's (1979) weighted incremental update.  A vote p counts as
 * p identical tokens (KeepKV eq 6).
 * Reads K, V, votes at evict_idx[u][0..n_evict[u]) (before compaction).
 */
KVC_API kvc_status kvc_moment_update(const kvc_params *p, const kvc_cache *cache,
                             int32_t kmax, const int32_t *evict_idx,
                             const int32_t *n_evict, const kvc_moments *mom,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * kvc_correct -- retained-only attention and the moment-based normalization
 * correction.
 *
 * Defined by: MomentKV Algorithm 1 inference phase, sec 4.1 eq 9
 * (fhat_E = v_bar + S_tilde q / (n_e sqrt d)), sec 4.2 eqs 10-12 (Jensen
 * bound Zhat_E = n_e exp(q . k_bar / sqrt d), w_R = Z_R / (Z_R + Zhat_E)),
 * App. C.2 (log-domain weight); KeepKV eq 3 (o' = (o - A_e v_e)/(1 - A_e)),
 * used to obtain the retained-only output from the full pass.
 *
 * Call after kvc_moment_update and before kvc_compact, with lse / f_all from
 * kvc_decode_attend of the same step.  Per unit and head:
 *   f_R, log Z_R over the live slots not in evict_idx: by the eviction-error
 *     identity when at most 16 slots go and their attention mass is <= 0.5,
 *     otherwise by a direct pass over the retained slots;
 *   n = 0 or correction off: o = f_R;
 *   else log Zhat_E = ln n + q . mu_k / sqrt(d),
 *        fhat_E = mu_v + C q / sqrt(d)   (first order) or mu_v (zero order),
 *        w_R = 1 / (1 + exp(log Zhat_E - log Z_R)),
 *        o = w_R f_R + (1 - w_R) fhat_E.
 * Outputs o [U][G][d] fp32 (required), f_R [U][G][d] and logZ_R [U][G]
 * (optional).
 */
KVC_API kvc_status kvc_correct(const kvc_params *p, const uint16_t *q,
                       const kvc_cache *cache, int32_t kmax,
                       const int32_t *evict_idx, const int32_t *n_evict,
                       const float *lse, const float *f_all,
                       const kvc_moments *mom, float *o, float *f_R,
                       float *logZ_R, void *ws, size_t ws_bytes, void *stream);

/*
 * kvc_mi_scores -- MomentKV moment-informed eviction scores.
 *
 * Defined by: MomentKV sec 4.2 ("moment residual", "moment-aware eviction
 * score") and Algorithm 1, phase 1.  For every live slot i < len[u]:
 *   r_i = v_i - mu_v - C (k_i - mu_k) / sqrt(d)   (the moments as they are:
 *         all zero before the first eviction, so r_i = v_i),
 *   scores[u][i] = probs[u][i] * ||r_i||_2,
 * probs being the head-mean probabilities kvc_decode_attend wrote for this
 * step (the slot's attention weight).  scores may alias probs.  With rule
 * KVC_RULE_MI, kvc_aggregate_evict takes these scores as the utilities of
 * every slot (refreshed every step) and evicts the lowest, for steps that
 * remove one slot; a unit removing more (which MomentKV Algorithm 1 does
 * one fold at a time, re-scoring in between) is refused there with device
 * status KVC_ERR_UNSUPPORTED: use kvc_mi_evict.  fp32 residuals (CUDA
 * cores), fp64 scores.  max_len bounds len[u] (<= cap).
 */
KVC_API kvc_status kvc_mi_scores(const kvc_params *p, const kvc_cache *cache,
                                 const kvc_moments *mom, int32_t max_len,
                                 const double *probs, double *scores, void *stream);

/*
 * kvc_mi_evict -- MomentKV's moment-aware eviction phase for a step that
 * removes several slots.
 *
 * Defined by: MomentKV Algorithm 1, phase 1 (while |R| > L: re-form the
 * means and S_tilde from the running statistics, alpha = softmax over R,
 * score(j) = alpha_j ||r_j||, evict the argmin, fold it, remove it), sec 4.2
 * ("moment residual", "moment-aware eviction score"), sec 4.1 "efficient
 * statistics update".
 *
 * Call right after kvc_decode_attend of the same step, with probs requested
 * there: it reads the logits that call left in the workspace, and lse is
 * that call's output.  For each unit with k = len[u] - L > 0, k rounds:
 * alpha_i = (1/G) sum_h exp(x_hi - lse_h) / Z_h with Z_h summed over the
 * slots still present (fp64), r_i = v_i - mu_v - C (k_i - mu_k) / sqrt(d)
 * with the moments as they stand, the lowest alpha_i ||r_i|| goes (ties to
 * the smaller position) and is folded into the moments (weighted by its
 * vote, KeepKV eq 6).  evict_idx / evict_pos (optional) [U][kmax] receive
 * the victims in eviction order, n_evict[u] = k, util[i] the last score of
 * each slot still present.  Nothing is compacted: kvc_correct (whose
 * moments are then already folded: do not call kvc_moment_update) and
 * kvc_compact follow.  Each round re-scores the whole unit (O(len d^2)):
 * max_len <= 8192 and (max_len - L) * max_len <= 2^22, else
 * KVC_ERR_UNSUPPORTED (compress a long prompt first).  kmax >=
 * max_len - L.  fp32 residuals, fp64 weights and scores.
 */
KVC_API kvc_status kvc_mi_evict(const kvc_params *p, int32_t max_len, const kvc_cache *cache,
                                const kvc_moments *mom, const float *lse, int32_t kmax,
                                int32_t *evict_idx, int32_t *evict_pos, int32_t *n_evict,
                                void *ws, size_t ws_bytes, void *stream);

/*
 * kvc_zip_merge -- merge each unit's single victim into its most similar
 * slot instead of evicting it.
 *
 * Defined by: KeepKV reading notes, "ZIP-Merging" (eq 7 votes p_r = p_e +
 * p_c, eq 8 score condition, eq 10 value, eq 12 key, Thm 3 single-step
 * lossless), "why cosine similarity" (partner = most similar key, the most
 * recent R tokens excluded) and "numerical stability" item 2 (guard).
 *
 * Call after kvc_aggregate_evict and before kvc_moment_update, with q and
 * new_pos of the same step; needs cache->votes.  For each unit with
 * n_evict[u] == 1 and victim slot e = evict_idx[u][0]:
 *   candidates c: live slots other than e with pos <= new_pos - R
 *     (R = p->merge_recent); partner = the largest cos(k_e, k_c) (0 when a
 *     key is zero), ties to the smaller position.  No candidate: nothing
 *     happens (the victim is evicted by the calls that follow).
 *   xbar_j = (1/G) sum_h q_h . k_j / sqrt(d) (the group's mean query;
 *     G = 1 is the page's single-head score), w_j = p_j exp(xbar_j),
 *     lambda_j = w_j / (w_e + w_c), xt = lambda_e xbar_e + lambda_c xbar_c,
 *     ell = ln((w_e + w_c) / (p_e + p_c));
 *   v_c := lambda_e v_e + lambda_c v_c;
 *   k_c := (lambda_e k_e + lambda_c k_c) ell / xt, or (k_e + k_c) / 2 when
 *     |xt| < KVC_ZIP_EPS (both rounded to bf16, nearest even);
 *   votes[c] := p_e + p_c; util[c] := util[c] + util[e]; pos[c] kept;
 *   slot e is refilled from slot len - 1 (all fields), len[u] -= 1 and
 *   n_evict[u] := 0, so the moment fold, the correction (which then returns
 *   the output over every slot of the step, as KeepKV attends before it
 *   compresses) and the compaction leave the unit alone.
 * partner_pos [U] (optional) receives the partner's position or -1.
 * Scores and weights are fp32; cosine near-ties (|difference| ~ 1e-6) may
 * resolve either way.
 */
KVC_API kvc_status kvc_zip_merge(const kvc_params *p, int32_t new_pos, const uint16_t *q,
                                 const kvc_cache *cache, int32_t kmax,
                                 const int32_t *evict_idx, int32_t *n_evict,
                                 int32_t *partner_pos, void *ws, size_t ws_bytes,
                                 void *stream);

/*
 * kvc_compact -- remove the evicted slots (MomentKV Algorithm 1, end of the
 * eviction phase).
 * Live slots keep their contents; the slot order is not significant (slots
 * are identified by position).  With n = len - k, every evicted slot below
 * n is filled by a live slot at or above n (both taken in ascending order);
 * K, V, votes, pos and util move together; len[u] = n.
 */
KVC_API kvc_status kvc_compact(const kvc_params *p, const kvc_cache *cache,
                       int32_t kmax, const int32_t *evict_idx,
                       const int32_t *n_evict, void *ws, size_t ws_bytes,
                       void *stream);

/*
 * kvc_decode_step -- the whole decode step, fused: the same results as
 * kvc_decode_attend, kvc_aggregate_evict, kvc_moment_update, kvc_correct and
 * kvc_compact called in that order (same sets; outputs within fp32
 * rounding); with p->merge = 1, kvc_zip_merge runs between
 * kvc_aggregate_evict and kvc_moment_update; with rule KVC_RULE_MI,
 * kvc_mi_scores runs between kvc_decode_attend and kvc_aggregate_evict when
 * one slot goes, and kvc_mi_evict replaces kvc_mi_scores,
 * kvc_aggregate_evict and kvc_moment_update when several go (the call
 * sequence; no fused kernel; evict_idx / evict_pos then in eviction order,
 * and the bounds of kvc_mi_evict apply).
 *
 * In the steady state (max_len == L + 1: every unit enters with len = L and
 * evicts exactly one slot) one cluster kernel per step does everything: the
 * new token is written straight into the victim's slot.  Otherwise (e.g.
 * step 1 over the prefill cache) the five-call sequence runs.
 * probs (optional [U][cap] fp64) receives the head-mean probabilities on refresh
 * steps in the slot order of the step's input (the new token at index
 * len); evict_pos / evict_idx (optional [U][kmax]) the evicted positions /
 * slot indices; n_evict [U] (required) the victim counts; o [U][G][d] the
 * corrected output.
 */
KVC_API kvc_status kvc_decode_step(const kvc_params *p, int32_t t, int32_t new_pos,
                           int32_t max_len, const uint16_t *q,
                           const uint16_t *k_new, const uint16_t *v_new,
                           const kvc_cache *cache, const kvc_moments *mom,
                           float *o, double *probs, int32_t kmax,
                           int32_t *evict_idx, int32_t *evict_pos,
                           int32_t *n_evict, void *ws, size_t ws_bytes,
                           void *stream);

/*
 * kvc_decode_attend_noalloc -- kvc_decode_attend for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point; it exists for hosts that own every device allocation (a serving
 * runtime that reserves its memory pool at start-up and allows no cudaMalloc
 * afterwards, a plugin interface that passes tensors but no workspace).
 *
 * Same arguments, arithmetic, outputs and argument checks (with the same
 * status codes) as kvc_decode_attend, without the workspace: the scratch
 * (status word, logits, split partials, lengths) lives in a static device
 * array of 32 MiB inside the library, which every GPU that loads the library
 * holds until the process exits.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 * - Sizes whose scratch exceeds 32 MiB are rejected with KVC_ERR_WORKSPACE
 *   and a message.  The scratch is about U*ceil(cap/1024)*G*520 bytes, plus
 *   U*G*cap*4 bytes of logits when probs != NULL (the logits are only kept
 *   to form the probabilities).
 * - Each call looks up the array's device address in the calling thread's
 *   current device context (cudaGetSymbolAddress), so a device reset or a
 *   change of context needs nothing from the caller.  The first call on a
 *   device also loads the library's device code there, the 32 MiB array
 *   with it: make that first call before any stream capture, and while
 *   32 MiB of device memory are free (a host that reserves the whole device
 *   for its pool calls once before reserving it, or loads modules eagerly,
 *   CUDA_MODULE_LOADING=EAGER); a load that finds no room returns
 *   KVC_ERR_CUDA.
 * - Every call on a device shares the one array and it keeps the previous
 *   call's contents: calls whose kernels overlap on the GPU race and must be
 *   ordered by the caller (one stream, or events).
 * - device_status (optional device pointer to one int32) receives the device
 *   status of this call (KVC_OK or the KVC_ERR_* a kernel recorded, e.g.
 *   KVC_ERR_SHAPE for a unit with len + 1 > max_len, which is left
 *   untouched).  With device_status = NULL such device-side errors are
 *   discarded: there is no workspace to read them from later.
 */
KVC_API kvc_status kvc_decode_attend_noalloc(const kvc_params *p, int32_t t,
                                             int32_t new_pos, int32_t max_len,
                                             const uint16_t *q, const uint16_t *k_new,
                                             const uint16_t *v_new,
                                             const kvc_cache *cache, float *lse,
                                             float *f_all, double *probs,
                                             int32_t *device_status, void *stream);

/* ------------------------------------------------------------------ */
/* prefill -> decode hand-off                                           */
/* ------------------------------------------------------------------ */

/* Bytes of workspace kvc_prefill_handoff needs for U units of N prompt
 * tokens. */
KVC_API size_t kvc_prefill_handoff_workspace_size(int32_t U, int32_t N);

/*
 * kvc_prefill_handoff -- start a decode stream from a prefill selection.
 *
 * Defined by: LaProx key design 3 (the kept set of a global or per-layer
 * selection gives every (layer, KV head) its own budget) and MomentKV's
 * setup (the prompt is compressed before decoding, sec A4; the moment
 * statistics start at zero at the start of each generation and every
 * evicted token is folded, Algorithm 1 / sec 4.1 "efficient statistics
 * update"); KeepKV eq 15 for the optional initial utilities.
 *
 * keep [U][N] uint8 is the kept mask of a prefill selection (the
 * [NL][Hkv][N] output of kvc_prefill_score / kvc_prefill_snapkv of one
 * sequence is [U][N] with U = NL * Hkv; B sequences stack their masks);
 * K_src, V_src [U][N][d] bf16 are the prompt's keys and values in the same
 * order; votes_src [U][N] int32 or NULL (all 1); util_init [U][N] fp64 or
 * NULL.  For every unit u, with c = the number of kept tokens:
 *   slots [0, c) of cache receive the kept tokens in ascending position
 *     (K, V rows; pos = the token's index i in the prompt; votes (when the
 *     cache has votes) = votes_src or 1; util = util_init[u][i], i.e.
 *     scored, or +inf (unscored) when util_init is NULL); len[u] = c;
 *   the moments are reset and every token not kept is folded into them,
 *     weighted by its vote (the vote-weighted mean / covariance of the
 *     prompt's evicted set);
 *   budget[u] (optional DEVICE output [U]) = max(c, 1): the budget to
 *     decode with (pass it as kvc_params.budget, with L >= every budget).
 *     A unit that kept nothing decodes with budget 1 (every decode step
 *     appends before it evicts); its first step leaves it at length 1, so
 *     that step must not take the fused steady-state path (pass max_len !=
 *     L + 1, e.g. L + 2 when cap allows).
 * p: the decode stream's parameters (U, G, d, cap; budget is not read
 * here).  A unit whose c exceeds cap - 1 records KVC_ERR_SHAPE and gets
 * len 0.  Device memory ws of kvc_prefill_handoff_workspace_size(U, N)
 * bytes (256-byte aligned) carries the evicted lists and a status word
 * (KVC_ERR_* of the call; read it with kvc_get_device_status(ws, ...)).
 */
KVC_API kvc_status kvc_prefill_handoff(const kvc_params *p, int32_t N, const uint8_t *keep,
                                       const uint16_t *K_src, const uint16_t *V_src,
                                       const int32_t *votes_src, const double *util_init,
                                       const kvc_cache *cache, const kvc_moments *mom,
                                       int32_t *budget, void *ws, size_t ws_bytes,
                                       void *stream);

/* ------------------------------------------------------------------ */
/* prefill scorer                                                       */
/* ------------------------------------------------------------------ */

/*
 * kvc_prefill_prepare -- per-group value-norm factors of the output
 * projection, once per weight set.
 *
 * Defined by: LaProx key design 1 (Output = sum_h A^h (V^h W_O^h)) and its
 * GQA group-mean paragraph.  Reading: the group's attention is the mean over
 * its query heads, so the group's product is A_bar V_g W_g with
 * W_g = sum of W_O^h over the group's heads (W_O^h = rows [h d, (h+1) d)).
 * Gram = W_g W_g^T is accumulated in fp64 and factored in fp64 by pivoted
 * Cholesky; R[l][g] (d x d, fp32) satisfies R^T R = Gram, so that
 * ||(V W_g)[i,:]||_2 = ||R v_i||_2 (a sum of squares, free of cancellation).
 * W_O [NL][Hq*d][D] bf16; R [NL][Hkv][d][d] fp32, 16-byte aligned.
 */
KVC_API kvc_status kvc_prefill_prepare(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d,
                               int32_t D, const uint16_t *W_O, float *R,
                               void *stream);

/* Bytes of workspace kvc_prefill_score needs. */
KVC_API size_t kvc_prefill_workspace_size(int32_t NL, int32_t Hkv, int32_t N,
                                  int64_t B_total);

/*
 * kvc_prefill_score -- LaProx indicator, per-layer normalization and one
 * model-wide top-K.
 *
 * Defined by: LaProx key design 1 (p_i = ||A[:,i]||_2 ||(V W_O)[i,:]||_2),
 * key design 2 (s_{l,j} = p_{l,j} / sum_k p_{l,k}), key design 3 (global
 * top-K under B_total), the GQA group-mean attention paragraph; the
 * observation window of the last w prompt queries (SnapKV protocol, MomentKV
 * sec A4).
 *   window query j (0..w-1) sits at position N - w + j and sees keys
 *   0..N-w+j; A^h = row softmax of q K^T / sqrt(d); A_bar = mean over the
 *   group's G heads; c_i = ||A_bar[:, i]||_2; r_i = ||R v_i||_2;
 *   p = c r; s = p / (sum of p over the layer's heads and tokens) when
 *   normalize != 0, else s = p; keep the B_total largest s over all
 *   (l, g, i), equal scores kept in ascending flat index (l*Hkv + g)*N + i.
 * alloc selects the budget allocation of LaProx's ablation table:
 *   KVC_ALLOC_GLOBAL  the above (head- and layer-flatten: LaProx itself);
 *   KVC_ALLOC_LAYER   head-flatten only: each layer keeps its B_total / NL
 *                     largest s over its heads and tokens (Hkv <= 64);
 *   KVC_ALLOC_HEAD    uniform: each (layer, KV head) keeps its
 *                     B_total / (NL Hkv) largest s;
 *   B_total must be a multiple of the number of segments
 *   (KVC_ERR_INVALID_ARG); ties as above; idx stays ascending.
 * q_win [NL][Hq][w][d] bf16 (4-byte aligned), K, V [NL][Hkv][N][d] bf16
 * (16-byte aligned); R from kvc_prefill_prepare.  Outputs: scores
 * [NL][Hkv][N] fp32, keep [NL][Hkv][N] uint8 (0/1), counts [NL][Hkv] int32,
 * idx [B_total] int64 kept flat indices ascending.  Any output except keep
 * may be NULL.  Supported: d = 128, Hq = 4 Hkv, 1 <= w <= min(32, N),
 * NL * Hkv * N + 128 < 2^31 (else KVC_ERR_UNSUPPORTED).  ws: device memory of
 * kvc_prefill_workspace_size bytes, 256-byte aligned (KVC_ERR_WORKSPACE).
 * A kernel wait that ran out (a fault) leaves NaN scores.
 * Streams: the value norms run on a stream the library owns (one per
 * context and device, created on the first call in that context, never
 * destroyed), forked from and joined back into `stream` through events, so
 * every output is ordered on `stream` as usual and a stream capture of
 * `stream` takes both branches.  Calls on different caller streams share
 * that stream and queue there.
 */
KVC_API kvc_status kvc_prefill_score(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d,
                             int32_t N, int32_t w, int64_t B_total,
                             int32_t normalize, int32_t alloc, const uint16_t *q_win,
                             const uint16_t *K, const uint16_t *V,
                             const float *R, float *scores, uint8_t *keep,
                             int32_t *counts, int64_t *idx, void *ws,
                             size_t ws_bytes, void *stream);

/*
 * kvc_prefill_window_attention -- weighted column sums of the group-mean
 * window attention.
 *
 * Defined by: KeepKV reading notes eq 15 at the end of the prefill
 * (S = sum over the last w queries of (1 - alpha) alpha^(age) s^k, the
 * windowed EMA initialization of the utilities: row_weight[j] =
 * (1 - alpha) alpha^(w-1-j)); MomentKV sec A4 setup, SnapKV's prefill
 * protocol (attention accumulated over the observation window:
 * row_weight[j] = 1).  With the window and the causal mask of
 * kvc_prefill_score (query j of w at position N - w + j sees keys
 * 0..N-w+j; A_bar the mean over the group's query heads of the row
 * softmax of q K^T / sqrt(d)):
 *   S[l][g][i] = sum_{j<w} row_weight[j] A_bar[j, i].
 * row_weight: HOST array of w floats.  q_win [NL][Hq][w][d], K
 * [NL][Hkv][N][d] bf16 as in kvc_prefill_score; S [NL][Hkv][N] fp32.
 * Supported: d = 128, Hq = 4 Hkv, 1 <= w <= min(32, N).  ws: device memory
 * of kvc_prefill_workspace_size(NL, Hkv, N, 0) bytes, 256-byte aligned.
 * Tensor cores (tcgen05) for the logits, fp32 probabilities.
 */
KVC_API kvc_status kvc_prefill_window_attention(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d,
                                                int32_t N, int32_t w, const float *row_weight,
                                                const uint16_t *q_win, const uint16_t *K,
                                                float *S, void *ws, size_t ws_bytes,
                                                void *stream);

/*
 * kvc_prefill_snapkv -- the prompt selection of MomentKV's prefill protocol.
 *
 * Defined by: MomentKV sec A4 setup ("SnapKV's prefill protocol": attention
 * scores accumulated over a 32-token observation window at the end of the
 * prompt; the first token kept as the attention sink; adjacent tokens
 * merged into blocks of 4 before scoring; the cache budget allocated
 * adaptively over the heads of a layer from their attention).
 *   acc = kvc_prefill_window_attention with every row weight 1;
 *   scores[l][g][i] = mean of acc over the block of `pool` consecutive
 *     positions holding i ([b pool, (b + 1) pool), the last block ragged);
 *     with sink != 0, scores[l][g][0] = +infinity;
 *   each layer keeps its B_total / NL largest scores over all its KV heads
 *     and tokens (equal scores in ascending flat index).
 * Outputs as kvc_prefill_score (scores [NL][Hkv][N] fp32 optional, keep
 * [NL][Hkv][N] uint8 required, counts [NL][Hkv] and idx [B_total] optional,
 * idx ascending within each layer's slice [l B_total/NL, (l+1) B_total/NL)).
 * B_total must be a multiple of NL (KVC_ERR_INVALID_ARG); 1 <= pool <= 64;
 * Hkv <= 64; other limits and the workspace as kvc_prefill_window_attention.
 */
KVC_API kvc_status kvc_prefill_snapkv(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t N,
                                      int32_t w, int64_t B_total, int32_t pool, int32_t sink,
                                      const uint16_t *q_win, const uint16_t *K, float *scores,
                                      uint8_t *keep, int32_t *counts, int64_t *idx, void *ws,
                                      size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
