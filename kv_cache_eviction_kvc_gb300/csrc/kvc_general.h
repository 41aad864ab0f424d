// kvc_general.h -- host launchers of the general decode step's path for steps
// that remove many slots per unit (the first step over the prompt): the
// tensor-core moment fold, and the retained output taken after compaction.
#pragma once

#include <cuda_runtime.h>

#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace kvc {

// Folds the n_evict[u] victims evict_idx[u][0..n_evict[u]) (slots below
// len[u] of the cache view c, rows of cap slots) into the moments m: one CTA
// per unit, tcgen05 products per 128-victim tile merged in fp32 (Chan's
// pairwise update).  Units with n_evict <= 0 are left as they are; a victim
// list out of range records KVC_ERR_INVALID_ARG, a wait that ran out
// KVC_ERR_TIMEOUT (in status).
// minor_only: only the units where at most half of the len[u] slots go (the
// others take the complement in launch_prompt_pass's retained mode).
cudaError_t launch_fold_tc(const kvc_cache &c, int cap, int U, int kmax, const int32_t *evict_idx,
                           const int32_t *n_evict, const kvc_moments &m, int32_t *status,
                           cudaStream_t st, bool minor_only = false);

// Victims per unit (kmax) from which the moment fold takes the tensor-core
// kernel.
constexpr int kFoldTcMin = 256;

// Steps removing more than this many slots from some unit (max_len - L)
// take the retained output after compaction (the direct pass over the slots
// that stay, as contiguous rows) instead of the per-unit correction pass.
constexpr int kRetainedMin = 16;

// Attention of the group's queries over each unit's len[u] live slots as they
// are (no token appended, no logits or probabilities kept): lse [U][G] and the
// normalized output f [U][G][d].  After compaction the live slots are the
// retained set, so these are log Z_R and f_R.  max_len bounds len over units.
cudaError_t launch_attend_retained(const kvc_params &p, int max_len, const uint16_t *q,
                                   const kvc_cache &c, float *lse, float *f, const DecodeWs &ws,
                                   cudaStream_t st);

// MomentKV's normalization-corrected output from f_R, log Z_R (as given) and
// the moments: o = w_R f_R + (1 - w_R) (mu_v + C q / sqrt(d)) per head.
// With lse_all, f_all and n_evict given, units with n_evict = 0 take those
// instead (the output over every slot: nothing went, or merge mode merged).
cudaError_t launch_correct_retained(const kvc_params &p, const uint16_t *q, const kvc_cache &c,
                                    const float *lse_R, const float *f_R, const kvc_moments &m,
                                    float *o, const DecodeWs &ws, cudaStream_t st,
                                    const float *lse_all = nullptr, const float *f_all = nullptr,
                                    const int32_t *n_evict = nullptr);

// The split-attention merge alone (lse, f and, with probs, the head-mean
// probabilities from the kept logits) over the partials in the workspace.
cudaError_t launch_attend_final(const kvc_params &p, int max_len, const kvc_cache &c, float *lse,
                                float *f, double *probs, const DecodeWs &ws, cudaStream_t st);

// One pass over every live slot of each unit (one CTA per unit, keys and
// values once through a TMA ring): the split attention partials of the
// group's queries (and the logits when want_x) plus the weighted moments of
// the slots on tensor cores.  append: the step's token joins at slot len and
// the moments of all slots go to the workspace.  Otherwise (after the
// victims were compacted away) the retained slots' moments are taken out of
// those and the evicted set's merged into m, for the units where more than
// half of the slots went (n_evict[u] > len[u]).
cudaError_t launch_prompt_pass(const kvc_params &p, int new_pos, int max_len, const uint16_t *q,
                               const uint16_t *k_new, const uint16_t *v_new, const kvc_cache &c,
                               bool append, bool want_x, const int32_t *n_evict,
                               const kvc_moments &m, const DecodeWs &ws, cudaStream_t st);

}  // namespace kvc
