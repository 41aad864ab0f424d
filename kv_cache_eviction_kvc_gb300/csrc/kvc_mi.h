// kvc_mi.h -- host launcher of the MomentKV moment-informed score kernel.
#pragma once

#include <cuda_runtime.h>

#include "../../include/kvc.h"

namespace kvc {

// scores[u][i] = probs[u][i] * ||v_i - mu_v - C (k_i - mu_k) / sqrt(d)|| for
// i < len[u]; scores may alias probs.  max_len bounds len over the units.
cudaError_t launch_mi_scores(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             int max_len, const double *probs, double *scores, cudaStream_t st);

// MomentKV Algorithm 1 phase 1 for steps removing k = len - L > 0 slots:
// k rounds of (scores over the slots present, argmin, fold); xbuf / lse are
// the logits and log-partition functions of this step's attend pass.
// evict_idx / evict_pos receive the victims in eviction order, n_evict = k;
// the moments and the utilities (each slot's last score) are updated.
// Units with len > kMiGreedyMaxSlots or k > kmax record KVC_ERR_SHAPE.
constexpr int kMiGreedyMaxSlots = 8192;
// rounds x slots a greedy call may take (host bound: O(rounds n d^2) work)
constexpr long long kMiGreedyMaxWork = 1ll << 22;
cudaError_t launch_mi_greedy(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             const float *xbuf, const float *lse, int kmax, int32_t *evict_idx,
                             int32_t *evict_pos, int32_t *n_evict, int32_t *status,
                             cudaStream_t st);

// ||r_i|| of every live slot i < len[u] of every unit into rr[u][i], and of
// the step's new token (k_new, v_new) into rr[u][len[u]] (fp32): the
// contraction on tensor cores (tcgen05, C as three bf16 terms), the moments
// as they are.  Returns cudaErrorNotSupported when the key tensor map cannot
// be encoded (more than 2^31 rows).
cudaError_t launch_mi_norms(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                            const uint16_t *k_new, const uint16_t *v_new, float *rr,
                            int32_t *status, cudaStream_t st);

}  // namespace kvc
