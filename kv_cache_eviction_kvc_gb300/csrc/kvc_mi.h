// kvc_mi.h -- host launcher of the MomentKV moment-informed score kernel.
#pragma once

#include <cuda_runtime.h>

#include "../../include/kvc.h"

namespace kvc {

// scores[u][i] = probs[u][i] * ||v_i - mu_v - C (k_i - mu_k) / sqrt(d)|| for
// i < len[u]; scores may alias probs.  max_len bounds len over the units.
cudaError_t launch_mi_scores(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             int max_len, const double *probs, double *scores, cudaStream_t st);

}  // namespace kvc
