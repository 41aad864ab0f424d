// kvc_fold.h -- host launcher of the tensor-core moment fold.
#pragma once

#include <cuda_runtime.h>

#include "../../include/kvc.h"

namespace kvc {

// Folds the n_evict[u] victims evict_idx[u][0..n_evict[u]) (slots below
// len[u] of the cache view c, rows of cap slots) into the moments m: one CTA
// per unit, tcgen05 products per 128-victim tile merged in fp32 (Chan's
// pairwise update).  Units with n_evict <= 0 are left as they are; a victim
// list out of range records KVC_ERR_INVALID_ARG, a wait that ran out
// KVC_ERR_TIMEOUT (in status).
cudaError_t launch_fold_tc(const kvc_cache &c, int cap, int U, int kmax, const int32_t *evict_idx,
                           const int32_t *n_evict, const kvc_moments &m, int32_t *status,
                           cudaStream_t st);

// Victims per unit (kmax) from which the moment fold takes the tensor-core
// kernel.
constexpr int kFoldTcMin = 256;

}  // namespace kvc
