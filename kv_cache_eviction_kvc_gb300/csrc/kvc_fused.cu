// kvc_fused.cu -- fused steady-state decode step (placeholder: the general
// five-kernel sequence is used until the fused kernel is enabled).
#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace kvc {

cudaError_t launch_fused_step(const kvc_params &, int, int, const uint16_t *,
                              const uint16_t *, const uint16_t *, const kvc_cache &,
                              const kvc_moments &, float *, double *, int, int32_t *,
                              int32_t *, int32_t *, const DecodeWs &, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace kvc
