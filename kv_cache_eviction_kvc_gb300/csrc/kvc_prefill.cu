// kvc_prefill.cu -- LaProx prefill scorer (not yet enabled).
#include "kvc_common.cuh"
#include "kvc_internal.h"

using namespace kvc;

extern "C" {

kvc_status kvc_prefill_prepare(int32_t, int32_t, int32_t, int32_t, int32_t, const uint16_t *,
                               float *, void *)
{
    set_error("kvc_prefill_prepare: not available in this build");
    return KVC_ERR_UNSUPPORTED;
}

size_t kvc_prefill_workspace_size(int32_t, int32_t, int32_t, int64_t) { return 0; }

kvc_status kvc_prefill_score(int32_t, int32_t, int32_t, int32_t, int32_t, int32_t, int64_t,
                             int32_t, const uint16_t *, const uint16_t *, const uint16_t *,
                             const float *, float *, uint8_t *, int32_t *, int64_t *, void *,
                             size_t, void *)
{
    set_error("kvc_prefill_score: not available in this build");
    return KVC_ERR_UNSUPPORTED;
}

}  // extern "C"
