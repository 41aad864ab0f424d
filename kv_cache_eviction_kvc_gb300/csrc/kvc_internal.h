// kvc_internal.h -- host-side declarations shared by the libkvc sources.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kAttendChunk = 1024;    // slots per CTA of the split attention
constexpr int kProbsChunk = 4096;     // slots per CTA of the probability pass
constexpr int kMaxCap = 1 << 19;      // largest supported slot capacity
constexpr size_t kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Carve-up of a decode workspace (all offsets 256-byte aligned).
struct DecodeWs {
    int32_t *status;   // WsHeader
    float *xbuf;       // [U][G][cap]         logits of the last attend pass
    float *part;       // [U][S][G][2 + d]    split-K partials (m, l, o)
    int32_t *nlen;     // [U]                 post-append length
    int32_t *pend;     // [U][kPendStride]    fused-step victim queues
    float *lse;        // [U][G]              general-step scratch
    float *fall;       // [U][G][d]           general-step scratch
    double *probs;     // [U][cap]            general-step scratch
    float *pmom;       // [U][kPMomStride]    general-step moments of all slots
    size_t bytes;
};

// one unit's moments in the workspace: M [d][d], mu_k [d], mu_v [d], n
constexpr int kPMomStride = 16768;

constexpr int kPendStride = 72;  // [0] refresh step, [1] count, [2..] slots

DecodeWs decode_ws_layout(const kvc_params &p, void *base);

// thread-local error message
void set_error(const char *fmt, ...);

// host-side argument checks shared by the entry points (each sets the error
// message and returns the status the entry point returns)
kvc_status check_params(const kvc_params *p);
kvc_status check_cache(const kvc_cache *c);
kvc_status check_attend_args(const kvc_params *p, int32_t t, int32_t max_len, const uint16_t *q,
                             const uint16_t *k_new, const uint16_t *v_new, const float *lse,
                             const float *f_all);

// launchers (return cudaError_t of the launch)
cudaError_t launch_attend(const kvc_params &p, int t, int new_pos, int max_len,
                          const uint16_t *q, const uint16_t *k_new,
                          const uint16_t *v_new, const kvc_cache &c,
                          float *lse, float *f_all, double *probs,
                          const DecodeWs &ws, cudaStream_t st);
cudaError_t launch_aggregate(const kvc_params &p, int t, const double *probs,
                             const kvc_cache &c, int kmax, int32_t *evict_idx,
                             int32_t *evict_pos, int32_t *n_evict,
                             const DecodeWs &ws, cudaStream_t st);
cudaError_t launch_moment(const kvc_params &p, const kvc_cache &c, int kmax,
                          const int32_t *evict_idx, const int32_t *n_evict,
                          const kvc_moments &m, const DecodeWs &ws,
                          cudaStream_t st);
cudaError_t launch_correct(const kvc_params &p, const uint16_t *q,
                           const kvc_cache &c, int kmax,
                           const int32_t *evict_idx, const int32_t *n_evict,
                           const float *lse, const float *f_all,
                           const kvc_moments &m, float *o, float *f_R,
                           float *logZ_R, const DecodeWs &ws, cudaStream_t st);
cudaError_t launch_zip_merge(const kvc_params &p, int new_pos, const uint16_t *q,
                             const kvc_cache &c, int kmax, const int32_t *evict_idx,
                             int32_t *n_evict, int32_t *partner_pos, const DecodeWs &ws,
                             cudaStream_t st);
cudaError_t launch_compact(const kvc_params &p, const kvc_cache &c, int kmax,
                           const int32_t *evict_idx, const int32_t *n_evict,
                           const DecodeWs &ws, cudaStream_t st);
cudaError_t launch_fused_step(const kvc_params &p, int t, int new_pos,
                              const uint16_t *q, const uint16_t *k_new,
                              const uint16_t *v_new, const kvc_cache &c,
                              const kvc_moments &m, float *o, double *probs,
                              int kmax, int32_t *evict_idx,
                              int32_t *evict_pos, int32_t *n_evict,
                              const DecodeWs &ws, cudaStream_t st,
                              const float *rr = nullptr);

}  // namespace kvc
