// kvc_api.cu -- the extern "C" entry points of libkvc: host-side argument
// validation, workspace carve-up, error reporting and kernel dispatch.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_general.h"
#include "kvc_internal.h"
#include "kvc_mi.h"

namespace kvc {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

DecodeWs decode_ws_layout(const kvc_params &p, void *base)
{
    DecodeWs w{};
    char *b = static_cast<char *>(base);
    size_t off = 0;
    const size_t U = (size_t)p.U, G = (size_t)p.G, cap = (size_t)p.cap;
    const size_t S = (cap + kAttendChunk - 1) / kAttendChunk;
    w.status = reinterpret_cast<int32_t *>(b ? b + off : nullptr);
    off += align_up(sizeof(WsHeader));
    w.xbuf = reinterpret_cast<float *>(b ? b + off : nullptr);
    off += align_up(U * G * cap * sizeof(float));
    w.part = reinterpret_cast<float *>(b ? b + off : nullptr);
    off += align_up(U * S * G * (kD + 2) * sizeof(float));
    w.nlen = reinterpret_cast<int32_t *>(b ? b + off : nullptr);
    off += align_up(U * sizeof(int32_t));
    w.pend = reinterpret_cast<int32_t *>(b ? b + off : nullptr);
    off += align_up(U * kPendStride * sizeof(int32_t));
    w.lse = reinterpret_cast<float *>(b ? b + off : nullptr);
    off += align_up(U * G * sizeof(float));
    w.fall = reinterpret_cast<float *>(b ? b + off : nullptr);
    off += align_up(U * G * kD * sizeof(float));
    w.probs = reinterpret_cast<double *>(b ? b + off : nullptr);
    off += align_up(U * cap * sizeof(double));
    w.pmom = reinterpret_cast<float *>(b ? b + off : nullptr);
    off += align_up(U * (size_t)kPMomStride * sizeof(float));
    w.bytes = off;
    return w;
}

}  // namespace kvc

#define KVC_CHECK_ARG(cond, code, ...)       \
    do {                                     \
        if (!(cond)) {                       \
            set_error(__VA_ARGS__);          \
            return (code);                   \
        }                                    \
    } while (0)

namespace kvc {

static kvc_status cuda_status(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return KVC_OK;
    set_error("%s: %s", what, cudaGetErrorString(e));
    return KVC_ERR_CUDA;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

kvc_status check_params(const kvc_params *p)
{
    KVC_CHECK_ARG(p != nullptr, KVC_ERR_INVALID_ARG, "params is NULL");
    KVC_CHECK_ARG(p->d == kD, KVC_ERR_UNSUPPORTED, "d = %d unsupported (only 128)", p->d);
    KVC_CHECK_ARG(p->G == 1 || p->G == 2 || p->G == 4 || p->G == 8, KVC_ERR_UNSUPPORTED,
                  "G = %d unsupported (1, 2, 4, 8)", p->G);
    KVC_CHECK_ARG(p->U >= 1, KVC_ERR_INVALID_ARG, "U = %d must be >= 1", p->U);
    KVC_CHECK_ARG(p->cap >= 1 && p->cap <= kMaxCap, KVC_ERR_UNSUPPORTED,
                  "cap = %d outside [1, %d]", p->cap, kMaxCap);
    KVC_CHECK_ARG(p->L >= 1 && p->L < p->cap, KVC_ERR_INVALID_ARG,
                  "L = %d must satisfy 1 <= L < cap = %d", p->L, p->cap);
    KVC_CHECK_ARG(p->rule >= KVC_RULE_SINGLE && p->rule <= KVC_RULE_EMA_CHAINED,
                  KVC_ERR_INVALID_ARG, "rule = %d unknown", p->rule);
    KVC_CHECK_ARG(p->rule != KVC_RULE_EMA_CHAINED ||
                      (p->chain_layers >= 1 && p->chain_heads >= 1 &&
                       p->U % (p->chain_layers * p->chain_heads) == 0),
                  KVC_ERR_INVALID_ARG,
                  "the layer-chained EMA needs chain_layers, chain_heads >= 1 dividing U = %d "
                  "(got %d x %d)", p->U, p->chain_layers, p->chain_heads);
    KVC_CHECK_ARG(p->rule != KVC_RULE_EMA_CHAINED || !p->merge, KVC_ERR_INVALID_ARG,
                  "the layer-chained EMA is not combined with merging");
    KVC_CHECK_ARG(p->rule != KVC_RULE_MI || p->refresh_period == 1, KVC_ERR_INVALID_ARG,
                  "the moment-informed rule scores every step: refresh period must be 1");
    KVC_CHECK_ARG((p->rule != KVC_RULE_EMA && p->rule != KVC_RULE_EMA_CHAINED) ||
                      (p->alpha >= 0.f && p->alpha < 1.f),
                  KVC_ERR_INVALID_ARG, "alpha = %g outside [0, 1)", (double)p->alpha);
    KVC_CHECK_ARG(p->refresh_period >= 0 && p->refresh_period <= p->L, KVC_ERR_INVALID_ARG,
                  "refresh period T = %d must satisfy 0 <= T <= L = %d (0 = Score-Free)",
                  p->refresh_period, p->L);
    KVC_CHECK_ARG(p->correction >= KVC_CORR_OFF && p->correction <= KVC_CORR_FIRST_ORDER,
                  KVC_ERR_INVALID_ARG, "correction = %d unknown", p->correction);
    KVC_CHECK_ARG(p->merge == 0 || p->merge == 1, KVC_ERR_INVALID_ARG,
                  "merge = %d must be 0 or 1", p->merge);
    KVC_CHECK_ARG(p->merge_recent >= 0, KVC_ERR_INVALID_ARG,
                  "merge_recent = %d must be >= 0", p->merge_recent);
    KVC_CHECK_ARG(!(p->merge && p->rule == KVC_RULE_MI), KVC_ERR_INVALID_ARG,
                  "the moment-informed rule evicts (and folds); it is not combined with merging");
    return KVC_OK;
}

kvc_status check_cache(const kvc_cache *c)
{
    KVC_CHECK_ARG(c != nullptr, KVC_ERR_INVALID_ARG, "cache is NULL");
    KVC_CHECK_ARG(c->K && c->V && c->pos && c->util && c->len, KVC_ERR_INVALID_ARG,
                  "cache K, V, pos, util and len must be non-NULL");
    KVC_CHECK_ARG(aligned16(c->K) && aligned16(c->V), KVC_ERR_INVALID_ARG,
                  "cache K and V must be 16-byte aligned");
    KVC_CHECK_ARG(((uintptr_t)c->util & 7u) == 0, KVC_ERR_INVALID_ARG,
                  "cache util must be 8-byte aligned");
    return KVC_OK;
}

static kvc_status check_ws(const kvc_params *p, void *ws, size_t bytes, DecodeWs *out)
{
    DecodeWs w = decode_ws_layout(*p, nullptr);
    KVC_CHECK_ARG(ws != nullptr, KVC_ERR_WORKSPACE, "workspace is NULL");
    KVC_CHECK_ARG(((uintptr_t)ws & (kAlign - 1)) == 0, KVC_ERR_WORKSPACE,
                  "workspace must be 256-byte aligned");
    KVC_CHECK_ARG(bytes >= w.bytes, KVC_ERR_WORKSPACE,
                  "workspace has %zu bytes, needs %zu", bytes, w.bytes);
    *out = decode_ws_layout(*p, ws);
    return KVC_OK;
}

static kvc_status check_moments(const kvc_moments *m)
{
    KVC_CHECK_ARG(m != nullptr && m->n && m->mu_k && m->mu_v && m->C, KVC_ERR_INVALID_ARG,
                  "moments and all their arrays must be non-NULL");
    KVC_CHECK_ARG(aligned16(m->C), KVC_ERR_INVALID_ARG, "moments C must be 16-byte aligned");
    return KVC_OK;
}

#define KVC_TRY(expr)                     \
    do {                                  \
        kvc_status _s = (expr);           \
        if (_s != KVC_OK) return _s;      \
    } while (0)

// The greedy moment-aware phase costs O(rounds x slots x d^2): bound it.
static kvc_status check_mi_greedy(const kvc_params *p, int32_t max_len)
{
    const long long rounds = (long long)max_len - p->L;
    KVC_CHECK_ARG(max_len <= kMiGreedyMaxSlots && rounds * max_len <= kMiGreedyMaxWork,
                  KVC_ERR_UNSUPPORTED,
                  "a moment-informed step removing %lld slots from %d takes %lld rounds of "
                  "scoring over the whole cache (MomentKV Algorithm 1); supported up to %d slots "
                  "and %lld rounds x slots: compress the prompt first (e.g. the prefill scorer "
                  "and kvc_prefill_handoff) or take the first step with an attention rule",
                  rounds, max_len, rounds, kMiGreedyMaxSlots, kMiGreedyMaxWork);
    return KVC_OK;
}

kvc_status check_attend_args(const kvc_params *p, int32_t t, int32_t max_len, const uint16_t *q,
                             const uint16_t *k_new, const uint16_t *v_new, const float *lse,
                             const float *f_all)
{
    KVC_CHECK_ARG(t >= 1, KVC_ERR_INVALID_ARG, "step t = %d must be >= 1", t);
    KVC_CHECK_ARG(max_len >= 1 && max_len <= p->cap, KVC_ERR_SHAPE,
                  "max_len = %d must satisfy 1 <= max_len <= cap = %d", max_len, p->cap);
    KVC_CHECK_ARG(q && k_new && v_new && lse && f_all, KVC_ERR_INVALID_ARG,
                  "q, k_new, v_new, lse and f_all must be non-NULL");
    KVC_CHECK_ARG(aligned16(q) && aligned16(k_new) && aligned16(v_new), KVC_ERR_INVALID_ARG,
                  "q, k_new and v_new must be 16-byte aligned");
    return KVC_OK;
}

}  // namespace kvc

using namespace kvc;

extern "C" {

int32_t kvc_version(void) { return KVC_VERSION; }

const char *kvc_last_error(void) { return g_err; }

const char *kvc_status_string(int32_t s)
{
    switch (s) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARG: return "KVC_ERR_INVALID_ARG";
    case KVC_ERR_SHAPE: return "KVC_ERR_SHAPE";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_TIMEOUT: return "KVC_ERR_TIMEOUT";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
    default: return "KVC_ERR_UNKNOWN";
    }
}

size_t kvc_decode_workspace_size(const kvc_params *p)
{
    if (check_params(p) != KVC_OK) return 0;
    return decode_ws_layout(*p, nullptr).bytes;
}

kvc_status kvc_decode_workspace_init(const kvc_params *p, void *ws, size_t ws_bytes,
                                     void *stream)
{
    KVC_TRY(check_params(p));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    KVC_TRY(cuda_status(cudaMemsetAsync(w.status, 0, sizeof(WsHeader), st), "workspace init"));
    KVC_TRY(cuda_status(cudaMemsetAsync(w.pend, 0, (size_t)p->U * kPendStride * sizeof(int32_t), st),
                        "workspace init"));
    return KVC_OK;
}

kvc_status kvc_get_device_status(void *ws, size_t ws_bytes, void *stream, int32_t *device_status)
{
    KVC_CHECK_ARG(ws != nullptr && ws_bytes >= sizeof(WsHeader), KVC_ERR_WORKSPACE,
                  "workspace missing or too small");
    KVC_CHECK_ARG(device_status != nullptr, KVC_ERR_INVALID_ARG, "device_status is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    KVC_TRY(cuda_status(cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st), "status read"));
    KVC_TRY(cuda_status(cudaStreamSynchronize(st), "status read"));
    KVC_TRY(cuda_status(cudaMemsetAsync(ws, 0, sizeof(int32_t), st), "status clear"));
    *device_status = v;
    return KVC_OK;
}

kvc_status kvc_decode_attend(const kvc_params *p, int32_t t, int32_t new_pos, int32_t max_len,
                             const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                             const kvc_cache *cache, float *lse, float *f_all, double *probs,
                             void *ws, size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_TRY(check_attend_args(p, t, max_len, q, k_new, v_new, lse, f_all));
    return cuda_status(launch_attend(*p, t, new_pos, max_len, q, k_new, v_new, *cache, lse, f_all,
                                     probs, w, static_cast<cudaStream_t>(stream)),
                       "kvc_decode_attend launch");
}

kvc_status kvc_aggregate_evict(const kvc_params *p, int32_t t, const double *probs,
                               const kvc_cache *cache, int32_t kmax, int32_t *evict_idx,
                               int32_t *evict_pos, int32_t *n_evict, void *ws, size_t ws_bytes,
                               void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(t >= 1, KVC_ERR_INVALID_ARG, "step t = %d must be >= 1", t);
    KVC_CHECK_ARG(kmax >= 1, KVC_ERR_INVALID_ARG, "kmax = %d must be >= 1", kmax);
    KVC_CHECK_ARG(evict_idx && n_evict, KVC_ERR_INVALID_ARG, "evict_idx and n_evict must be non-NULL");
    KVC_CHECK_ARG(probs || !is_refresh(t, p->refresh_period), KVC_ERR_INVALID_ARG,
                  "probs is required on refresh step t = %d", t);
    return cuda_status(launch_aggregate(*p, t, probs, *cache, kmax, evict_idx, evict_pos, n_evict,
                                        w, static_cast<cudaStream_t>(stream)),
                       "kvc_aggregate_evict launch");
}

kvc_status kvc_moment_update(const kvc_params *p, const kvc_cache *cache, int32_t kmax,
                             const int32_t *evict_idx, const int32_t *n_evict,
                             const kvc_moments *mom, void *ws, size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    KVC_TRY(check_moments(mom));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(kmax >= 1 && evict_idx && n_evict, KVC_ERR_INVALID_ARG,
                  "kmax >= 1, evict_idx and n_evict required");
    return cuda_status(launch_moment(*p, *cache, kmax, evict_idx, n_evict, *mom, w,
                                     static_cast<cudaStream_t>(stream)),
                       "kvc_moment_update launch");
}

kvc_status kvc_correct(const kvc_params *p, const uint16_t *q, const kvc_cache *cache,
                       int32_t kmax, const int32_t *evict_idx, const int32_t *n_evict,
                       const float *lse, const float *f_all, const kvc_moments *mom, float *o,
                       float *f_R, float *logZ_R, void *ws, size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    KVC_TRY(check_moments(mom));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(q && lse && f_all && o, KVC_ERR_INVALID_ARG, "q, lse, f_all and o must be non-NULL");
    KVC_CHECK_ARG(kmax >= 1 && evict_idx && n_evict, KVC_ERR_INVALID_ARG,
                  "kmax >= 1, evict_idx and n_evict required");
    return cuda_status(launch_correct(*p, q, *cache, kmax, evict_idx, n_evict, lse, f_all, *mom, o,
                                      f_R, logZ_R, w, static_cast<cudaStream_t>(stream)),
                       "kvc_correct launch");
}

kvc_status kvc_compact(const kvc_params *p, const kvc_cache *cache, int32_t kmax,
                       const int32_t *evict_idx, const int32_t *n_evict, void *ws,
                       size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(kmax >= 1 && evict_idx && n_evict, KVC_ERR_INVALID_ARG,
                  "kmax >= 1, evict_idx and n_evict required");
    return cuda_status(launch_compact(*p, *cache, kmax, evict_idx, n_evict, w,
                                      static_cast<cudaStream_t>(stream)),
                       "kvc_compact launch");
}

kvc_status kvc_mi_scores(const kvc_params *p, const kvc_cache *cache, const kvc_moments *mom,
                         int32_t max_len, const double *probs, double *scores, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    KVC_TRY(check_moments(mom));
    KVC_CHECK_ARG(probs && scores, KVC_ERR_INVALID_ARG, "probs and scores are required");
    KVC_CHECK_ARG(max_len >= 1 && max_len <= p->cap, KVC_ERR_SHAPE,
                  "max_len = %d must satisfy 1 <= max_len <= cap = %d", max_len, p->cap);
    return cuda_status(launch_mi_scores(*p, *cache, *mom, max_len, probs, scores,
                                        static_cast<cudaStream_t>(stream)),
                       "kvc_mi_scores launch");
}

kvc_status kvc_mi_evict(const kvc_params *p, int32_t max_len, const kvc_cache *cache,
                        const kvc_moments *mom, const float *lse, int32_t kmax,
                        int32_t *evict_idx, int32_t *evict_pos, int32_t *n_evict, void *ws,
                        size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    KVC_TRY(check_moments(mom));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(lse && evict_idx && n_evict, KVC_ERR_INVALID_ARG,
                  "lse, evict_idx and n_evict are required");
    KVC_CHECK_ARG(max_len >= 1 && max_len <= p->cap, KVC_ERR_SHAPE,
                  "max_len = %d must satisfy 1 <= max_len <= cap = %d", max_len, p->cap);
    KVC_CHECK_ARG(kmax >= 1 && kmax >= max_len - p->L, KVC_ERR_SHAPE,
                  "kmax = %d must be >= max(1, max_len - L = %d)", kmax, max_len - p->L);
    KVC_TRY(check_mi_greedy(p, max_len));
    return cuda_status(launch_mi_greedy(*p, *cache, *mom, w.xbuf, lse, kmax, evict_idx, evict_pos,
                                        n_evict, w.status, static_cast<cudaStream_t>(stream)),
                       "kvc_mi_evict launch");
}

kvc_status kvc_zip_merge(const kvc_params *p, int32_t new_pos, const uint16_t *q,
                         const kvc_cache *cache, int32_t kmax, const int32_t *evict_idx,
                         int32_t *n_evict, int32_t *partner_pos, void *ws, size_t ws_bytes,
                         void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(cache->votes != nullptr, KVC_ERR_INVALID_ARG,
                  "kvc_zip_merge needs cache votes (merged slots carry p_e + p_c)");
    KVC_CHECK_ARG(q && evict_idx && n_evict && kmax >= 1, KVC_ERR_INVALID_ARG,
                  "q, evict_idx, n_evict and kmax >= 1 required");
    return cuda_status(launch_zip_merge(*p, new_pos, q, *cache, kmax, evict_idx, n_evict,
                                        partner_pos, w, static_cast<cudaStream_t>(stream)),
                       "kvc_zip_merge launch");
}

kvc_status kvc_decode_step(const kvc_params *p, int32_t t, int32_t new_pos, int32_t max_len,
                           const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                           const kvc_cache *cache, const kvc_moments *mom, float *o,
                           double *probs, int32_t kmax, int32_t *evict_idx, int32_t *evict_pos,
                           int32_t *n_evict, void *ws, size_t ws_bytes, void *stream)
{
    KVC_TRY(check_params(p));
    KVC_TRY(check_cache(cache));
    KVC_TRY(check_moments(mom));
    DecodeWs w;
    KVC_TRY(check_ws(p, ws, ws_bytes, &w));
    KVC_CHECK_ARG(t >= 1, KVC_ERR_INVALID_ARG, "step t = %d must be >= 1", t);
    KVC_CHECK_ARG(max_len >= 1 && max_len <= p->cap, KVC_ERR_SHAPE,
                  "max_len = %d must satisfy 1 <= max_len <= cap = %d", max_len, p->cap);
    KVC_CHECK_ARG(q && k_new && v_new && o && n_evict, KVC_ERR_INVALID_ARG,
                  "q, k_new, v_new, o and n_evict must be non-NULL");
    KVC_CHECK_ARG(aligned16(q) && aligned16(k_new) && aligned16(v_new), KVC_ERR_INVALID_ARG,
                  "q, k_new and v_new must be 16-byte aligned");
    KVC_CHECK_ARG(kmax >= 1 && kmax >= max_len - p->L, KVC_ERR_SHAPE,
                  "kmax = %d must be >= max(1, max_len - L = %d)", kmax, max_len - p->L);
    KVC_CHECK_ARG(!p->merge || cache->votes != nullptr, KVC_ERR_INVALID_ARG,
                  "merge mode needs cache votes (merged slots carry p_e + p_c)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (max_len == p->L + 1 && p->rule != KVC_RULE_EMA_CHAINED) {
        // the moment-informed rule: the residual norms of every slot and the
        // new token first (tensor cores), then the fused step scores
        // alpha ||r|| in its refresh epilogue
        float *rr = nullptr;
        cudaError_t e = cudaSuccess;
        if (p->rule == KVC_RULE_MI) {
            rr = w.xbuf;
            e = launch_mi_norms(*p, *cache, *mom, k_new, v_new, rr, w.status, st);
        }
        if (e == cudaSuccess)
            e = launch_fused_step(*p, t, new_pos, q, k_new, v_new, *cache, *mom, o, probs, kmax,
                                  evict_idx, evict_pos, n_evict, w, st, rr);
        if (e != cudaErrorNotSupported) {
            if (e != cudaSuccess || !p->merge) return cuda_status(e, "kvc_decode_step fused launch");
            // merge mode: the fused kernel attended over every slot, appended
            // the new token and published the victims; the merge follows
            return cuda_status(launch_zip_merge(*p, new_pos, q, *cache, kmax, evict_idx, n_evict,
                                                nullptr, w, st),
                               "kvc_decode_step zip merge");
        }
    }
    // general case: the five-call sequence with workspace scratch
    KVC_CHECK_ARG(evict_idx != nullptr, KVC_ERR_INVALID_ARG,
                  "evict_idx is required when the step is not in the steady state");
    if (p->rule == KVC_RULE_MI && max_len - p->L > 1) KVC_TRY(check_mi_greedy(p, max_len));
    const bool refresh = is_refresh(t, p->refresh_period);
    double *pr = probs ? probs : w.probs;
    // most of every unit goes (the first step over the prompt): one pass
    // gives the attention and the moments of all slots; after compaction a
    // second pass over the retained slots gives f_R, log Z_R and, by the
    // reverse of Chan's update, the evicted set's moments
    if (p->rule != KVC_RULE_MI && max_len - p->L >= kFoldTcMin && 2 * (max_len - p->L) > max_len) {
        cudaError_t e = launch_prompt_pass(*p, new_pos, max_len, q, k_new, v_new, *cache, true,
                                           refresh, nullptr, *mom, w, st);
        if (e != cudaErrorNotSupported) {
            KVC_TRY(cuda_status(e, "kvc_decode_step prompt pass"));
            KVC_TRY(cuda_status(launch_attend_final(*p, max_len, *cache, w.lse, w.fall,
                                                    refresh ? pr : nullptr, w, st),
                                "kvc_decode_step attend merge"));
            KVC_TRY(cuda_status(launch_aggregate(*p, t, pr, *cache, kmax, evict_idx, evict_pos,
                                                 n_evict, w, st),
                                "kvc_decode_step aggregate"));
            if (p->merge) {
                // a unit with a single victim merges it (and then keeps the
                // output over every slot); the others evict
                KVC_TRY(cuda_status(launch_zip_merge(*p, new_pos, q, *cache, kmax, evict_idx, n_evict,
                                                     nullptr, w, st),
                                    "kvc_decode_step zip merge"));
            }
            KVC_TRY(cuda_status(launch_fold_tc(*cache, p->cap, p->U, kmax, evict_idx, n_evict, *mom,
                                               w.status, st, true),
                                "kvc_decode_step moments"));
            KVC_TRY(cuda_status(launch_compact(*p, *cache, kmax, evict_idx, n_evict, w, st),
                                "kvc_decode_step compact"));
            KVC_TRY(cuda_status(launch_prompt_pass(*p, new_pos, p->L, q, nullptr, nullptr, *cache,
                                                   false, false, n_evict, *mom, w, st),
                                "kvc_decode_step retained pass"));
            // the retained pass's lse and output go where the logits were
            // (the probabilities are formed by now; this pass keeps none)
            float *lse_r = w.xbuf;
            float *f_r = w.xbuf + align_up((size_t)p->U * p->G * sizeof(float)) / sizeof(float);
            KVC_TRY(cuda_status(launch_attend_final(*p, p->L, *cache, lse_r, f_r, nullptr, w, st),
                                "kvc_decode_step retained merge"));
            return cuda_status(launch_correct_retained(*p, q, *cache, lse_r, f_r, *mom, o, w, st,
                                                       w.lse, w.fall, n_evict),
                               "kvc_decode_step correct");
        }
    }
    KVC_TRY(cuda_status(launch_attend(*p, t, new_pos, max_len, q, k_new, v_new, *cache, w.lse,
                                      w.fall, refresh ? pr : nullptr, w, st),
                        "kvc_decode_step attend"));
    if (p->rule == KVC_RULE_MI && max_len - p->L > 1) {
        // several slots go: MomentKV Algorithm 1's loop (score, evict the
        // lowest, fold, score again) in one kernel, then the inference phase
        KVC_TRY(cuda_status(launch_mi_greedy(*p, *cache, *mom, w.xbuf, w.lse, kmax, evict_idx,
                                             evict_pos, n_evict, w.status, st),
                            "kvc_decode_step moment-aware eviction"));
        KVC_TRY(cuda_status(launch_correct(*p, q, *cache, kmax, evict_idx, n_evict, w.lse, w.fall,
                                           *mom, o, nullptr, nullptr, w, st),
                            "kvc_decode_step correct"));
        return cuda_status(launch_compact(*p, *cache, kmax, evict_idx, n_evict, w, st),
                           "kvc_decode_step compact");
    }
    if (p->rule == KVC_RULE_MI) {
        // one slot goes: one scoring pass and the argmin, as separate kernels;
        // the scores take the probabilities' place as the aggregate's input
        // (in the workspace; the caller's probs keep the probabilities)
        KVC_TRY(cuda_status(launch_mi_scores(*p, *cache, *mom, max_len, pr, w.probs, st),
                            "kvc_decode_step moment-informed scores"));
        pr = w.probs;
    }
    KVC_TRY(cuda_status(launch_aggregate(*p, t, pr, *cache, kmax, evict_idx, evict_pos, n_evict, w, st),
                        "kvc_decode_step aggregate"));
    if (!p->merge && max_len - p->L > kRetainedMin) {
        // many slots go: fold them, compact, then attend over the slots that
        // stay (contiguous now) for f_R and log Z_R, and correct
        KVC_TRY(cuda_status(launch_moment(*p, *cache, kmax, evict_idx, n_evict, *mom, w, st),
                            "kvc_decode_step moments"));
        KVC_TRY(cuda_status(launch_compact(*p, *cache, kmax, evict_idx, n_evict, w, st),
                            "kvc_decode_step compact"));
        KVC_TRY(cuda_status(launch_attend_retained(*p, p->L, q, *cache, w.lse, w.fall, w, st),
                            "kvc_decode_step retained attention"));
        return cuda_status(launch_correct_retained(*p, q, *cache, w.lse, w.fall, *mom, o, w, st),
                           "kvc_decode_step correct");
    }
    if (p->merge) {
        KVC_TRY(cuda_status(launch_zip_merge(*p, new_pos, q, *cache, kmax, evict_idx, n_evict,
                                             nullptr, w, st),
                            "kvc_decode_step zip merge"));
    }
    KVC_TRY(cuda_status(launch_moment(*p, *cache, kmax, evict_idx, n_evict, *mom, w, st),
                        "kvc_decode_step moments"));
    KVC_TRY(cuda_status(launch_correct(*p, q, *cache, kmax, evict_idx, n_evict, w.lse, w.fall, *mom,
                                       o, nullptr, nullptr, w, st),
                        "kvc_decode_step correct"));
    return cuda_status(launch_compact(*p, *cache, kmax, evict_idx, n_evict, w, st),
                       "kvc_decode_step compact");
}

}  // extern "C"
