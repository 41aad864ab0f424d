// kvc_noalloc.cu -- kvc_decode_attend_noalloc: the attention entry point for
// callers that cannot allocate device memory.
//
// Some hosts own every device allocation themselves: an inference server
// that reserves its whole memory pool at start-up and forbids cudaMalloc
// afterwards, or a framework plugin interface that hands the plugin its
// tensors but no workspace.  Such a caller cannot allocate the scratch that
// kvc_decode_attend takes as a workspace.  This variant keeps that scratch in
// a file-scope device array instead: it is part of the library image, so
// every GPU that loads the library holds it (kNoAllocScratchBytes) until the
// process exits, and a call never allocates.
//
// The caller still passes every input and output.  All calls share the one
// array (per device): two calls whose kernels overlap on the GPU race on it
// and must be ordered by the caller (one stream, or events).
#include <mutex>

#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

// Scratch for the split-K partials, per-unit lengths, logits and the status
// word of one attention call.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in; the address a kernel may use
// comes from cudaGetSymbolAddress, resolved once per device with that device
// current (the first call on a device does this set-up).
kvc_status scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("kvc_decode_attend_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error("kvc_decode_attend_noalloc: device %d out of range", dev);
        return KVC_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_error("kvc_decode_attend_noalloc: cudaGetSymbolAddress: %s",
                      cudaGetErrorString(e));
            return KVC_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return KVC_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" KVC_API kvc_status kvc_decode_attend_noalloc(
    const kvc_params *p, int32_t t, int32_t new_pos, int32_t max_len, const uint16_t *q,
    const uint16_t *k_new, const uint16_t *v_new, const kvc_cache *cache, float *lse,
    float *f_all, double *probs, int32_t *device_status, void *stream)
{
    if (p == nullptr || cache == nullptr) {
        set_error("kvc_decode_attend_noalloc: params and cache are required");
        return KVC_ERR_INVALID_ARG;
    }
    // argument checks of kvc_decode_attend, without a workspace
    if (p->d != kD || !(p->G == 1 || p->G == 2 || p->G == 4 || p->G == 8)) {
        set_error("kvc_decode_attend_noalloc: d = %d, G = %d unsupported", p->d, p->G);
        return KVC_ERR_UNSUPPORTED;
    }
    if (p->U < 1 || p->cap < 1 || p->cap > kMaxCap) {
        set_error("kvc_decode_attend_noalloc: U = %d or cap = %d out of range", p->U, p->cap);
        return KVC_ERR_INVALID_ARG;
    }
    if (t < 1 || max_len < 1 || max_len > p->cap) {
        set_error("kvc_decode_attend_noalloc: t = %d or max_len = %d out of range", t, max_len);
        return t < 1 ? KVC_ERR_INVALID_ARG : KVC_ERR_SHAPE;
    }
    if (!cache->K || !cache->V || !cache->pos || !cache->util || !cache->len || !q || !k_new ||
        !v_new || !lse || !f_all) {
        set_error("kvc_decode_attend_noalloc: a required pointer is NULL");
        return KVC_ERR_INVALID_ARG;
    }
    if (!aligned16(cache->K) || !aligned16(cache->V) || !aligned16(q) || !aligned16(k_new) ||
        !aligned16(v_new) || ((uintptr_t)cache->util & 7u)) {
        set_error("kvc_decode_attend_noalloc: K, V, q, k_new, v_new must be 16-byte aligned, "
                  "util 8-byte aligned");
        return KVC_ERR_INVALID_ARG;
    }
    // the attention pass uses the first regions of the decode workspace
    // layout: status word, logits, split partials and per-unit lengths
    void *base = nullptr;
    kvc_status s = scratch_address(&base);
    if (s != KVC_OK) return s;
    DecodeWs w = decode_ws_layout(*p, base);
    const size_t bytes = (size_t)(reinterpret_cast<char *>(w.pend) - static_cast<char *>(base));
    if (bytes > kNoAllocScratchBytes) {
        set_error("kvc_decode_attend_noalloc: U = %d, G = %d, cap = %d need %zu bytes of "
                  "scratch; the static scratch holds %zu bytes (use kvc_decode_attend with a "
                  "workspace)", p->U, p->G, p->cap, bytes, kNoAllocScratchBytes);
        return KVC_ERR_WORKSPACE;
    }
    w.pend = nullptr;        // regions past the attention scratch are not used
    w.lse = nullptr;
    w.fall = nullptr;
    w.probs = nullptr;
    w.bytes = bytes;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the status word must
    // start at zero; every other region is written before it is read
    cudaError_t e = cudaMemsetAsync(w.status, 0, sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = launch_attend(*p, t, new_pos, max_len, q, k_new, v_new, *cache, lse, f_all, probs, w,
                          st);
    if (e == cudaSuccess && device_status)
        e = cudaMemcpyAsync(device_status, w.status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) {
        set_error("kvc_decode_attend_noalloc: %s", cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    return KVC_OK;
}
