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
#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

// Scratch for the status word, logits, split-K partials and per-unit lengths
// of one attention call.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the calling thread's current
// device context.  In host code the array's name is only a host-side
// stand-in; the address a kernel may use comes from cudaGetSymbolAddress.
// It is looked up on every call (a cheap host-side lookup once the library's
// device code is loaded), so it stays right after a device reset or when
// another context is made current; the first call on a device also loads
// the device code there.
kvc_status scratch_address(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        set_error("kvc_decode_attend_noalloc: cudaGetSymbolAddress: %s",
                  cudaGetErrorString(e));
        return KVC_ERR_CUDA;
    }
    *out = p;
    return KVC_OK;
}

// The regions of the decode workspace that the attention pass uses, packed
// into the static array: the status word, the logits (only written when
// probabilities are wanted), the split partials and the per-unit lengths.
DecodeWs noalloc_layout(const kvc_params &p, char *base, bool want_logits)
{
    const size_t U = (size_t)p.U, G = (size_t)p.G, cap = (size_t)p.cap;
    const size_t S = (cap + kAttendChunk - 1) / kAttendChunk;
    DecodeWs w{};
    size_t off = 0;
    auto at = [&](size_t o) { return base ? base + o : nullptr; };   // sizes only: no base
    w.status = reinterpret_cast<int32_t *>(at(off));
    off += align_up(sizeof(WsHeader));
    if (want_logits) {
        w.xbuf = reinterpret_cast<float *>(at(off));
        off += align_up(U * G * cap * sizeof(float));
    }
    w.part = reinterpret_cast<float *>(at(off));
    off += align_up(U * S * G * (kD + 2) * sizeof(float));
    w.nlen = reinterpret_cast<int32_t *>(at(off));
    off += align_up(U * sizeof(int32_t));
    w.bytes = off;
    return w;
}

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" KVC_API kvc_status kvc_decode_attend_noalloc(
    const kvc_params *p, int32_t t, int32_t new_pos, int32_t max_len, const uint16_t *q,
    const uint16_t *k_new, const uint16_t *v_new, const kvc_cache *cache, float *lse,
    float *f_all, double *probs, int32_t *device_status, void *stream)
{
    // the same checks, in the same order and with the same status codes, as
    // kvc_decode_attend (the workspace checks excepted)
    kvc_status s = check_params(p);
    if (s == KVC_OK) s = check_cache(cache);
    if (s == KVC_OK) s = check_attend_args(p, t, max_len, q, k_new, v_new, lse, f_all);
    if (s != KVC_OK) return s;
    const size_t bytes = noalloc_layout(*p, nullptr, probs != nullptr).bytes;
    if (bytes > kNoAllocScratchBytes) {
        set_error("kvc_decode_attend_noalloc: U = %d, G = %d, cap = %d need %zu bytes of "
                  "scratch; the static scratch holds %zu bytes (use kvc_decode_attend with a "
                  "workspace)", p->U, p->G, p->cap, bytes, kNoAllocScratchBytes);
        return KVC_ERR_WORKSPACE;
    }
    void *base = nullptr;
    s = scratch_address(&base);
    if (s != KVC_OK) return s;
    const DecodeWs w = noalloc_layout(*p, static_cast<char *>(base), probs != nullptr);
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
