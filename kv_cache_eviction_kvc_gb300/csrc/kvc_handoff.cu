// kvc_handoff.cu -- the prefill-to-decode hand-off: a decode cache built
// from a prefill selection's kept set, with every prompt token that was not
// kept folded into the moment statistics.
//
// LaProx key design 3 gives every (layer, KV head) the share of the global
// budget its tokens won, so units enter decoding with different lengths
// (their budgets); MomentKV starts the moment statistics at zero at the start
// of a generation and folds every evicted token (Algorithm 1, sec 4.1), so
// the prompt's evicted tokens are its first eviction set.
//
// One CTA per unit makes one ordered pass over the unit's N tokens (a block
// scan of the kept flags): a kept token's rank is its slot, a dropped
// token's rank its place in the unit's evicted list.  The moment fold of the
// dropped tokens is the library's batched fold (tiles of 32 victims merged
// by Chan, Golub and LeVeque), run over the prompt arrays.
#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kHoThreads = 512;

struct HandoffArgs {
    const uint8_t *keep;         // [U][N]
    const uint16_t *Ks, *Vs;     // [U][N][d] prompt keys / values
    const int32_t *votes_src;    // [U][N] or NULL
    const double *util_init;     // [U][N] or NULL
    uint16_t *K, *V;             // cache [U][cap][d]
    int32_t *votes, *pos, *len;
    double *util;
    int32_t *budget;             // [U] or NULL
    int32_t *ev, *nev, *srclen;  // workspace: [U][N] dropped tokens, [U] counts, [U] = N
    int32_t *status;
    int N, cap;
};

__global__ void __launch_bounds__(kHoThreads) handoff_kernel(HandoffArgs a)
{
    __shared__ int scan[40];
    __shared__ int carry[1];
    const int u = blockIdx.x, tid = threadIdx.x;
    const size_t sbase = (size_t)u * a.N, cbase = (size_t)u * a.cap;
    const uint8_t *kp = a.keep + sbase;
    // kept count first: a unit that does not fit is refused whole
    int cnt = 0;
    for (int i = tid; i < a.N; i += kHoThreads) cnt += kp[i] != 0;
    int c;
    block_exscan(cnt, scan, &c);
    if (c > a.cap - 1) {
        if (tid == 0) {
            record_status(a.status, KVC_ERR_SHAPE);
            a.len[u] = 0;
            a.nev[u] = 0;
            a.srclen[u] = a.N;
            if (a.budget) a.budget[u] = 1;
        }
        return;
    }
    if (tid == 0) carry[0] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < a.N; i0 += kHoThreads) {
        const int i = i0 + tid;
        const bool in = i < a.N;
        const int k = in && kp[i] != 0;
        int tk;
        const int rk = carry[0] + block_exscan(k, scan, &tk);   // kept tokens before i
        if (in) {
            if (k) {
                const uint4 *ks = reinterpret_cast<const uint4 *>(a.Ks + (sbase + i) * kD);
                const uint4 *vs = reinterpret_cast<const uint4 *>(a.Vs + (sbase + i) * kD);
                uint4 *kd = reinterpret_cast<uint4 *>(a.K + (cbase + rk) * kD);
                uint4 *vd = reinterpret_cast<uint4 *>(a.V + (cbase + rk) * kD);
#pragma unroll
                for (int j = 0; j < kD / 8; j++) kd[j] = ks[j];
#pragma unroll
                for (int j = 0; j < kD / 8; j++) vd[j] = vs[j];
                a.pos[cbase + rk] = i;
                if (a.votes) a.votes[cbase + rk] = a.votes_src ? a.votes_src[sbase + i] : 1;
                a.util[cbase + rk] = a.util_init ? a.util_init[sbase + i]
                                                 : __longlong_as_double(0x7ff0000000000000ll);
            } else {
                // dropped tokens before i: i minus the kept ones before i
                a.ev[sbase + (i - rk)] = i;
            }
        }
        __syncthreads();
        if (tid == 0) carry[0] += tk;
        __syncthreads();
    }
    if (tid == 0) {
        a.len[u] = c;
        a.nev[u] = a.N - c;
        a.srclen[u] = a.N;
        if (a.budget) a.budget[u] = c > 0 ? c : 1;
    }
}

struct HoWs {
    int32_t *status;
    int32_t *ev, *nev, *srclen;
    size_t bytes;
};

HoWs handoff_layout(int U, int N, void *base)
{
    HoWs w{};
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t n) {
        char *p = b ? b + off : nullptr;
        off += align_up(n);
        return p;
    };
    w.status = reinterpret_cast<int32_t *>(take(sizeof(WsHeader)));
    w.ev = reinterpret_cast<int32_t *>(take((size_t)U * N * 4));
    w.nev = reinterpret_cast<int32_t *>(take((size_t)U * 4));
    w.srclen = reinterpret_cast<int32_t *>(take((size_t)U * 4));
    w.bytes = off;
    return w;
}

}  // namespace
}  // namespace kvc

using namespace kvc;

#define HO_CHECK(cond, code, ...)      \
    do {                               \
        if (!(cond)) {                 \
            set_error(__VA_ARGS__);    \
            return (code);             \
        }                              \
    } while (0)

static kvc_status ho_cuda(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return KVC_OK;
    set_error("kvc_prefill_handoff: %s: %s", what, cudaGetErrorString(e));
    return KVC_ERR_CUDA;
}

extern "C" {

size_t kvc_prefill_handoff_workspace_size(int32_t U, int32_t N)
{
    if (U < 1 || N < 1) return 0;
    return handoff_layout(U, N, nullptr).bytes;
}

kvc_status kvc_prefill_handoff(const kvc_params *p, int32_t N, const uint8_t *keep,
                               const uint16_t *K_src, const uint16_t *V_src,
                               const int32_t *votes_src, const double *util_init,
                               const kvc_cache *cache, const kvc_moments *mom, int32_t *budget,
                               void *ws, size_t ws_bytes, void *stream)
{
    kvc_status s = check_params(p);
    if (s == KVC_OK) s = check_cache(cache);
    if (s != KVC_OK) return s;
    HO_CHECK(N >= 1, KVC_ERR_INVALID_ARG, "kvc_prefill_handoff: N = %d must be >= 1", N);
    HO_CHECK((int64_t)p->U * N < (1ll << 31), KVC_ERR_UNSUPPORTED,
             "kvc_prefill_handoff: U * N too large");
    HO_CHECK(keep && K_src && V_src, KVC_ERR_INVALID_ARG,
             "kvc_prefill_handoff: keep, K_src and V_src are required");
    HO_CHECK(((uintptr_t)K_src & 15u) == 0 && ((uintptr_t)V_src & 15u) == 0, KVC_ERR_INVALID_ARG,
             "kvc_prefill_handoff: K_src and V_src must be 16-byte aligned");
    HO_CHECK(((uintptr_t)util_init & 7u) == 0, KVC_ERR_INVALID_ARG,
             "kvc_prefill_handoff: util_init must be 8-byte aligned");
    HO_CHECK(mom && mom->n && mom->mu_k && mom->mu_v && mom->C && ((uintptr_t)mom->C & 15u) == 0,
             KVC_ERR_INVALID_ARG, "kvc_prefill_handoff: moments (C 16-byte aligned) required");
    HoWs w = handoff_layout(p->U, N, nullptr);
    HO_CHECK(ws && ws_bytes >= w.bytes && ((uintptr_t)ws & (kAlign - 1)) == 0, KVC_ERR_WORKSPACE,
             "kvc_prefill_handoff: workspace of %zu bytes (256-byte aligned) required", w.bytes);
    w = handoff_layout(p->U, N, ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    kvc_status r = ho_cuda(cudaMemsetAsync(w.status, 0, sizeof(WsHeader), st), "memset");
    // the moments start from zero: the prompt's dropped tokens are the first
    // eviction set of the generation
    const size_t U = (size_t)p->U;
    if (r == KVC_OK) r = ho_cuda(cudaMemsetAsync(mom->n, 0, U * 4, st), "memset");
    if (r == KVC_OK) r = ho_cuda(cudaMemsetAsync(mom->mu_k, 0, U * kD * 4, st), "memset");
    if (r == KVC_OK) r = ho_cuda(cudaMemsetAsync(mom->mu_v, 0, U * kD * 4, st), "memset");
    if (r == KVC_OK) r = ho_cuda(cudaMemsetAsync(mom->C, 0, U * kD * kD * 4, st), "memset");
    if (r != KVC_OK) return r;
    HandoffArgs a{keep, K_src, V_src, votes_src, util_init, cache->K, cache->V, cache->votes,
                  cache->pos, cache->len, cache->util, budget, w.ev, w.nev, w.srclen, w.status,
                  N, p->cap};
    handoff_kernel<<<p->U, kHoThreads, 0, st>>>(a);
    if ((r = ho_cuda(cudaGetLastError(), "launch")) != KVC_OK) return r;
    // fold the dropped tokens: the batched moment fold over the prompt arrays
    kvc_params ps = *p;
    ps.cap = N;
    const kvc_cache src{const_cast<uint16_t *>(K_src), const_cast<uint16_t *>(V_src),
                        const_cast<int32_t *>(votes_src), nullptr, nullptr, w.srclen};
    DecodeWs dw{};
    dw.status = w.status;
    return ho_cuda(launch_moment(ps, src, N, w.ev, w.nev, *mom, dw, st), "moment fold launch");
}

}  // extern "C"
