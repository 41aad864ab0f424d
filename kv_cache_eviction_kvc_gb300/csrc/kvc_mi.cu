// kvc_mi.cu -- MomentKV moment-informed eviction scores (MomentKV sec 4.2,
// "moment residual" and "moment-aware eviction score"; Algorithm 1, phase 1):
//   r_i = v_i - mu_v - C (k_i - mu_k) / sqrt(d),   score_i = alpha_i ||r_i||,
// with C = S_tilde / n_e the stored value-key covariance of the eviction set
// and alpha_i the slot's attention weight (the head-mean probability the
// attend pass wrote).  While nothing has been evicted the moments are zero
// and r_i = v_i.
//
// One CTA per kMiChunks chunks of 64 slots of a unit (256 threads; C is
// staged once for all of them).  C is staged transposed in
// shared memory (CsT[b][a], fp32) and the chunk's keys transposed and
// centred on mu_k (XsT[b][j]); thread (ty, tx) forms C (k_j - mu_k) for the
// 4 slots 4 ty .. 4 ty + 3 and the 8 output dimensions 4 tx .. 4 tx + 3 and
// 64 + 4 tx .. 64 + 4 tx + 3, so that one step of the contraction takes three
// 16-byte shared-memory loads (conflict-free: a half-warp reads 256
// contiguous bytes of a CsT row, the two halves of a warp two 16-byte pieces
// of an XsT row) for 32 FMAs.  The values then take the keys' place (also
// transposed), and the residual norm is reduced over the 16 lanes of the
// slot's half-warp.  CUDA-core fp32: a 128 x 128 x L contraction per unit
// against a matrix that changes at every eviction.
#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_mi.h"

namespace kvc {

namespace {

constexpr int kMiSlots = 64;              // slots per chunk
constexpr int kMiChunks = 8;              // chunks per CTA (C staged once)
constexpr int kMiThreads = 256;
constexpr size_t kMiSmem = ((size_t)kD * kD + (size_t)kD * kMiSlots + 2 * kD) * sizeof(float);

struct MiArgs {
    const uint16_t *K, *V;    // [U][cap][d]
    const int32_t *len;       // [U]
    const float *mu_k, *mu_v, *C;
    const double *probs;      // [U][cap]
    double *scores;           // [U][cap] (may alias probs)
    int cap;
};

__global__ void __launch_bounds__(kMiThreads, 2) mi_score_kernel(MiArgs a)
{
    extern __shared__ __align__(16) float sm[];
    float *CsT = sm;                              // [kD (b)][kD (a)]
    float *XsT = CsT + kD * kD;                   // [kD][kMiSlots]: k - mu_k, then v
    float *mk = XsT + kD * kMiSlots;              // [kD]
    float *mv = mk + kD;                          // [kD]
    const int u = blockIdx.y, jc0 = blockIdx.x * kMiSlots * kMiChunks;
    const int n = min(a.len[u], a.cap);
    if (jc0 >= n) return;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const size_t ubase = (size_t)u * a.cap;
    const float *Cu = a.C + (size_t)u * kD * kD;
    for (int e = tid; e < kD; e += kMiThreads) {
        mk[e] = a.mu_k[(size_t)u * kD + e];
        mv[e] = a.mu_v[(size_t)u * kD + e];
    }
    // C transposed: lanes run along the row index a, so the stores into
    // CsT[b][a] hit consecutive banks
    for (int e = tid; e < kD * kD / 4; e += kMiThreads) {
        const int row = e % kD, b4 = (e / kD) * 4;
        const float4 c4 = *reinterpret_cast<const float4 *>(Cu + (size_t)row * kD + b4);
        CsT[(b4 + 0) * kD + row] = c4.x;
        CsT[(b4 + 1) * kD + row] = c4.y;
        CsT[(b4 + 2) * kD + row] = c4.z;
        CsT[(b4 + 3) * kD + row] = c4.w;
    }
    for (int j0 = jc0; j0 < min(n, jc0 + kMiSlots * kMiChunks); j0 += kMiSlots) {
    __syncthreads();                              // C staged / the last chunk's values consumed
    const int nj = min(kMiSlots, n - j0);
    // keys of the chunk, centred and transposed (lanes run along the slot)
    for (int e = tid; e < kMiSlots * (kD / 8); e += kMiThreads) {
        const int j = e % kMiSlots, c8 = (e / kMiSlots) * 8;
        float f[8];
        if (j < nj) unpack8(ldg_nc_v4(a.K + (ubase + j0 + j) * kD + c8), f);
        else for (int t = 0; t < 8; t++) f[t] = mk[c8 + t];
        for (int t = 0; t < 8; t++) XsT[(c8 + t) * kMiSlots + j] = f[t] - mk[c8 + t];
    }
    __syncthreads();
    float acc[4][8];
#pragma unroll
    for (int jj = 0; jj < 4; jj++)
#pragma unroll
        for (int i = 0; i < 8; i++) acc[jj][i] = 0.f;
#pragma unroll 4
    for (int b = 0; b < kD; b++) {
        const float4 x = *reinterpret_cast<const float4 *>(XsT + b * kMiSlots + 4 * ty);
        const float4 c0 = *reinterpret_cast<const float4 *>(CsT + b * kD + 4 * tx);
        const float4 c1 = *reinterpret_cast<const float4 *>(CsT + b * kD + 64 + 4 * tx);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int jj = 0; jj < 4; jj++)
#pragma unroll
            for (int i = 0; i < 8; i++) acc[jj][i] = fmaf(cv[i], xv[jj], acc[jj][i]);
    }
    __syncthreads();                              // the keys are consumed
    for (int e = tid; e < kMiSlots * (kD / 8); e += kMiThreads) {
        const int j = e % kMiSlots, c8 = (e / kMiSlots) * 8;
        float f[8];
        if (j < nj) unpack8(ldg_nc_v4(a.V + (ubase + j0 + j) * kD + c8), f);
        else for (int t = 0; t < 8; t++) f[t] = 0.f;
        for (int t = 0; t < 8; t++) XsT[(c8 + t) * kMiSlots + j] = f[t];
    }
    __syncthreads();
    const float rs = rsqrtf((float)kD);
    float rr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int aa = (i < 4 ? 0 : 64) + 4 * tx + (i & 3);
        const float4 v4 = *reinterpret_cast<const float4 *>(XsT + aa * kMiSlots + 4 * ty);
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
            const float r = vv[jj] - mv[aa] - acc[jj][i] * rs;
            rr[jj] = fmaf(r, r, rr[jj]);
        }
    }
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
        float q = rr[jj];
#pragma unroll
        for (int m = 8; m > 0; m >>= 1) q += __shfl_xor_sync(kFull, q, m);
        const int j = 4 * ty + jj;
        if (tx == 0 && j < nj) {
            const size_t i = ubase + j0 + j;
            a.scores[i] = a.probs[i] * sqrt((double)q);
        }
    }
    }                                             // chunks
}

// ============================================================ greedy rounds
//
// MomentKV Algorithm 1, phase 1, for a step that removes k = len - L slots:
// every round re-forms the attention weights over the slots still present
// (per head, the vote-weighted softmax renormalized over R; alpha_i the head
// mean), scores every present slot by alpha_i ||r_i|| with the moments as
// they stand, removes the lowest (ties to the smaller position) and folds it
// into the moments (West's weighted one-token update of the mean /
// covariance form: with n' = n + w, dk = k - mu_k, dv = v - mu_v:
// mu += (w / n') d, C' = (n / n') (C + (w / n') dv dk^T)).
//
// One CTA of 512 threads per unit, the whole loop in one launch.  C lives in
// shared memory with a padded row (stride 129: lanes reading column b of
// rows a = lane + 32 j hit distinct banks); each warp scores one slot at a
// time: the centred key is broadcast from shared memory, lane l forms
// (C (k - mu_k))_a for a = l, l + 32, l + 64, l + 96.  The logits are the
// ones the attend pass left in the workspace (vote bias included), the
// per-head partition functions over R are re-summed in fp64 every round.
// Cost per round O(n d^2): the kernel serves steps with few rounds over
// short caches (the host bounds rounds x slots); long prompts are
// compressed before decoding.

constexpr int kGrThreads = 512;
constexpr int kGrWarps = kGrThreads / 32;
constexpr int kGrStride = kD + 1;
constexpr int kGrMaxSlots = 8192;           // slots per unit (alive bitmap)

struct GreedyArgs {
    const uint16_t *K, *V;
    const int32_t *votes, *pos, *len, *budget;
    double *util;
    float *n, *mu_k, *mu_v, *C;
    const float *xbuf;        // [U][G][cap] logits of the attend pass
    const float *lse;         // [U][G]
    int32_t *evict_idx, *evict_pos, *n_evict, *status;
    int cap, L, kmax;
};

template <int G>
__global__ void __launch_bounds__(kGrThreads, 1) mi_greedy_kernel(GreedyArgs a)
{
    extern __shared__ __align__(16) float gsm[];
    float *Cs = gsm;                                  // [kD][kGrStride]
    float *mk = Cs + kD * kGrStride;                  // [kD]
    float *mv = mk + kD;                              // [kD]
    float *dks = mv + kD;                             // [kGrWarps][kD]
    float *dd = dks + kGrWarps * kD;                  // [2][kD] fold deltas
    uint32_t *alive = reinterpret_cast<uint32_t *>(dd + 2 * kD);   // [kGrMaxSlots / 32]
    double *zred = reinterpret_cast<double *>(alive + kGrMaxSlots / 32);  // [kGrWarps][G]
    double *zs = zred + kGrWarps * G;                 // [G]
    double *wsc = zs + G;                             // [kGrWarps] warp-best score
    int *wpos = reinterpret_cast<int *>(wsc + kGrWarps);   // [kGrWarps]
    int *wslot = wpos + kGrWarps;                     // [kGrWarps]
    int *pick = wslot + kGrWarps;                     // [1]
    float *nsh = reinterpret_cast<float *>(pick + 1); // [1]

    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int n = a.len[u];
    const int Lb = a.budget ? a.budget[u] : a.L;      // this unit's budget
    const int k = n - Lb;
    if (Lb < 1 || Lb > a.L) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    if (k <= 0) {
        if (tid == 0) a.n_evict[u] = 0;
        return;
    }
    if (n > a.cap || n > kGrMaxSlots || k > a.kmax) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    const size_t ubase = (size_t)u * a.cap;
    float *Cu = a.C + (size_t)u * kD * kD;
    for (int e = tid; e < kD * kD; e += kGrThreads) Cs[(e / kD) * kGrStride + (e % kD)] = Cu[e];
    for (int e = tid; e < kD; e += kGrThreads) {
        mk[e] = a.mu_k[(size_t)u * kD + e];
        mv[e] = a.mu_v[(size_t)u * kD + e];
    }
    for (int e = tid; e < kGrMaxSlots / 32; e += kGrThreads) {
        const int lo = e * 32;
        alive[e] = lo >= n ? 0u : (n - lo >= 32 ? 0xffffffffu : ((1u << (n - lo)) - 1u));
    }
    if (tid == 0) nsh[0] = a.n[u];
    float lse[G];
#pragma unroll
    for (int h = 0; h < G; h++) lse[h] = a.lse[(size_t)u * G + h];
    const float *xu = a.xbuf + (size_t)u * G * a.cap;
    const float rs = rsqrtf((float)kD);
    __syncthreads();

    for (int r = 0; r < k; r++) {
        // per-head partition function over the slots present (fp64)
        double z[G];
#pragma unroll
        for (int h = 0; h < G; h++) z[h] = 0.0;
        for (int i = tid; i < n; i += kGrThreads) {
            if (!((alive[i >> 5] >> (i & 31)) & 1u)) continue;
#pragma unroll
            for (int h = 0; h < G; h++) z[h] += exp_wide(xu[(size_t)h * a.cap + i] - lse[h]);
        }
#pragma unroll
        for (int h = 0; h < G; h++) {
            double v = z[h];
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
            if (lane == 0) zred[w * G + h] = v;
        }
        __syncthreads();
        if (tid < G) {
            double v = 0.0;
            for (int j = 0; j < kGrWarps; j++) v += zred[j * G + tid];
            zs[tid] = v;
        }
        __syncthreads();
        double rz[G];
#pragma unroll
        for (int h = 0; h < G; h++) rz[h] = 1.0 / zs[h];

        // scores of the slots present; warp-local lowest (score, position)
        double best = __longlong_as_double(0x7ff0000000000000ll);
        int bpos = 0x7fffffff, bslot = -1;
        float *dk = dks + w * kD;
        for (int i = w; i < n; i += kGrWarps) {
            if (!((alive[i >> 5] >> (i & 31)) & 1u)) continue;
            const uint16_t *kr = a.K + (ubase + i) * kD;
            const uint2 kw = *reinterpret_cast<const uint2 *>(kr + 4 * lane);
            dk[4 * lane + 0] = bf_lo(kw.x) - mk[4 * lane + 0];
            dk[4 * lane + 1] = bf_hi(kw.x) - mk[4 * lane + 1];
            dk[4 * lane + 2] = bf_lo(kw.y) - mk[4 * lane + 2];
            dk[4 * lane + 3] = bf_hi(kw.y) - mk[4 * lane + 3];
            __syncwarp();
            float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
            const float *c0 = Cs + lane * kGrStride;
#pragma unroll 8
            for (int b = 0; b < kD; b++) {
                const float x = dk[b];
                t0 = fmaf(c0[b], x, t0);
                t1 = fmaf(c0[32 * kGrStride + b], x, t1);
                t2 = fmaf(c0[64 * kGrStride + b], x, t2);
                t3 = fmaf(c0[96 * kGrStride + b], x, t3);
            }
            __syncwarp();
            const uint16_t *vr = a.V + (ubase + i) * kD;
            const float r0 = bf2f(vr[lane]) - mv[lane] - t0 * rs;
            const float r1 = bf2f(vr[lane + 32]) - mv[lane + 32] - t1 * rs;
            const float r2 = bf2f(vr[lane + 64]) - mv[lane + 64] - t2 * rs;
            const float r3 = bf2f(vr[lane + 96]) - mv[lane + 96] - t3 * rs;
            const float rr = warp_sum(r0 * r0 + r1 * r1 + r2 * r2 + r3 * r3);
            if (lane == 0) {
                double al = 0.0;
#pragma unroll
                for (int h = 0; h < G; h++) al += exp_wide(xu[(size_t)h * a.cap + i] - lse[h]) * rz[h];
                const double sc = al / G * sqrt((double)rr);
                a.util[ubase + i] = sc;               // the slot's score as its utility
                const int p = a.pos[ubase + i];
                if (sc < best || (sc == best && p < bpos)) { best = sc; bpos = p; bslot = i; }
            }
        }
        if (lane == 0) { wsc[w] = best; wpos[w] = bpos; wslot[w] = bslot; }
        __syncthreads();
        if (tid == 0) {
            int jb = 0;
            for (int j = 1; j < kGrWarps; j++)
                if (wsc[j] < wsc[jb] || (wsc[j] == wsc[jb] && wpos[j] < wpos[jb])) jb = j;
            pick[0] = wslot[jb];
        }
        __syncthreads();
        const int js = pick[0];
        if (js < 0) {                                   // nothing present (cannot happen)
            if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
            return;
        }
        // fold the victim into the moments
        const float wv = a.votes ? (float)a.votes[ubase + js] : 1.f;
        const float n0 = nsh[0], n1 = n0 + wv;
        if (tid < kD) dd[tid] = bf2f(a.K[(ubase + js) * kD + tid]) - mk[tid];
        else if (tid < 2 * kD) dd[tid] = bf2f(a.V[(ubase + js) * kD + tid - kD]) - mv[tid - kD];
        __syncthreads();
        const float f0 = n0 / n1, f1 = wv / n1;
        for (int e = tid; e < kD * kD; e += kGrThreads) {
            const int ra = e / kD, cb = e % kD;
            float *c = &Cs[ra * kGrStride + cb];
            *c = f0 * fmaf(f1 * dd[kD + ra], dd[cb], *c);
        }
        if (tid < kD) mk[tid] = fmaf(f1, dd[tid], mk[tid]);
        else if (tid < 2 * kD) mv[tid - kD] = fmaf(f1, dd[tid], mv[tid - kD]);
        if (tid == 0) {
            nsh[0] = n1;
            alive[js >> 5] &= ~(1u << (js & 31));
            a.evict_idx[(size_t)u * a.kmax + r] = js;
            if (a.evict_pos) a.evict_pos[(size_t)u * a.kmax + r] = a.pos[ubase + js];
        }
        __syncthreads();
    }
    for (int e = tid; e < kD * kD; e += kGrThreads) Cu[e] = Cs[(e / kD) * kGrStride + (e % kD)];
    for (int e = tid; e < kD; e += kGrThreads) {
        a.mu_k[(size_t)u * kD + e] = mk[e];
        a.mu_v[(size_t)u * kD + e] = mv[e];
    }
    if (tid == 0) { a.n[u] = nsh[0]; a.n_evict[u] = k; }
}

template <int G>
constexpr size_t greedy_smem()
{
    return (size_t)(kD * kGrStride + 2 * kD + kGrWarps * kD + 2 * kD) * sizeof(float)
         + (kGrMaxSlots / 32) * sizeof(uint32_t)
         + (size_t)(kGrWarps * G + G + kGrWarps) * sizeof(double)
         + (3 * kGrWarps + 1) * sizeof(int) + sizeof(float);
}

template <int G>
cudaError_t launch_greedy_g(const GreedyArgs &a, int U, cudaStream_t st)
{
    constexpr size_t smem = greedy_smem<G>();
    cudaError_t e = cudaFuncSetAttribute(mi_greedy_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mi_greedy_kernel<G><<<U, kGrThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mi_greedy(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             const float *xbuf, const float *lse, int kmax, int32_t *evict_idx,
                             int32_t *evict_pos, int32_t *n_evict, int32_t *status,
                             cudaStream_t st)
{
    GreedyArgs a{c.K, c.V, c.votes, c.pos, c.len, p.budget, c.util, m.n, m.mu_k, m.mu_v, m.C, xbuf, lse,
                 evict_idx, evict_pos, n_evict, status, p.cap, p.L, kmax};
    switch (p.G) {
    case 1: return launch_greedy_g<1>(a, p.U, st);
    case 2: return launch_greedy_g<2>(a, p.U, st);
    case 4: return launch_greedy_g<4>(a, p.U, st);
    case 8: return launch_greedy_g<8>(a, p.U, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mi_scores(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             int max_len, const double *probs, double *scores, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(mi_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMiSmem);
    if (e != cudaSuccess) return e;
    MiArgs a{c.K, c.V, c.len, m.mu_k, m.mu_v, m.C, probs, scores, p.cap};
    const int span = kMiSlots * kMiChunks;
    const dim3 grid((unsigned)((max_len + span - 1) / span), (unsigned)p.U);
    mi_score_kernel<<<grid, kMiThreads, kMiSmem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
