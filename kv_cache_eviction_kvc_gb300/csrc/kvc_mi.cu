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

}  // namespace

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
