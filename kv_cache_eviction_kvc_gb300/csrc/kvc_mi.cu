// kvc_mi.cu -- MomentKV moment-informed eviction scores (MomentKV sec 4.2,
// "moment residual" and "moment-aware eviction score"; Algorithm 1, phase 1):
//   r_i = v_i - mu_v - C (k_i - mu_k) / sqrt(d),   score_i = alpha_i ||r_i||,
// with C = S_tilde / n_e the stored value-key covariance of the eviction set
// and alpha_i the slot's attention weight (the head-mean probability the
// attend pass wrote).  While nothing has been evicted the moments are zero
// and r_i = v_i.
//
// One CTA per 64 slots of a unit (256 threads).  C is staged in shared memory
// as fp32 with a padded row stride (129 floats: the 16 lanes of a half-warp
// read 16 rows of one column from 16 banks); the chunk's keys are staged
// centred on mu_k.  Thread (ty, tx) forms C (k_j - mu_k) for 4 slots and 8
// output dimensions (tx + 16 i), so every shared-memory load feeds 2.7 FMAs;
// the values then take the keys' place in shared memory, and the residual
// norm is reduced over the 16 lanes of the slot's half-warp.  CUDA-core
// fp32: this is a 128 x 128 x L contraction per unit against a matrix that
// changes at every eviction.
#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_mi.h"

namespace kvc {

namespace {

constexpr int kMiSlots = 64;              // slots per CTA
constexpr int kMiThreads = 256;
constexpr int kMiLd = kD + 1;             // padded row stride (floats)
constexpr size_t kMiSmem = (size_t)(kD + kMiSlots) * kMiLd * sizeof(float) + 2 * kD * sizeof(float);

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
    extern __shared__ float sm[];
    float *Cs = sm;                               // [kD][kMiLd]
    float *Xs = Cs + kD * kMiLd;                  // [kMiSlots][kMiLd]: k - mu_k, then v
    float *mk = Xs + kMiSlots * kMiLd;            // [kD]
    float *mv = mk + kD;                          // [kD]
    const int u = blockIdx.y, j0 = blockIdx.x * kMiSlots;
    const int n = min(a.len[u], a.cap);
    if (j0 >= n) return;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const size_t ubase = (size_t)u * a.cap;
    const float *Cu = a.C + (size_t)u * kD * kD;
    for (int e = tid; e < kD; e += kMiThreads) {
        mk[e] = a.mu_k[(size_t)u * kD + e];
        mv[e] = a.mu_v[(size_t)u * kD + e];
    }
    for (int e = tid; e < kD * kD / 4; e += kMiThreads) {
        const float4 c4 = reinterpret_cast<const float4 *>(Cu)[e];
        const int r = (4 * e) / kD, col = (4 * e) % kD;
        float *dst = Cs + r * kMiLd + col;
        dst[0] = c4.x; dst[1] = c4.y; dst[2] = c4.z; dst[3] = c4.w;
    }
    __syncthreads();
    const int nj = min(kMiSlots, n - j0);
    // keys of the chunk, centred (8 bf16 per 16-byte load)
    for (int e = tid; e < kMiSlots * (kD / 8); e += kMiThreads) {
        const int j = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
        float f[8];
        if (j < nj) unpack8(ldg_nc_v4(a.K + (ubase + j0 + j) * kD + c8), f);
        else for (int t = 0; t < 8; t++) f[t] = mk[c8 + t];
        for (int t = 0; t < 8; t++) Xs[j * kMiLd + c8 + t] = f[t] - mk[c8 + t];
    }
    __syncthreads();
    float acc[4][8];
#pragma unroll
    for (int jj = 0; jj < 4; jj++)
#pragma unroll
        for (int i = 0; i < 8; i++) acc[jj][i] = 0.f;
#pragma unroll 4
    for (int b = 0; b < kD; b++) {
        float x[4], c[8];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) x[jj] = Xs[(4 * ty + jj) * kMiLd + b];
#pragma unroll
        for (int i = 0; i < 8; i++) c[i] = Cs[(tx + 16 * i) * kMiLd + b];
#pragma unroll
        for (int jj = 0; jj < 4; jj++)
#pragma unroll
            for (int i = 0; i < 8; i++) acc[jj][i] = fmaf(c[i], x[jj], acc[jj][i]);
    }
    __syncthreads();                              // the keys are consumed
    for (int e = tid; e < kMiSlots * (kD / 8); e += kMiThreads) {
        const int j = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
        float f[8];
        if (j < nj) unpack8(ldg_nc_v4(a.V + (ubase + j0 + j) * kD + c8), f);
        else for (int t = 0; t < 8; t++) f[t] = 0.f;
        for (int t = 0; t < 8; t++) Xs[j * kMiLd + c8 + t] = f[t];
    }
    __syncthreads();
    const float rs = rsqrtf((float)kD);
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
        const int j = 4 * ty + jj;
        float rr = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int aa = tx + 16 * i;
            const float r = Xs[j * kMiLd + aa] - mv[aa] - acc[jj][i] * rs;
            rr = fmaf(r, r, rr);
        }
#pragma unroll
        for (int m = 8; m > 0; m >>= 1) rr += __shfl_xor_sync(kFull, rr, m);
        if (tx == 0 && j < nj) {
            const size_t i = ubase + j0 + j;
            a.scores[i] = a.probs[i] * sqrt((double)rr);
        }
    }
}

}  // namespace

cudaError_t launch_mi_scores(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                             int max_len, const double *probs, double *scores, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(mi_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMiSmem);
    if (e != cudaSuccess) return e;
    MiArgs a{c.K, c.V, c.len, m.mu_k, m.mu_v, m.C, probs, scores, p.cap};
    const dim3 grid((unsigned)((max_len + kMiSlots - 1) / kMiSlots), (unsigned)p.U);
    mi_score_kernel<<<grid, kMiThreads, kMiSmem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
