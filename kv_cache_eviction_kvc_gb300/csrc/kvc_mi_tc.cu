// kvc_mi_tc.cu -- MomentKV moment residual norms on the fifth-generation
// tensor cores (MomentKV sec 4.2 "moment residual"; Algorithm 1 phase 1):
//   ||r_i|| = || v_i - mu_v - C (k_i - mu_k) / sqrt(d) ||
// for every live slot i of every unit and for the step's new token, with the
// moments as they enter the step.  The contraction C (k_i - mu_k) is
// D_i - C mu_k with D = K C^T: per 128-slot tile, D (128 slots x 128 dims)
// accumulates in tensor memory from the key tile (bf16, exact) and C split
// into three bf16 terms (hi + mid + lo carry its fp32 value), so the products
// are those of an fp32 contraction.
//
// Persistent: one CTA per SM takes the units blockIdx.x, + gridDim.x, ...
//   warp 0      TMA producer: 128-slot key tiles (two 128-byte-swizzled
//               boxes) into a ring
//   warp 1      tensor-memory owner and MMA issuer (one thread): 3 x 8 MMAs
//               of 128 x 128 x 16 per tile into one of four accumulators
//   warps 2-9   epilogue, two sets of four warps taking alternate tiles; one
//               slot per thread (the warp's tensor-memory lane quarter): D
//               row from tensor memory, the value row from L2 (the producer
//               bulk-prefetches each tile's value rows), ||r||
//   warps 10-13 converter: per unit C (fp32) -> three bf16 operand tiles in
//               shared memory, C mu_k, and the new token's ||r|| on CUDA cores
// Every wait is bounded (~2 s); a wait that ran out records KVC_ERR_TIMEOUT.
#include <cuda_runtime.h>

#include <algorithm>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_mi.h"
#include "kvc_tma.cuh"
#include "kvc_umma.cuh"

namespace kvc {
namespace {

constexpr int kTs = 128;                 // slots per tile
constexpr int kOpB = 2 * kUmmaBox;       // one 128 x 128 bf16 operand: 32 KB
constexpr int kNs = 3;                   // ring stages
constexpr int kNacc = 4;                 // tensor-memory accumulators (128 columns each)
constexpr int kNEpi = 8;                 // epilogue warps: two sets of four
constexpr int kNConv0 = 2 + kNEpi;       // first converter warp
constexpr int kNThreads = (kNConv0 + 4) * 32;
constexpr size_t kNDyn = 1024 + (size_t)3 * kOpB + (size_t)kNs * kOpB;
constexpr uint32_t kNIdesc = umma_idesc_bf16(128, 128);

// Byte offset of 16-byte chunk c (0..15) of row r (0..127) in an operand tile
// (the layout a 128-byte-swizzled TMA load of two 64-column boxes writes).
__device__ __forceinline__ uint32_t op_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kUmmaBox + (r << 7) + (((c & 7) ^ (r & 7)) << 4));
}

struct NormArgs {
    const uint16_t *V;           // [U][cap][d]
    const int32_t *len;          // [U]
    const float *mu_k, *mu_v, *C;
    const uint16_t *k_new, *v_new;   // [U][d]
    float *rr;                   // [U][cap] out: ||r_i||, the new token at index len[u]
    int32_t *status;
    int U, cap;
    float rs;                    // 1 / sqrt(d)
};

struct NormSmem {
    uint64_t full[kNs], empty[kNs];
    uint64_t accf[kNacc], acce[kNacc];
    uint64_t cfull[2];           // the unit's C terms, C mu_k, mu_v are in place (converter)
    uint64_t cfree;              // every MMA of the previous unit completed (MMA commit)
    uint64_t cdone[2];           // the epilogue finished the unit that used the buffer
    float cmu[2][kD];            // C mu_k of the unit (parity)
    float mv[2][kD];             // mu_v of the unit (parity)
    float red[4];
    uint32_t tmem;
    int bad;
};

__device__ __forceinline__ void proxy_fence_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kNThreads, 1)
mi_norm_kernel(NormArgs a, const __grid_constant__ CUtensorMap tmK)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    __shared__ __align__(16) NormSmem S;
    extern __shared__ __align__(1024) unsigned char dyn[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    unsigned char *ring = sm + 3 * kOpB;
    const uint32_t c_s = smem_u32(sm), ring_s = smem_u32(ring);
    const int nmine = blockIdx.x < a.U ? (a.U - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto unit_of = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };
    auto tiles_of = [&](int u) {
        const int n = min(max(a.len[u], 0), a.cap);
        return (n + kTs - 1) / kTs;
    };

    if (tid == 0) {
        S.bad = 0;
        for (int j = 0; j < kNs; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], 1);
        }
        for (int j = 0; j < kNacc; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], 4);
        }
        for (int j = 0; j < 2; j++) {
            mbar_init(&S.cfull[j], 1);
            mbar_init(&S.cdone[j], kNEpi);
        }
        mbar_init(&S.cfree, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 1) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (w == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int jt = 0, issued = 0;
            const uint64_t once = l2_policy_evict_first();
            for (int j = 0; j < nmine && ok; j++) {
                const int u = unit_of(j), nt = tiles_of(u);
                for (int t = 0; t < nt; t++, jt++) {
                    const int s = jt % kNs;
                    if (!mbar_wait(&S.empty[s], ((uint32_t)(jt / kNs) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&S.full[s], (uint32_t)kOpB);
                    unsigned char *dst = ring + (size_t)s * kOpB;
                    const int row = (int)((size_t)u * a.cap + (size_t)t * kTs);
                    tma_2d_hint(dst, &tmK, 0, row, &S.full[s], once);
                    tma_2d_hint(dst + kUmmaBox, &tmK, 64, row, &S.full[s], once);
                    // the tile's value rows (contiguous) into L2 for the epilogue
                    const size_t rows_left = (size_t)a.U * a.cap - (size_t)row;
                    const uint32_t vbytes = (uint32_t)(min((size_t)kTs, rows_left) * kD * 2);
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.V + (size_t)row * kD),
                                 "r"(vbytes)
                                 : "memory");
                    if (t == 0 && j + 1 < nmine) {
                        // the next unit's C for the converter
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                         a.C + (size_t)unit_of(j + 1) * kD * kD),
                                     "r"((uint32_t)(kD * kD * 4))
                                     : "memory");
                    }
                    issued = jt + 1;
                }
            }
            if (!ok) {
                atomicExch(&S.bad, 1);
                for (int q = max(0, issued - kNs); q < issued; q++)   // copies in flight land
                    mbar_wait(&S.full[q % kNs], (uint32_t)(q / kNs) & 1u);
            }
        }
        __syncwarp();
    } else if (w == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            int jt = 0;
            for (int j = 0; j < nmine && ok; j++) {
                const int u = unit_of(j), nt = tiles_of(u);
                if (!mbar_wait(&S.cfull[j & 1], (uint32_t)(j >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int t = 0; t < nt; t++, jt++) {
                    const int s = jt % kNs, b = jt % kNacc;
                    if (!mbar_wait(&S.full[s], (uint32_t)(jt / kNs) & 1u) ||
                        !mbar_wait(&S.acce[b], ((uint32_t)(jt / kNacc) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(b * 128);
                    const uint64_t dk = umma_sdesc(ring_s + (uint32_t)(s * kOpB));
#pragma unroll
                    for (int sp = 0; sp < 3; sp++) {
                        const uint64_t dc = umma_sdesc(c_s + (uint32_t)(sp * kOpB));
#pragma unroll
                        for (int ks = 0; ks < 8; ks++)
                            umma_bf16(d, umma_sdesc_step(dk, ks), umma_sdesc_step(dc, ks), kNIdesc,
                                      sp > 0 || ks > 0);
                    }
                    umma_commit(&S.accf[b]);
                    umma_commit(&S.empty[s]);       // the key tile is free once its MMAs completed
                }
                umma_commit(&S.cfree);              // the C terms are free once the unit's MMAs completed
            }
            if (!ok) atomicExch(&S.bad, 1);
        }
        __syncwarp();
    } else if (w < kNConv0) {
        // ------------------------------------------------ epilogue (warps 2-9)
        // Set `set` takes the tiles jt with jt % 2 == set; a set's four warps
        // cover the four tensor-memory lane quarters (warp w reaches lanes
        // 32 (w % 4) ..).  A tile's value rows are loaded before its
        // accumulator is awaited.
        const int set = (w - 2) >> 2, qd = w & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        bool good = true;
        int jt = 0;
        for (int j = 0; j < nmine && good; j++) {
            const int u = unit_of(j), nt = tiles_of(u), n = min(max(a.len[u], 0), a.cap);
            bool ok = mbar_wait(&S.cfull[j & 1], (uint32_t)(j >> 1) & 1u);
            good = __all_sync(kFull, ok);
            if (!good) break;
            const float *cmu = S.cmu[j & 1], *mv = S.mv[j & 1];
            for (int t = 0; t < nt; t++, jt++) {
                if ((jt & 1) != set) continue;
                const int b = jt % kNacc;
                const int slot = t * kTs + 32 * qd + lane;
                const bool valid = slot < n;
                uint4 vr[16];
                const uint4 *vp = reinterpret_cast<const uint4 *>(a.V + ((size_t)u * a.cap + slot) * kD);
#pragma unroll
                for (int c = 0; c < 16; c++) vr[c] = valid ? __ldg(vp + c) : make_uint4(0, 0, 0, 0);
                ok = good && mbar_wait(&S.accf[b], (uint32_t)(jt / kNacc) & 1u);
                good = __all_sync(kFull, ok);
                if (good) {
                    tc_fence_after();
                    float acc = 0.f;
#pragma unroll
                    for (int h = 0; h < 4; h++) {            // 32 dims at a time
                        float x[32];
                        tmem_ld32(lane_base + (uint32_t)(b * 128 + 32 * h), x);
#pragma unroll
                        for (int c = 0; c < 4; c++) {
                            float v8[8];
                            unpack8(vr[4 * h + c], v8);
#pragma unroll
                            for (int e = 0; e < 8; e++) {
                                const int dd = 32 * h + 8 * c + e;
                                const float r = v8[e] - mv[dd] - (x[8 * c + e] - cmu[dd]) * a.rs;
                                acc = fmaf(r, r, acc);
                            }
                        }
                    }
                    if (valid) a.rr[(size_t)u * a.cap + slot] = sqrtf(acc);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && good) mbar_arrive(&S.acce[b]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.cdone[j & 1]);    // this unit's vectors are no longer read
        }
        if (!good) atomicExch(&S.bad, 1);
    } else {
        // ------------------------------------------------ converter (warps 10-13)
        // Thread ct owns row ct of C.  Once the previous unit's MMAs are done
        // with the terms, the row (in L2: the producer prefetched it) is
        // split in two halves of 64 columns.
        const int ct = tid - kNConv0 * 32;           // 0..127: row a of C
        bool good = true;
        for (int j = 0; j < nmine && good; j++) {
            const int u = unit_of(j), n = min(max(a.len[u], 0), a.cap);
            const float *Cr = a.C + (size_t)u * kD * kD + (size_t)ct * kD;
            const float *mk = a.mu_k + (size_t)u * kD;
            const uint16_t *kn = a.k_new + (size_t)u * kD;
            const float muv = a.mu_v[(size_t)u * kD + ct];
            // the previous unit's MMAs read the terms; the epilogue of unit
            // j - 2 read this parity's vectors
            bool ok = j < 1 || mbar_wait(&S.cfree, (uint32_t)(j - 1) & 1u);
            ok = ok && (j < 2 || mbar_wait(&S.cdone[j & 1], (uint32_t)((j - 2) >> 1) & 1u));
            if (!ok) good = false;
            float dot_mu = 0.f, dot_new = 0.f;
#pragma unroll 1
            for (int half = 0; half < 2 && good; half++) {
                float4 cr[16];
#pragma unroll
                for (int c = 0; c < 16; c++) cr[c] = *reinterpret_cast<const float4 *>(Cr + 64 * half + 4 * c);
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 mk4 = *reinterpret_cast<const float4 *>(mk + 64 * half + 4 * c);
                    const uint2 kn4 = *reinterpret_cast<const uint2 *>(kn + 64 * half + 4 * c);
                    dot_mu = fmaf(cr[c].x, mk4.x, dot_mu);
                    dot_mu = fmaf(cr[c].y, mk4.y, dot_mu);
                    dot_mu = fmaf(cr[c].z, mk4.z, dot_mu);
                    dot_mu = fmaf(cr[c].w, mk4.w, dot_mu);
                    dot_new = fmaf(cr[c].x, bf_lo(kn4.x), dot_new);
                    dot_new = fmaf(cr[c].y, bf_hi(kn4.x), dot_new);
                    dot_new = fmaf(cr[c].z, bf_lo(kn4.y), dot_new);
                    dot_new = fmaf(cr[c].w, bf_hi(kn4.y), dot_new);
                }
#pragma unroll
                for (int c = 0; c < 8; c++) {        // chunk 8 half + c: columns 8 (8 half + c) ..
                    const float x[8] = {cr[2 * c].x, cr[2 * c].y, cr[2 * c].z, cr[2 * c].w,
                                        cr[2 * c + 1].x, cr[2 * c + 1].y, cr[2 * c + 1].z,
                                        cr[2 * c + 1].w};
                    uint32_t tw[3][4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        float x0 = x[e], x1 = x[e + 1];
#pragma unroll
                        for (int sp = 0; sp < 3; sp++) {
                            const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                            tw[sp][e >> 1] = (uint32_t)__bfloat16_as_ushort(h0) |
                                             ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                            x0 -= __bfloat162float(h0);
                            x1 -= __bfloat162float(h1);
                        }
                    }
#pragma unroll
                    for (int sp = 0; sp < 3; sp++)
                        *reinterpret_cast<uint4 *>(sm + (size_t)sp * kOpB + op_off(ct, 8 * half + c)) =
                            make_uint4(tw[sp][0], tw[sp][1], tw[sp][2], tw[sp][3]);
                }
            }
            if (good) {
                S.cmu[j & 1][ct] = dot_mu;
                S.mv[j & 1][ct] = muv;
            }
            proxy_fence_smem();                      // the terms reach the tensor cores' view
            // the new token: r = v_new - mu_v - (C k_new - C mu_k) / sqrt(d)
            const float rn = bf2f(a.v_new[(size_t)u * kD + ct]) - muv - (dot_new - dot_mu) * a.rs;
            const float q = warp_sum(rn * rn);
            if (lane == 0) S.red[w - kNConv0] = q;
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (ct == 0) {
                if (good && n < a.cap)
                    a.rr[(size_t)u * a.cap + n] = sqrtf((S.red[0] + S.red[1]) + (S.red[2] + S.red[3]));
                mbar_arrive(&S.cfull[j & 1]);
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");   // S.red is reused by the next unit
        }
        if (!good) atomicExch(&S.bad, 1);
    }
    __syncthreads();
    if (w == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && S.bad) record_status(a.status, KVC_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_mi_norms(const kvc_params &p, const kvc_cache &c, const kvc_moments &m,
                            const uint16_t *k_new, const uint16_t *v_new, float *rr,
                            int32_t *status, cudaStream_t st)
{
    const uint64_t rows = (uint64_t)p.U * (uint64_t)p.cap;
    CUtensorMap tmK;
    if (rows + kTs >= (1ull << 31) || !make_row_map(&tmK, c.K, rows, kTs)) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(mi_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kNDyn);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    NormArgs a{c.V, c.len, m.mu_k, m.mu_v, m.C, k_new, v_new, rr, status, p.U, p.cap,
               1.f / sqrtf((float)kD)};
    const int grid = std::max(1, std::min(p.U, nsm));
    mi_norm_kernel<<<grid, kNThreads, kNDyn, st>>>(a, tmK);
    return cudaGetLastError();
}

}  // namespace kvc
