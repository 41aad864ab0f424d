// kvc_fold_tc.cu -- the eviction-set moment fold on the fifth-generation
// tensor cores, for steps that remove many tokens per unit (the first decode
// step over the whole prompt, a prompt hand-off).
//
// MomentKV sec 4.1 keeps, for the evicted set E of a unit, the weight n, the
// means mu_k, mu_v and the cross co-moment S~ = sum_E w (v - mu_v)(k - mu_k)^T
// (C = S~ / n); KeepKV's votes are the weights w.  Victims are taken in tiles
// of 128: the tile's raw product P = sum w v k^T (128 x 128) accumulates in
// tensor memory from the gathered value and key rows (bf16, exact products;
// with votes, w v is carried as two bf16 terms hi + lo, exact while w < 256),
// the tile's weighted sums on CUDA cores; the tile's centred co-moment
// P - (sum w v)(sum w k)^T / n_t is merged into the running (n, mu_k, mu_v,
// M = n C) by the pairwise update of Chan, Golub and LeVeque (1979), so every
// fp32 accumulation is at most one tile long.  M lives in tensor memory.
//
// One CTA per unit (416 threads, one CTA per SM):
//   warps 0-3   epilogue, thread i owns row i of M (value dimension i; the
//               warp's tensor-memory lane quarter), and mu_k[i], mu_v[i]
//   warp 4      tensor-memory owner and MMA issuer (one thread): 8 (or 16
//               with votes) MMAs of 128 x 128 x 16 per tile, both operands
//               MN-major, into one of two accumulators
//   warps 5-12  gather: the tile's victim rows from global memory into the
//               ring (cp.async, 128-byte swizzle, two tiles in flight per
//               thread), w v split, per-warp tile sums
// Every wait is bounded (~2 s); a wait that ran out records KVC_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvc_common.cuh"
#include "kvc_general.h"
#include "kvc_tma.cuh"
#include "kvc_umma.cuh"

namespace kvc {
namespace {

constexpr int kFt = 128;                       // victims per tile
constexpr int kFEpi = 4;                       // epilogue warps (0-3)
constexpr int kFMma = 4;                       // MMA warp
constexpr int kFLoad0 = 5;                     // first gather warp
constexpr int kFLoadWarps = 8;
constexpr int kFThreads = (kFLoad0 + kFLoadWarps) * 32;
constexpr int kFOp = 2 * kUmmaBox;             // one 128 x 128 bf16 operand: 32 KB
constexpr int kFRing = 6 * kFOp;               // 3 stages of (A, B) or 2 of (A, A_lo, B)
constexpr size_t kFDyn = 1024 + (size_t)kFRing;
constexpr int kFMaxStages = 3;
constexpr uint32_t kColM = 256;                // tensor-memory columns of M

// Instruction descriptor: bf16 x bf16 -> fp32, M = N = 128, A and B MN-major
// (bits 15 and 16: the transposed forms).
constexpr uint32_t kFIdesc = umma_idesc_bf16(128, 128) | (1u << 15) | (1u << 16);

// Byte offset of 16-byte chunk c (0..15: dimensions 8c..8c+7) of victim row r
// (0..127) in an operand tile: two boxes of 64 dimensions, 128-byte rows, the
// 16-byte chunk index XOR-ed with r mod 8 (the 128-byte swizzle).
__device__ __forceinline__ uint32_t fop_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kUmmaBox + (r << 7) + (((c & 7) ^ (r & 7)) << 4));
}

// Descriptor of an MN-major operand in that layout: the contraction runs over
// the victim rows.  Leading byte offset = the stride between the two 64-wide
// dimension boxes (16 KB), stride byte offset = between 8-row groups (1 KB),
// version 1, 128-byte swizzle.  Step ks (16 rows) starts 2 KB further.
__device__ __forceinline__ uint64_t fold_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((uint32_t)kUmmaBox >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

__device__ __forceinline__ void tmem_st32(uint32_t addr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf2(float x0, float x1)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
}

struct FoldArgs {
    const uint16_t *K, *V;
    const int32_t *votes, *len;
    const int32_t *evict_idx, *n_evict;
    float *n, *mu_k, *mu_v, *C;
    int32_t *status;
    int cap, kmax;
    int minor_only;
};

struct FoldSmem {
    // first member: the gather warps store it as float4 (16-byte aligned)
    alignas(16) float part[kFMaxStages][kFLoadWarps][2 * kD];   // per gather warp: sum w k | sum w v
    uint64_t full[kFMaxStages], empty[kFMaxStages];
    uint64_t accf[2], acce[2], done;
    float partw[kFMaxStages][kFLoadWarps];           // per gather warp: sum w
    float vsk[2][kD], vdk[2][kD];                    // tile sum w k, mean shift of k
    uint32_t tmem;
    int bad, okv, epibad;
};

__global__ void __launch_bounds__(kFThreads, 1) fold_tc_kernel(FoldArgs a)
{
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    __shared__ __align__(16) FoldSmem S;
    extern __shared__ __align__(1024) unsigned char fdyn[];
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(fdyn) + 1023) & ~uintptr_t(1023));
    const int k = a.n_evict[u];
    if (k <= 0) return;
    const int n_len = a.len[u];
    if (a.minor_only && 2 * k > n_len) return;       // left for the complement
    const int32_t *ev = a.evict_idx + (size_t)u * a.kmax;
    // the victim list: k <= kmax, every slot below the unit's length
    if (tid == 0) S.okv = (k <= a.kmax && n_len >= 0 && n_len <= a.cap) ? 1 : 0;
    __syncthreads();
    if (k <= a.kmax)
        for (int e = tid; e < k; e += blockDim.x) {
            const int s = ev[e];
            if (s < 0 || s >= n_len) S.okv = 0;
        }
    __syncthreads();
    if (!S.okv) {
        if (tid == 0) record_status(a.status, KVC_ERR_INVALID_ARG);
        return;
    }
    const bool wv = a.votes != nullptr;
    const int NS = wv ? 2 : 3;
    const int stage_bytes = wv ? 3 * kFOp : 2 * kFOp;   // A (w v hi), B (k), [A_lo]
    const int nt = (k + kFt - 1) / kFt;
    const size_t ubase = (size_t)u * a.cap;

    if (tid == 0) {
        S.bad = 0;
        S.epibad = 0;
        for (int j = 0; j < kFMaxStages; j++) {
            mbar_init(&S.full[j], kFLoadWarps * 32);
            mbar_init(&S.empty[j], 2);                    // MMA commit + epilogue
        }
        for (int j = 0; j < 2; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], kFEpi);
        }
        mbar_init(&S.done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == kFMma) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (w >= kFLoad0) {
        // ------------------------------------------------ gather
        // Thread lt: 16-byte chunk c of the rows rg, rg + 16, ..., rg + 112,
        // copied straight into the operand tiles (cp.async, 16 bytes each;
        // rows past k are zero-filled).  Two tiles are in flight per thread:
        // tile t + 1 is requested before tile t is finished (its sums read
        // back from shared memory, with votes w v split into hi and lo).
        const int lt = tid - kFLoad0 * 32, c = lt & 15, rg = lt >> 4, wl = w - kFLoad0;
        bool good = true;
        float wnext[8], wcur[8];
        // victim slots of the tile to issue next (loaded one tile ahead, so
        // the copies do not wait on the index loads)
        int slot_n[8];
        auto load_slots = [&](int t) {
#pragma unroll
            for (int jj = 0; jj < 8; jj++) {
                const int e = t * kFt + rg + 16 * jj;
                slot_n[jj] = e < k ? __ldg(ev + e) : -1;
            }
        };
        load_slots(0);
        auto issue = [&](int t, float (&wt)[8]) {
            const int s = t % NS;
            unsigned char *A = ring + (size_t)s * stage_bytes;
            unsigned char *B = A + kFOp;
            int slot_i[8];
#pragma unroll
            for (int jj = 0; jj < 8; jj++) slot_i[jj] = slot_n[jj];
            load_slots(t + 1);
#pragma unroll
            for (int jj = 0; jj < 8; jj++) {
                const int r = rg + 16 * jj, e = t * kFt + r;
                const int sl = slot_i[jj] >= 0 ? slot_i[jj] : 0;
                const size_t row = (ubase + (size_t)sl) * kD + 8 * c;
                const uint32_t bytes = e < k ? 16u : 0u;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(B + fop_off(r, c))),
                             "l"(a.K + row), "r"(bytes)
                             : "memory");
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(A + fop_off(r, c))),
                             "l"(a.V + row), "r"(bytes)
                             : "memory");
                wt[jj] = e < k ? (wv ? (float)__ldg(a.votes + ubase + sl) : 1.f) : 0.f;
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        if (mbar_wait(&S.empty[0], 1u)) issue(0, wnext);
        else good = false;
        if (!__all_sync(kFull, good)) good = false;
        for (int t = 0; t < nt && good; t++) {
            const int s = t % NS;
#pragma unroll
            for (int jj = 0; jj < 8; jj++) wcur[jj] = wnext[jj];
            if (t + 1 < nt) {
                const bool ok = mbar_wait(&S.empty[(t + 1) % NS], ((uint32_t)((t + 1) / NS) & 1u) ^ 1u);
                if (!__all_sync(kFull, ok)) {
                    good = false;
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    break;
                }
                issue(t + 1, wnext);
                asm volatile("cp.async.wait_group 1;" ::: "memory");   // tile t landed
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            unsigned char *A = ring + (size_t)s * stage_bytes;
            unsigned char *B = A + kFOp;
            unsigned char *Al = B + kFOp;
            float sk[8], sv[8], sw = 0.f;
#pragma unroll
            for (int q = 0; q < 8; q++) sk[q] = sv[q] = 0.f;
#pragma unroll
            for (int jj = 0; jj < 8; jj++) {
                const int r = rg + 16 * jj;
                const float wt = wcur[jj];
                float kf[8], vf[8];
                unpack8(*reinterpret_cast<const uint4 *>(B + fop_off(r, c)), kf);
                unpack8(*reinterpret_cast<const uint4 *>(A + fop_off(r, c)), vf);
                sw += wt;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    sk[q] = fmaf(wt, kf[q], sk[q]);
                    sv[q] = fmaf(wt, vf[q], sv[q]);
                }
                if (wv) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const float x = wt * vf[q];          // exact: w < 2^16
                        hi[q] = __bfloat162float(__float2bfloat16_rn(x));
                        lo[q] = x - hi[q];
                    }
                    *reinterpret_cast<uint4 *>(A + fop_off(r, c)) =
                        make_uint4(pack_bf2(hi[0], hi[1]), pack_bf2(hi[2], hi[3]),
                                   pack_bf2(hi[4], hi[5]), pack_bf2(hi[6], hi[7]));
                    *reinterpret_cast<uint4 *>(Al + fop_off(r, c)) =
                        make_uint4(pack_bf2(lo[0], lo[1]), pack_bf2(lo[2], lo[3]),
                                   pack_bf2(lo[4], lo[5]), pack_bf2(lo[6], lo[7]));
                }
            }
            // lanes l and l + 16 hold the same chunk of rows rg and rg + 1
#pragma unroll
            for (int q = 0; q < 8; q++) {
                sk[q] += __shfl_xor_sync(kFull, sk[q], 16);
                sv[q] += __shfl_xor_sync(kFull, sv[q], 16);
            }
            sw += __shfl_xor_sync(kFull, sw, 16);
            if (lane < 16) {
                float *pk = &S.part[s][wl][8 * c];
                float *pv = &S.part[s][wl][kD + 8 * c];
                *reinterpret_cast<float4 *>(pk) = make_float4(sk[0], sk[1], sk[2], sk[3]);
                *reinterpret_cast<float4 *>(pk + 4) = make_float4(sk[4], sk[5], sk[6], sk[7]);
                *reinterpret_cast<float4 *>(pv) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                *reinterpret_cast<float4 *>(pv + 4) = make_float4(sv[4], sv[5], sv[6], sv[7]);
                if (lane == 0) S.partw[s][wl] = sw;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // rows -> tensor cores
            mbar_arrive(&S.full[s]);
        }
        if (!good) atomicExch(&S.bad, 1);
    } else if (w == kFMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            const uint32_t ring_s = smem_u32(ring);
            for (int t = 0; t < nt && ok; t++) {
                const int s = t % NS, b = t & 1;
                if (!mbar_wait(&S.full[s], (uint32_t)(t / NS) & 1u) ||
                    !mbar_wait(&S.acce[b], ((uint32_t)(t >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * 128);
                const uint32_t aA = ring_s + (uint32_t)(s * stage_bytes);
                const uint32_t aB = aA + kFOp, aL = aB + kFOp;
#pragma unroll
                for (int ks = 0; ks < 8; ks++) {
                    const uint32_t off = (uint32_t)ks * 16u * 128u;
                    umma_bf16(d, fold_desc(aA + off), fold_desc(aB + off), kFIdesc, ks > 0);
                    if (wv) umma_bf16(d, fold_desc(aL + off), fold_desc(aB + off), kFIdesc, true);
                }
                umma_commit(&S.accf[b]);
                umma_commit(&S.empty[s]);
            }
            // every MMA issued has completed before tensor memory is released
            umma_commit(&S.done);
            mbar_wait(&S.done, 0);
            if (!ok) atomicExch(&S.bad, 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 0-3)
        const int i = tid;                                   // row of M: value dimension i
        const uint32_t lane_base = tmem + ((uint32_t)(32 * w) << 16);
        float n = a.n[u];
        float muk = a.mu_k[(size_t)u * kD + i], muv = a.mu_v[(size_t)u * kD + i];
        float *Cr = a.C + ((size_t)u * kD + i) * kD;
        // M = n C of the moments as they are
#pragma unroll 1
        for (int h = 0; h < 4; h++) {
            float m[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(Cr + 32 * h + e);
                m[e] = x.x * n; m[e + 1] = x.y * n; m[e + 2] = x.z * n; m[e + 3] = x.w * n;
            }
            tmem_st32(lane_base + kColM + (uint32_t)(32 * h), m);
        }
        tmem_wait_st();
        bool good = true;
        for (int t = 0; t < nt; t++) {
            const int s = t % NS, b = t & 1;
            bool ok = mbar_wait(&S.full[s], (uint32_t)(t / NS) & 1u);
            ok = ok && mbar_wait(&S.accf[b], (uint32_t)(t >> 1) & 1u);
            // a warp that gave up says so before the named barrier; after it
            // the four warps read the same flag and leave together
            if (!__all_sync(kFull, ok) && lane == 0) S.epibad = 1;
            tc_fence_after();
            float skt = 0.f, svt = 0.f, wt = 0.f;
#pragma unroll
            for (int q = 0; q < kFLoadWarps; q++) {
                skt += S.part[s][q][i];
                svt += S.part[s][q][kD + i];
                wt += S.partw[s][q];
            }
            named_sync<kFEpi * 32>();
            if (S.epibad) {
                good = false;
                break;
            }
            if (i == 0) mbar_arrive(&S.empty[s]);           // the sums were read
            const float nn = n + wt;
            float acoef = 0.f, bcoef = 0.f, dk = 0.f;
            if (wt > 0.f) {
                const float mkt = skt / wt, mvt = svt / wt;
                dk = mkt - muk;
                const float dv = mvt - muv;
                acoef = mvt;                                  // (sum w v_i) / n_t
                bcoef = (n * wt / nn) * dv;                   // Chan's cross term
                muk = fmaf(dk, wt / nn, muk);
                muv = fmaf(dv, wt / nn, muv);
                n = nn;
            }
            S.vsk[b][i] = skt;
            S.vdk[b][i] = dk;
            named_sync<kFEpi * 32>();
            {
#pragma unroll 1
                for (int h = 0; h < 4; h++) {
                    uint32_t xr[32], mr[32];
                    tmem_ld32_async(lane_base + (uint32_t)(b * 128 + 32 * h), xr);
                    tmem_ld32_async(lane_base + kColM + (uint32_t)(32 * h), mr);
                    tmem_wait_ld();
                    tmem_bind(xr);
                    tmem_bind(mr);
                    float m[32];
#pragma unroll
                    for (int e = 0; e < 32; e++) {
                        const int j = 32 * h + e;
                        const float ct = fmaf(bcoef, S.vdk[b][j],
                                              fmaf(-acoef, S.vsk[b][j], __uint_as_float(xr[e])));
                        m[e] = __uint_as_float(mr[e]) + ct;
                    }
                    tmem_st32(lane_base + kColM + (uint32_t)(32 * h), m);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.acce[b]);
        }
        if (good) {
            const float rn = 1.f / n;
#pragma unroll 1
            for (int h = 0; h < 4; h++) {
                float m[32];
                tmem_ld32(lane_base + kColM + (uint32_t)(32 * h), m);
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(Cr + 32 * h + e) =
                        make_float4(m[e] * rn, m[e + 1] * rn, m[e + 2] * rn, m[e + 3] * rn);
            }
            a.mu_k[(size_t)u * kD + i] = muk;
            a.mu_v[(size_t)u * kD + i] = muv;
            if (i == 0) a.n[u] = n;
        } else {
            atomicExch(&S.bad, 1);
        }
    }
    __syncthreads();
    if (w == kFMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && S.bad) record_status(a.status, KVC_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_fold_tc(const kvc_cache &c, int cap, int U, int kmax, const int32_t *evict_idx,
                           const int32_t *n_evict, const kvc_moments &m, int32_t *status,
                           cudaStream_t st, bool minor_only)
{
    cudaError_t e = cudaFuncSetAttribute(fold_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFDyn);
    if (e != cudaSuccess) return e;
    FoldArgs a{c.K, c.V, c.votes, c.len, evict_idx, n_evict, m.n, m.mu_k, m.mu_v, m.C,
               status, cap, kmax, minor_only ? 1 : 0};
    fold_tc_kernel<<<U, kFThreads, kFDyn, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
