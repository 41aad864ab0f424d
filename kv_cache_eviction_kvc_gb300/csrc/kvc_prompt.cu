// kvc_prompt.cu -- one pass over every live slot of a unit that gives both
// the attention of the step's queries (as split partials) and the weighted
// moments of those slots (n, mu_k, mu_v, M = sum w (v - mu_v)(k - mu_k)^T;
// MomentKV sec 4.1, KeepKV votes as weights), for the decode steps that
// remove most of a unit's slots (the first step over the prompt).
//
// Mode A (append): the step's token joins the unit at slot len (as the
// attention pass does); the moments of all n = len + 1 slots go to the
// workspace.  Mode B (after the victims were compacted away): no token is
// appended; the moments of the n retained slots are taken out of mode A's
// (the reverse of Chan's pairwise update gives the evicted set's), and the
// evicted set's moments are merged into the unit's.  Units where fewer than
// half of the slots went keep the direct fold (its moments are left alone
// here).  Both modes write the split partials that attend_final merges.
//
// One CTA per unit, 320 threads, one CTA per SM; 64-slot tiles, a stage
// holding the key tile and the value tile of the same slots (plus, with
// votes, w v as two bf16 terms):
//   warps 0-3   consumers: S = q K^T and O += P V on tensor cores
//               (mma.sync m16n8k16 from the 128-byte-swizzled tiles), an
//               online softmax per warp, one partial (max, sum, output) per
//               1024-slot chunk; logits for the probabilities
//   warp 4      producer (TMA)
//   warp 5      tensor-memory owner and MMA issuer: P = sum w v k^T of each
//               512-slot group (tcgen05, both operands MN-major) into one of
//               two accumulators
//   warps 6-9   moments: the group's sums from the tiles (a thread takes a
//               16-byte chunk of 8 rows per tile), then thread i (tensor-
//               memory lane i, dimension i) merges the group's centred
//               co-moment P - (sum w v)(sum w k)^T / n_g into M (tensor
//               memory) with Chan's cross term
// Every wait is bounded (~2 s); a wait that ran out records KVC_ERR_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kvc_common.cuh"
#include "kvc_general.h"
#include "kvc_tma.cuh"
#include "kvc_umma.cuh"

namespace kvc {
namespace {

constexpr int kPT = 64;                        // slots per tile
constexpr int kPBox = kPT * 128;               // 8 KB: 64 rows x 64 dimensions
constexpr int kPTile = 2 * kPBox;              // 16 KB: a tile of keys or values
constexpr int kPGroup = 8;                     // tiles per co-moment group (512 slots)
constexpr int kPNC = 8;                        // consumer warps: two sets of four
constexpr int kPProd = 8, kPMma = 9, kPEpi0 = 10;
constexpr int kPThreads = 14 * 32;
constexpr int kPChunkTiles = kAttendChunk / kPT;
constexpr int kPRing = 12 * kPTile;            // 6 stages of (K, V) or 3 of (K, V, hi, lo)
constexpr size_t kPDyn = 1024 + (size_t)kPRing + kPBox;   // + the all-ones operand
constexpr int kPMaxStages = 6;
constexpr uint32_t kPColM = 256;
constexpr uint32_t kPColS = 384;               // sums: [b] at 384 + 32 b (k at +0, v at +16)
static_assert(kAttendChunk % kPT == 0, "attention chunks hold whole tiles");

constexpr uint32_t kPIdesc = umma_idesc_bf16(128, 128) | (1u << 15) | (1u << 16);
constexpr uint32_t kPIdesc16 = umma_idesc_bf16(128, 16) | (1u << 15) | (1u << 16);

__device__ __forceinline__ uint32_t p_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kPBox + (r << 7) + (((c & 7) ^ (r & 7)) << 4));
}

// MN-major operand of a 64-slot tile: leading byte offset 8 KB (between the
// two 64-dimension boxes), stride byte offset 1 KB (8-row groups), version 1,
// 128-byte swizzle; k-step ks (16 slots) starts 2 KB further.
__device__ __forceinline__ uint64_t p_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((uint32_t)kPBox >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

__device__ __forceinline__ void p_tmem_st32(uint32_t addr, const float (&v)[32])
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

__device__ __forceinline__ void p_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pk_bf2(float x0, float x1)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
}

struct PromptArgs {
    const uint16_t *q, *k_new, *v_new;
    uint16_t *K, *V;
    int32_t *votes, *pos;
    double *util;
    const int32_t *len;
    float *xbuf, *part;
    int32_t *nlen, *status;
    float *pmom;                 // [U][kPMomStride]: mode A's moments of all slots
    const int32_t *n_evict;      // mode B: the step's victims per unit
    float *mn, *mu_k, *mu_v, *C; // mode B: the unit's moments
    int U, cap, max_len, new_pos, S;
    int want_x, append;
};

template <int G>
struct PromptSmem {
    // read as float4: 16-byte aligned, first
    alignas(16) float vsk[2][kD];
    alignas(16) float vdk[2][kD];
    uint64_t full[kPMaxStages], ready[kPMaxStages], empty[kPMaxStages];
    uint64_t accf[2], acce[2], done;
    float xs[kPNC][G][16];       // a consumer warp's logits of the current tile
    float wm[kPNC][G], wl[kPNC][G];
    float po[G][kD];
    float gm[G];
    float gk[8][kD], gv[8][kD];  // a group's sums per row group (moments warps)
    float gw[8];
    uint32_t tmem;
    int bad, epibad;
};

template <int G>
__global__ void __launch_bounds__(kPThreads, 1)
prompt_pass_kernel(PromptArgs a, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV)
{
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    __shared__ __align__(16) PromptSmem<G> S;
    extern __shared__ __align__(1024) unsigned char pdyn[];
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(pdyn) + 1023) & ~uintptr_t(1023));
    const int n_old = a.len[u];
    const int n = a.append ? n_old + 1 : n_old;
    if (n_old < 0 || n > a.max_len || n > a.cap) {
        if (tid == 0) {
            record_status(a.status, KVC_ERR_SHAPE);
            a.nlen[u] = -1;
        }
        return;
    }
    if (tid == 0) a.nlen[u] = n;
    if (n == 0) return;
    const bool wv = a.votes != nullptr;
    const int NS = wv ? 3 : 6;
    const int stage_bytes = wv ? 4 * kPTile : 2 * kPTile;   // K, V [, w v hi, w v lo]
    const int nt = (n + kPT - 1) / kPT;
    const int ng = (nt + kPGroup - 1) / kPGroup;
    const size_t ubase = (size_t)u * a.cap;
    const uint16_t *knew = a.append ? a.k_new + (size_t)u * kD : nullptr;
    const uint16_t *vnew = a.append ? a.v_new + (size_t)u * kD : nullptr;

    // the all-ones operand (column 0 of a 64-row box = 1, the rest 0):
    // without votes, sum_r v_r and sum_r k_r come from MMAs against it
    unsigned char *ones = ring + kPRing;
    for (int e = tid; e < kPBox / 16; e += blockDim.x) {
        const int r = e >> 3, c = e & 7;
        const uint32_t lo = (c == ((0 ^ (r & 7)))) ? 0x3F80u : 0u;   // bf16 1.0 in element 0 of chunk 0
        *reinterpret_cast<uint4 *>(ones + (r << 7) + (c << 4)) = make_uint4(lo, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (tid == 0) {
        S.bad = 0;
        S.epibad = 0;
        // ready: the consumers patched the stage (and, with votes, the
        // moments warps wrote w v and took the sums); empty: the consumers
        // and the MMAs are done with it
        for (int j = 0; j < kPMaxStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.ready[j], 4 + (wv ? 4 : 0));
            mbar_init(&S.empty[j], 4 + 1);
        }
        for (int j = 0; j < 2; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], 4);
        }
        mbar_init(&S.done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == kPMma) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (w == kPProd) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            const int row0 = (int)ubase;
            for (int t = 0; t < nt; t++) {
                const int s = t % NS;
                if (!mbar_wait(&S.empty[s], ((uint32_t)(t / NS) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&S.full[s], (uint32_t)(2 * kPTile));
                unsigned char *dst = ring + (size_t)s * stage_bytes;
                tma_2d(dst, &tmK, 0, row0 + t * kPT, &S.full[s]);
                tma_2d(dst + kPBox, &tmK, 64, row0 + t * kPT, &S.full[s]);
                tma_2d(dst + kPTile, &tmV, 0, row0 + t * kPT, &S.full[s]);
                tma_2d(dst + kPTile + kPBox, &tmV, 64, row0 + t * kPT, &S.full[s]);
                issued = t + 1;
            }
            if (!ok) {
                atomicExch(&S.bad, 1);
                for (int q = max(0, issued - NS); q < issued; q++)   // copies in flight land
                    mbar_wait(&S.full[q % NS], (uint32_t)(q / NS) & 1u);
            }
        }
        __syncwarp();
    } else if (w == kPMma) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            const uint32_t ring_s = smem_u32(ring);
            for (int g = 0; g < ng && ok; g++) {
                const int b = g & 1;
                if (!mbar_wait(&S.acce[b], ((uint32_t)(g >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem + (uint32_t)(b * 128);
                const uint32_t ds = tmem + kPColS + (uint32_t)(32 * b);
                const uint32_t aO = ring_s + (uint32_t)kPRing;
                const int t0 = g * kPGroup, t1 = min(nt, t0 + kPGroup);
                for (int t = t0; t < t1 && ok; t++) {
                    const int s = t % NS;
                    if (!mbar_wait(&S.ready[s], (uint32_t)(t / NS) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = ring_s + (uint32_t)(s * stage_bytes);
                    const uint32_t aK = st, aV = st + kPTile, aH = st + 2 * kPTile, aL = st + 3 * kPTile;
#pragma unroll
                    for (int ks = 0; ks < 4; ks++) {
                        const uint32_t off = (uint32_t)ks * 16u * 128u;
                        const bool acc = (t > t0) || ks > 0;
                        if (wv) {
                            umma_bf16(d, p_desc(aH + off), p_desc(aK + off), kPIdesc, acc);
                            umma_bf16(d, p_desc(aL + off), p_desc(aK + off), kPIdesc, true);
                        } else {
                            umma_bf16(d, p_desc(aV + off), p_desc(aK + off), kPIdesc, acc);
                            // sum_r k_r and sum_r v_r (column 0 of each 16-column block)
                            umma_bf16(ds, p_desc(aK + off), p_desc(aO + off), kPIdesc16, acc);
                            umma_bf16(ds + 16, p_desc(aV + off), p_desc(aO + off), kPIdesc16, acc);
                        }
                    }
                    umma_commit(&S.empty[s]);
                }
                if (ok) umma_commit(&S.accf[b]);
            }
            umma_commit(&S.done);
            mbar_wait(&S.done, 0);
            if (!ok) atomicExch(&S.bad, 1);
        }
        __syncwarp();
    } else if (w >= kPEpi0) {
        // ------------------------------------------------ moments (warps 6-9)
        const int qd = w & 3;
        const int i = 32 * qd + lane;                        // dimension i = tensor-memory lane i
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        float n_run = 0.f, muk = 0.f, muv = 0.f;
        {
            float z[32];
#pragma unroll
            for (int e = 0; e < 32; e++) z[e] = 0.f;
#pragma unroll 1
            for (int h = 0; h < 4; h++) p_tmem_st32(lane_base + kPColM + (uint32_t)(32 * h), z);
            p_wait_st();
        }
        // sums: thread mt takes 16-byte chunk c16 of the rows rg, rg + 8, ...
        // of every tile (16-byte shared loads), reduced per group below
        const int mt = tid - kPEpi0 * 32, c16 = mt & 15, rg = mt >> 4;
        bool good = true;
        for (int g = 0; g < ng && good; g++) {
            const int b = g & 1;
            const int t0 = g * kPGroup, t1 = min(nt, t0 + kPGroup);
            float sk8[8], sv8[8], swp = 0.f;
#pragma unroll
            for (int e = 0; e < 8; e++) sk8[e] = sv8[e] = 0.f;
            for (int t = t0; t < t1 && wv; t++) {
                const int s = t % NS;
                // this thread's eight rows' votes, requested before the wait
                int vv[kPT / 8];
#pragma unroll
                for (int j = 0; j < kPT / 8; j++) {
                    const int slot = t * kPT + rg + 8 * j;
                    vv[j] = (slot < n && !(a.append && slot == n_old)) ? __ldg(a.votes + ubase + slot) : 1;
                }
                const bool ok = mbar_wait(&S.full[s], (uint32_t)(t / NS) & 1u);
                if (!__all_sync(kFull, ok)) {
                    good = false;
                    break;
                }
                unsigned char *st = ring + (size_t)s * stage_bytes;
#pragma unroll
                for (int j = 0; j < kPT / 8; j++) {
                    const int r = rg + 8 * j, slot = t * kPT + r;
                    const uint32_t o = p_off(r, c16);
                    uint4 kc = make_uint4(0, 0, 0, 0), vc = make_uint4(0, 0, 0, 0);
                    float wt = 0.f;
                    if (slot < n) {
                        if (a.append && slot == n_old) {
                            kc = *reinterpret_cast<const uint4 *>(knew + 8 * c16);
                            vc = *reinterpret_cast<const uint4 *>(vnew + 8 * c16);
                            wt = 1.f;
                        } else {
                            kc = *reinterpret_cast<const uint4 *>(st + o);
                            vc = *reinterpret_cast<const uint4 *>(st + kPTile + o);
                            wt = (float)vv[j];
                        }
                    }
                    float kf[8], vf[8];
                    unpack8(kc, kf);
                    unpack8(vc, vf);
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        sk8[e] = fmaf(wt, kf[e], sk8[e]);
                        sv8[e] = fmaf(wt, vf[e], sv8[e]);
                    }
                    swp += wt;
                    if (wv) {
                        float hi[8], lo[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const float x = wt * vf[e];          // exact: w < 2^16
                            hi[e] = __bfloat162float(__float2bfloat16_rn(x));
                            lo[e] = x - hi[e];
                        }
                        *reinterpret_cast<uint4 *>(st + 2 * kPTile + o) =
                            make_uint4(pk_bf2(hi[0], hi[1]), pk_bf2(hi[2], hi[3]), pk_bf2(hi[4], hi[5]),
                                       pk_bf2(hi[6], hi[7]));
                        *reinterpret_cast<uint4 *>(st + 3 * kPTile + o) =
                            make_uint4(pk_bf2(lo[0], lo[1]), pk_bf2(lo[2], lo[3]), pk_bf2(lo[4], lo[5]),
                                       pk_bf2(lo[6], lo[7]));
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.ready[s]);
            }
            if (wv) {
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    S.gk[rg][8 * c16 + e] = sk8[e];
                    S.gv[rg][8 * c16 + e] = sv8[e];
                }
                if (c16 == 0) S.gw[rg] = swp;
            }
            // the group's centred co-moment into M (Chan)
            const bool okg = good && mbar_wait(&S.accf[b], (uint32_t)(g >> 1) & 1u);
            if (!__all_sync(kFull, okg) && lane == 0) S.epibad = 1;
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (S.epibad) {
                good = false;
                break;
            }
            tc_fence_after();
            float sk = 0.f, sv = 0.f, sw = 0.f;
            if (wv) {
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    sk += S.gk[q][i];
                    sv += S.gv[q][i];
                    sw += S.gw[q];
                }
            } else {
                // the sums from the MMAs against the all-ones operand; every
                // valid slot weighs 1
                float sr[32];
                tmem_ld32(lane_base + kPColS + (uint32_t)(32 * b), sr);
                sk = sr[0];
                sv = sr[16];
                sw = (float)(min(n, t1 * kPT) - t0 * kPT);
            }
            const float nn = n_run + sw;
            float acoef = 0.f, bcoef = 0.f, dk = 0.f;
            if (sw > 0.f) {
                const float mkt = sk / sw, mvt = sv / sw;
                dk = mkt - muk;
                const float dv = mvt - muv;
                acoef = mvt;
                bcoef = (n_run * sw / nn) * dv;
                muk = fmaf(dk, sw / nn, muk);
                muv = fmaf(dv, sw / nn, muv);
                n_run = nn;
            }
            S.vsk[b][i] = sk;
            S.vdk[b][i] = dk;
            asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll 1
            for (int h = 0; h < 4; h++) {
                uint32_t xr[32], mr[32];
                tmem_ld32_async(lane_base + (uint32_t)(b * 128 + 32 * h), xr);
                tmem_ld32_async(lane_base + kPColM + (uint32_t)(32 * h), mr);
                tmem_wait_ld();
                tmem_bind(xr);
                tmem_bind(mr);
                float m[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 dk4 = *reinterpret_cast<const float4 *>(&S.vdk[b][32 * h + e]);
                    const float4 sk4 = *reinterpret_cast<const float4 *>(&S.vsk[b][32 * h + e]);
                    const float dkv[4] = {dk4.x, dk4.y, dk4.z, dk4.w}, skv[4] = {sk4.x, sk4.y, sk4.z, sk4.w};
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const float ct = fmaf(bcoef, dkv[q], fmaf(-acoef, skv[q], __uint_as_float(xr[e + q])));
                        m[e + q] = __uint_as_float(mr[e + q]) + ct;
                    }
                }
                p_tmem_st32(lane_base + kPColM + (uint32_t)(32 * h), m);
            }
            p_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.acce[b]);
        }
        if (!good) {
            atomicExch(&S.bad, 1);
        } else {
            float *pm = a.pmom + (size_t)u * kPMomStride;
            if (a.append) {
                // mode A: the moments of all n slots
#pragma unroll 1
                for (int h = 0; h < 4; h++) {
                    float m[32];
                    tmem_ld32(lane_base + kPColM + (uint32_t)(32 * h), m);
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(pm + (size_t)i * kD + 32 * h + e) =
                            make_float4(m[e], m[e + 1], m[e + 2], m[e + 3]);
                }
                pm[kD * kD + i] = muk;
                pm[kD * kD + kD + i] = muv;
                if (i == 0) pm[kD * kD + 2 * kD] = n_run;
            } else {
                // mode B: evicted = all - retained (reverse Chan), merged
                // into the unit's moments, where most slots went
                const int kv = a.n_evict[u];
                const bool major = kv > 0 && kv > n;
                if (major) {
                    const float na = pm[kD * kD + 2 * kD];
                    const float ne = na - n_run;
                    const float mka = pm[kD * kD + i], mva = pm[kD * kD + kD + i];
                    const float mke = (na * mka - n_run * muk) / ne;
                    const float mve = (na * mva - n_run * muv) / ne;
                    const float cross_ek = ne * n_run / na;
                    const float dvk = mve - muv;                 // evicted minus retained
                    const float n0 = a.mn[u];
                    const float mk0 = a.mu_k[(size_t)u * kD + i], mv0 = a.mu_v[(size_t)u * kD + i];
                    const float n1 = n0 + ne;
                    const float dv0 = mve - mv0;                 // evicted minus the old moments
                    S.vsk[0][i] = mke - muk;                     // dk evicted - retained
                    S.vdk[0][i] = mke - mk0;                     // dk evicted - old
                    asm volatile("bar.sync 2, 128;" ::: "memory");
                    const float c1 = cross_ek * dvk, c2 = (n0 * ne / n1) * dv0;
                    float *Cr = a.C + ((size_t)u * kD + i) * kD;
#pragma unroll 1
                    for (int h = 0; h < 4; h++) {
                        float m[32];
                        tmem_ld32(lane_base + kPColM + (uint32_t)(32 * h), m);
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float4 ma = *reinterpret_cast<const float4 *>(pm + (size_t)i * kD + 32 * h + e);
                            const float4 c0 = *reinterpret_cast<const float4 *>(Cr + 32 * h + e);
                            const float av[4] = {ma.x, ma.y, ma.z, ma.w};
                            const float cv[4] = {c0.x, c0.y, c0.z, c0.w};
                            float o[4];
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                const int j = 32 * h + e + q;
                                const float me = av[q] - m[e + q] - c1 * S.vsk[0][j];   // M of the evicted set
                                o[q] = (n0 * cv[q] + me + c2 * S.vdk[0][j]) / n1;
                            }
                            *reinterpret_cast<float4 *>(Cr + 32 * h + e) = make_float4(o[0], o[1], o[2], o[3]);
                        }
                    }
                    a.mu_k[(size_t)u * kD + i] = mk0 + (mke - mk0) * (ne / n1);
                    a.mu_v[(size_t)u * kD + i] = mv0 + (mve - mv0) * (ne / n1);
                    asm volatile("bar.sync 2, 128;" ::: "memory");
                    if (i == 0) a.mn[u] = n1;
                }
            }
        }
    } else {
        // ------------------------------------------------ consumers (warps 0-3)
        // q K^T as D[slot][head] (A = 16 key rows by ldmatrix, B = q^T with
        // heads >= G zero), O^T[dim][head] += V^T P^T (A = V^T by
        // ldmatrix.trans, B = P^T with p split into bf16 hi + lo).  Lane
        // (gq, tq) holds logits of slots gq, gq + 8 for heads 2 tq, 2 tq + 1
        // and p of head gq.
        const int gq = lane >> 2, tq = lane & 3;
        const int cset = w >> 2;                     // set 0 takes the even tiles, set 1 the odd
        const int rb = (w & 3) * 16;
        const int h0 = 2 * tq, h1 = 2 * tq + 1;
        const float rs = rsqrtf((float)kD);
        uint32_t qb[8][2];
        {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q + (size_t)u * G * kD);
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                qb[ks][0] = gq < G ? q32[(gq * kD + 16 * ks + 2 * tq) >> 1] : 0u;
                qb[ks][1] = gq < G ? q32[(gq * kD + 16 * ks + 8 + 2 * tq) >> 1] : 0u;
            }
        }
        const uint32_t ring_s = smem_u32(ring);
        float O[8][4];
        float mrun[G];                 // running max per head (this warp's slots)
        float lsq = 0.f;               // sum of p of head gq over this lane's slots
#pragma unroll
        for (int h = 0; h < G; h++) mrun[h] = -INFINITY;
#pragma unroll
        for (int m = 0; m < 8; m++) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
        bool good = true;
        // votes of this lane's two slots (gq, gq + 8) of the set's next tile,
        // loaded one tile ahead so that the loads are in flight meanwhile
        auto load_votes = [&](int t, int &v0, int &v1) {
            const int i = t * kPT + rb + gq;
            v0 = (a.votes && i < n) ? a.votes[ubase + i] : 1;
            v1 = (a.votes && i + 8 < n) ? a.votes[ubase + i + 8] : 1;
        };
        int vn0 = 1, vn1 = 1;
        if (a.votes && cset < nt) load_votes(cset, vn0, vn1);
        const int nch = (nt + kPChunkTiles - 1) / kPChunkTiles;
        for (int cidx = 0; cidx < nch; cidx++) {
          const int tc1 = min(nt, (cidx + 1) * kPChunkTiles);
          for (int t = cidx * kPChunkTiles + cset; t < tc1; t += 2) {
            const int s = t % NS;
            const int vc[2] = {vn0, vn1};
            if (a.votes && t + 2 < nt) load_votes(t + 2, vn0, vn1);
            const uint32_t so = (uint32_t)(s * stage_bytes);
            const bool ok = good && mbar_wait(&S.full[s], (uint32_t)(t / NS) & 1u);
            good = __all_sync(kFull, ok);
            if (good) {
                // rows of this warp past the unit (zeroed) and the appended
                // token's row (written from k_new, v_new), in both tiles
                const int base = t * kPT + rb;
                bool any = false;
                if (base + 16 > n) {
                    for (int e = lane; e < 16 * 16; e += 32) {
                        const int r = e >> 4, j = e & 15;
                        if (base + r >= n) {
                            *reinterpret_cast<uint4 *>(ring + so + p_off(rb + r, j)) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(ring + so + kPTile + p_off(rb + r, j)) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    any = true;
                }
                if (a.append && n_old >= base && n_old < base + 16) {
                    if (lane < 16) {
                        *reinterpret_cast<uint4 *>(ring + so + p_off(n_old - t * kPT, lane)) =
                            *reinterpret_cast<const uint4 *>(knew + 8 * lane);
                        *reinterpret_cast<uint4 *>(ring + so + kPTile + p_off(n_old - t * kPT, lane)) =
                            *reinterpret_cast<const uint4 *>(vnew + 8 * lane);
                    }
                    any = true;
                }
                if (any) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.ready[s]);
                // logits
                float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    // two accumulator chains (k-steps 0-3, 4-7)
                    const int mi = lane >> 3;
                    const int lrow = rb + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < 4; ks++) {
                        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                        ldsm_x4(ring_s + so + p_off(lrow, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                        ldsm_x4(ring_s + so + p_off(lrow, 2 * (ks + 4) + (mi >> 1)), c0, c1, c2, c3);
                        mma16816(sacc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                        mma16816(sacc2, c0, c1, c2, c3, qb[ks + 4][0], qb[ks + 4][1]);
                    }
#pragma unroll
                    for (int e = 0; e < 4; e++) sacc[e] += sacc2[e];
                }
                float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
                for (int hf = 0; hf < 2; hf++) {
                    const int sl = gq + 8 * hf;
                    const int i = base + sl;
                    float x0 = -INFINITY, x1 = -INFINITY;
                    if (i < n) {
                        const bool isnew = a.append && i == n_old;
                        const float lnp = (!isnew && a.votes) ? logf((float)vc[hf]) : 0.f;
                        x0 = sacc[2 * hf] * rs + lnp;
                        x1 = sacc[2 * hf + 1] * rs + lnp;
                    }
                    if (h0 < G) {
                        S.xs[w][h0][sl] = x0;
                        tm0 = fmaxf(tm0, x0);
                        if (a.want_x && i < n) a.xbuf[((size_t)u * G + h0) * a.cap + i] = x0;
                    }
                    if (h1 < G) {
                        S.xs[w][h1][sl] = x1;
                        tm1 = fmaxf(tm1, x1);
                        if (a.want_x && i < n) a.xbuf[((size_t)u * G + h1) * a.cap + i] = x1;
                    }
                }
#pragma unroll
                for (int m = 4; m <= 16; m <<= 1) {
                    tm0 = fmaxf(tm0, __shfl_xor_sync(kFull, tm0, m));
                    tm1 = fmaxf(tm1, __shfl_xor_sync(kFull, tm1, m));
                }
                // the tile max of every head (lanes tq hold heads 2 tq, 2 tq + 1)
                float scl[G];
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float v0 = __shfl_sync(kFull, tm0, h >> 1), v1 = __shfl_sync(kFull, tm1, h >> 1);
                    const float mt = (h & 1) ? v1 : v0;
                    const float mn_ = fmaxf(mrun[h], mt);
                    scl[h] = (mrun[h] == -INFINITY) ? 0.f : expf(mrun[h] - mn_);
                    mrun[h] = mn_;
                }
                __syncwarp();
                // rescale the running output and sum (only when a max rose)
                const float s0 = h0 < G ? scl[h0] : 1.f, s1 = h1 < G ? scl[h1] : 1.f;
                if (__any_sync(kFull, s0 != 1.f || s1 != 1.f)) {
#pragma unroll
                    for (int m = 0; m < 8; m++) {
                        O[m][0] *= s0;
                        O[m][2] *= s0;
                        O[m][1] *= s1;
                        O[m][3] *= s1;
                    }
                }
                float mg = -INFINITY;
#pragma unroll
                for (int h = 0; h < G; h++)
                    if (h == gq) {
                        lsq *= scl[h];
                        mg = mrun[h];
                    }
                // O^T += V^T P^T
                float pv[4];
                const int sl4[4] = {2 * tq, 2 * tq + 1, 8 + 2 * tq, 9 + 2 * tq};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float x = gq < G ? S.xs[w][gq < G ? gq : 0][sl4[e]] : -INFINITY;
                    pv[e] = (gq < G && x != -INFINITY) ? expf(x - mg) : 0.f;
                    lsq += pv[e];
                }
                uint16_t hi0, lo0, hi1, lo1, hi2, lo2, hi3, lo3;
                split_bf16(pv[0], hi0, lo0);
                split_bf16(pv[1], hi1, lo1);
                split_bf16(pv[2], hi2, lo2);
                split_bf16(pv[3], hi3, lo3);
                const uint32_t bh0 = (uint32_t)hi0 | ((uint32_t)hi1 << 16), bh1 = (uint32_t)hi2 | ((uint32_t)hi3 << 16);
                const uint32_t bl0 = (uint32_t)lo0 | ((uint32_t)lo1 << 16), bl1 = (uint32_t)lo2 | ((uint32_t)lo3 << 16);
                {
                    const int mi = lane >> 3;
                    const int lrow = rb + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                    for (int mt = 0; mt < 8; mt++) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(ring_s + so + kPTile + p_off(lrow, 2 * mt + (mi & 1)), a0, a1, a2, a3);
                        mma16816(O[mt], a0, a1, a2, a3, bh0, bh1);
                        mma16816(O[mt], a0, a1, a2, a3, bl0, bl1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.empty[s]);
          }
            // a 1024-slot chunk ends: merge the eight warps into its partial
            {
                float l = lsq;
                l += __shfl_xor_sync(kFull, l, 1);
                l += __shfl_xor_sync(kFull, l, 2);
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < G; h++) S.wm[w][h] = mrun[h];
                if (tq == 0 && gq < G) S.wl[w][gq] = l;
                for (int e = tid; e < G * kD; e += kPNC * 32) S.po[e / kD][e % kD] = 0.f;
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (tid < G) {
                    float M = -INFINITY;
                    for (int q = 0; q < kPNC; q++) M = fmaxf(M, S.wm[q][tid]);
                    S.gm[tid] = M;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                const float f0 = (h0 < G && mrun[h0] != -INFINITY) ? expf(mrun[h0] - S.gm[h0]) : 0.f;
                const float f1 = (h1 < G && mrun[h1] != -INFINITY) ? expf(mrun[h1] - S.gm[h1]) : 0.f;
#pragma unroll
                for (int m = 0; m < 8; m++) {
                    if (h0 < G) {
                        atomicAdd(&S.po[h0][16 * m + gq], O[m][0] * f0);
                        atomicAdd(&S.po[h0][16 * m + gq + 8], O[m][2] * f0);
                    }
                    if (h1 < G) {
                        atomicAdd(&S.po[h1][16 * m + gq], O[m][1] * f1);
                        atomicAdd(&S.po[h1][16 * m + gq + 8], O[m][3] * f1);
                    }
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                const int sc = cidx;
                float *pp = a.part + ((size_t)u * a.S + sc) * G * (kD + 2);
                for (int e = tid; e < G * kD; e += kPNC * 32) {
                    const int h = e / kD, dd = e % kD;
                    pp[h * (kD + 2) + 2 + dd] = S.po[h][dd];
                }
                if (tid < G) {
                    float ll = 0.f;
                    for (int q = 0; q < kPNC; q++)
                        if (S.wm[q][tid] != -INFINITY) ll += S.wl[q][tid] * expf(S.wm[q][tid] - S.gm[tid]);
                    pp[tid * (kD + 2) + 0] = S.gm[tid];
                    pp[tid * (kD + 2) + 1] = ll;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
#pragma unroll
                for (int h = 0; h < G; h++) mrun[h] = -INFINITY;
                lsq = 0.f;
#pragma unroll
                for (int m = 0; m < 8; m++) O[m][0] = O[m][1] = O[m][2] = O[m][3] = 0.f;
            }
        }
        if (!good) atomicExch(&S.bad, 1);
        // the appended token joins the cache
        if (a.append && tid == 0) a.pos[ubase + n_old] = a.new_pos;
        if (a.append && tid == 1) {
            if (a.votes) a.votes[ubase + n_old] = 1;
            a.util[ubase + n_old] = __longlong_as_double(0x7ff0000000000000ll);
        }
        if (a.append && tid >= 32 && tid < 64) {
            uint16_t *kd = a.K + (ubase + n_old) * kD;
            uint16_t *vd = a.V + (ubase + n_old) * kD;
            reinterpret_cast<uint2 *>(kd)[tid - 32] = reinterpret_cast<const uint2 *>(knew)[tid - 32];
            reinterpret_cast<uint2 *>(vd)[tid - 32] = reinterpret_cast<const uint2 *>(vnew)[tid - 32];
        }
    }
    __syncthreads();
    if (w == kPMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && S.bad) record_status(a.status, KVC_ERR_TIMEOUT);
}

template <int G>
cudaError_t launch_prompt_g(const PromptArgs &a, int U, const CUtensorMap &tmK, const CUtensorMap &tmV,
                            cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(prompt_pass_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPDyn);
    if (e != cudaSuccess) return e;
    prompt_pass_kernel<G><<<U, kPThreads, kPDyn, st>>>(a, tmK, tmV);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prompt_pass(const kvc_params &p, int new_pos, int max_len, const uint16_t *q,
                               const uint16_t *k_new, const uint16_t *v_new, const kvc_cache &c,
                               bool append, bool want_x, const int32_t *n_evict,
                               const kvc_moments &m, const DecodeWs &ws, cudaStream_t st)
{
    const uint64_t rows = (uint64_t)p.U * (uint64_t)p.cap;
    CUtensorMap tmK, tmV;
    if (rows + kPT >= (1ull << 31) || !make_row_map(&tmK, c.K, rows, kPT) ||
        !make_row_map(&tmV, c.V, rows, kPT))
        return cudaErrorNotSupported;
    const int S = (p.cap + kAttendChunk - 1) / kAttendChunk;
    PromptArgs a{q, k_new, v_new, c.K, c.V, c.votes, c.pos, c.util, c.len,
                 ws.xbuf, ws.part, ws.nlen, ws.status, ws.pmom, n_evict,
                 m.n, m.mu_k, m.mu_v, m.C, p.U, p.cap, max_len, new_pos, S,
                 want_x ? 1 : 0, append ? 1 : 0};
    switch (p.G) {
    case 1: return launch_prompt_g<1>(a, p.U, tmK, tmV, st);
    case 2: return launch_prompt_g<2>(a, p.U, tmK, tmV, st);
    case 4: return launch_prompt_g<4>(a, p.U, tmK, tmV, st);
    case 8: return launch_prompt_g<8>(a, p.U, tmK, tmV, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvc
