// kvc_prefill.cu -- LaProx prefill scorer (sm_103a).
//
//   gram_kernel        W_g = sum of the group's W_O slices; Gram = W_g W_g^T
//                      (fp64 accumulation, once per weight set)
//   pack_kernel        per (layer, KV head): the window queries and the Gram
//                      matrix split into three bf16 terms, laid out as the
//                      scorer's shared-memory tensor-core operands
//   prefill_score      one cluster of kCS CTAs per (layer, KV head), 128-key
//                      tiles, every contraction on tcgen05 with the
//                      accumulators in tensor memory:
//                        stat   S = Q K^T (rows x keys): row max / sum of the
//                               window logits, merged over the cluster
//                        norm   S^T = K Q^T (keys x rows): group-mean
//                               attention column norms c_i = ||A_bar[:, i]||_2
//                        val    T = V Gram (keys x dims, three bf16 terms):
//                               r_i^2 = sum_b T[i][b] v_i[b]
//                      p_i = c_i r_i; per-layer sums (fp64)
//   normalize / top-K  s = p / layer sum; global radix select of the B_total
//                      largest (ties to the smaller flat index); keep mask,
//                      per-(layer, KV head) counts, ascending kept indices
//
// Method: LaProx key designs 1-3 and its GQA group-mean paragraph; the
// observation window of the last w prompt queries (SnapKV protocol, as used in
// MomentKV's experimental setup).
#include <cooperative_groups.h>
#include <math.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_tma.cuh"
#include "kvc_umma.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int kPG = 4;               // query heads per KV head (the supported GQA group)
constexpr int kRows = 128;           // window rows: row r = 4 j + h (j = window query, h = head)
constexpr int kCS = 8;               // CTAs per (layer, KV head)
constexpr int kTk = 128;             // keys per tile
constexpr int kOp = 2 * kUmmaBox;    // 32 KB: one 128 x 128 bf16 operand
constexpr int kStages = 3;           // K / V tile ring
constexpr int kAcc = 4;              // tensor-memory accumulators of 128 fp32 columns
constexpr int kEpiWarps = 8;         // two sets of four warps, one per tensor-memory lane quarter
constexpr int kPThreads = (2 + kEpiWarps) * 32;
constexpr int kPackBytes = 4 * kOp;  // [Q][Gram hi][Gram mid][Gram lo]
// shared memory: [Q | Gram x 3 | ring], 1024-byte aligned for the swizzle
constexpr size_t kPDyn = 1024 + (size_t)kPackBytes + (size_t)kStages * kOp;
constexpr uint32_t kIdesc = umma_idesc_bf16(128, 128);

enum JobKind : int { kStat = 0, kNorm = 1, kVal = 2 };

// Byte offset of 16-byte chunk c (0..15) of row r (0..127) in an operand tile.
__host__ __device__ __forceinline__ uint32_t opnd_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kUmmaBox + (r << 7) + (((c & 7) ^ (r & 7)) << 4));
}

// The value norms of tiles t with bit 1 clear run in stage A (with the
// statistics), the others in stage B just before the tile's column norms: both
// stages then mix tensor-bound and exponential-bound jobs.
__host__ __device__ __forceinline__ bool val_in_a(int t) { return ((t >> 1) & 1) == 0; }

// Job order, identical for the TMA producer, the MMA issuer and the epilogue:
// stage A walks the tiles forward, stage B backward (the K tiles read last in
// stage A are read again first, while still in L2).
template <class F>
__device__ __forceinline__ int jobs_stage_a(int nt, F &&f)
{
    int gi = 0;
    for (int t = 0; t < nt; t++) {
        f(gi++, kStat, t);
        if (val_in_a(t)) f(gi++, kVal, t);
    }
    return gi;
}

template <class F>
__device__ __forceinline__ void jobs_stage_b(int nt, int gi, F &&f)
{
    for (int t = nt - 1; t >= 0; t--) {
        if (!val_in_a(t)) f(gi++, kVal, t);
        f(gi++, kNorm, t);
    }
}

struct ScoreArgs {
    const unsigned char *pack;   // [NL][Hkv][kPackBytes] from pack_kernel
    float *p;                    // [NL][Hkv][N]: r^2 (after val), then p = c r
    float2 *stats;               // [NL][Hkv][kCS][2][kRows] partial (max, sum) per row
    double *layer_sum;           // [NL]
    int NL, Hkv, N, w, per_cta;
    float cs;                    // log2(e) / sqrt(d): logits in base-2 units
};

struct PfSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t accf[kAcc];         // accumulator ready (MMA commit)
    uint64_t acce[kAcc];         // accumulator drained (4 epilogue warps)
    uint64_t opnd;               // Q and Gram operands landed
    uint64_t fin;                // every MMA of the CTA completed
    float2 rs[kRows];            // per row: cluster max (base 2) and 1 / sum
    double red[kPThreads / 32];
    uint32_t tmem;
    int bad;
};

__global__ void __launch_bounds__(kPThreads, 1)
prefill_score_kernel(ScoreArgs a, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int cr = (int)cluster.block_rank();
    const int lg = blockIdx.x / kCS;
    const int l = lg / a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

    __shared__ __align__(16) PfSmem S;
    extern __shared__ __align__(1024) unsigned char dyn[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    unsigned char *ring = sm + kPackBytes;
    const uint32_t sm_s = smem_u32(sm), ring_s = smem_u32(ring);

    const int N = a.N, W = a.w;
    const int k0 = min(N, cr * a.per_cta), k1 = min(N, k0 + a.per_cta);
    const int nt = (k1 - k0 + kTk - 1) / kTk;
    float *pout = a.p + (size_t)lg * N + k0;

    if (tid == 0) {
        S.bad = 0;
        for (int j = 0; j < kStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], 1);
        }
        for (int j = 0; j < kAcc; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], 4);
        }
        mbar_init(&S.opnd, 1);
        mbar_init(&S.fin, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 1) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    double lsum = 0.0;

    if (w == 0) {
        // ------------------------------------------------ TMA producer
        cluster_arrive();                 // contributes nothing to the row statistics
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            mbar_expect_tx(&S.opnd, (uint32_t)kPackBytes);
            const unsigned char *src = a.pack + (size_t)lg * kPackBytes;
            for (int j = 0; j < 4; j++) bulk_g2s(sm + j * kOp, src + j * kOp, kOp, &S.opnd);
            const int row0 = lg * N + k0;
            auto issue = [&](int gi, int kind, int t) {
                if (!ok) return;
                const int s = gi % kStages;
                const uint32_t ph = (uint32_t)(gi / kStages) & 1u;
                if (!mbar_wait(&S.empty[s], ph ^ 1u)) { ok = false; return; }
                mbar_expect_tx(&S.full[s], (uint32_t)kOp);
                const CUtensorMap *map = kind == kVal ? &tmV : &tmK;
                unsigned char *dst = ring + (size_t)s * kOp;
                tma_2d(dst, map, 0, row0 + t * kTk, &S.full[s]);
                tma_2d(dst + kUmmaBox, map, 64, row0 + t * kTk, &S.full[s]);
                issued = gi + 1;
            };
            const int ga = jobs_stage_a(nt, issue);
            jobs_stage_b(nt, ga, issue);
            if (!ok) {
                // let the copies in flight land before the CTA may exit
                atomicExch(&S.bad, 1);
                mbar_wait(&S.opnd, 0);
                for (int j = max(0, issued - kStages); j < issued; j++)
                    mbar_wait(&S.full[j % kStages], (uint32_t)(j / kStages) & 1u);
            }
        }
        __syncwarp();
        cluster_wait();
    } else if (w == 1) {
        // ------------------------------------------------ MMA issuer
        cluster_arrive();
        if (lane == 0) {
            bool ok = mbar_wait(&S.opnd, 0);
            auto mma = [&](int gi, int kind, int t) {
                (void)t;
                if (!ok) return;
                const int s = gi % kStages, b = gi % kAcc;
                if (!mbar_wait(&S.full[s], (uint32_t)(gi / kStages) & 1u) ||
                    !mbar_wait(&S.acce[b], ((uint32_t)(gi / kAcc) & 1u) ^ 1u)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * 128);
                const uint32_t tile = ring_s + (uint32_t)(s * kOp);
                if (kind == kVal) {
#pragma unroll 1
                    for (int sp = 0; sp < 3; sp++) {
                        const uint32_t g = sm_s + (uint32_t)((1 + sp) * kOp);
#pragma unroll
                        for (int ks = 0; ks < 8; ks++)
                            umma_bf16(d, umma_sdesc(tile + umma_kstep(ks)),
                                      umma_sdesc(g + umma_kstep(ks)), kIdesc, sp > 0 || ks > 0);
                    }
                } else {
                    // stat: A = Q (rows), B = K tile (keys); norm: the transpose
                    const uint32_t A = kind == kStat ? sm_s : tile;
                    const uint32_t B = kind == kStat ? tile : sm_s;
#pragma unroll
                    for (int ks = 0; ks < 8; ks++)
                        umma_bf16(d, umma_sdesc(A + umma_kstep(ks)), umma_sdesc(B + umma_kstep(ks)),
                                  kIdesc, ks > 0);
                }
                umma_commit(&S.accf[b]);
                // a K tile is free once its MMAs completed; a V tile is also
                // read by the epilogue, which frees it
                if (kind != kVal) umma_commit(&S.empty[s]);
            };
            const int ga = jobs_stage_a(nt, mma);
            jobs_stage_b(nt, ga, mma);
            umma_commit(&S.fin);
            if (!mbar_wait(&S.fin, 0)) ok = false;
            if (!ok) atomicExch(&S.bad, 1);
        }
        __syncwarp();
        cluster_wait();
    } else {
        // ------------------------------------------------ epilogue warps
        const int set = (w - 2) >> 2;              // tiles t with t % 2 == set
        const int qd = w & 3;                      // tensor-memory lane quarter
        const int ln = 32 * qd + lane;             // row (stat) or tile key (norm, val)
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const float cs = a.cs;
        bool good = true;

        // wait for accumulator gi (uniform over the warp)
        auto acquire = [&](int gi) {
            bool ok = good && mbar_wait(&S.accf[gi % kAcc], (uint32_t)(gi / kAcc) & 1u);
            good = __all_sync(kFull, ok);
            if (good) tc_fence_after();
            return good;
        };
        auto release = [&](int gi) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.acce[gi % kAcc]);
        };

        // r^2 of this lane's key: T (keys x 128 dims) against the V tile in smem
        auto val_job = [&](int gi, int t) {
            const int s = gi % kStages;
            if (acquire(gi)) {
                // the V tile is read directly: observe its TMA completion
                bool ok = mbar_wait(&S.full[s], (uint32_t)(gi / kStages) & 1u);
                good = __all_sync(kFull, ok);
            }
            if (good) {
                const unsigned char *vt = ring + (size_t)s * kOp;
                const uint32_t tb = lane_base + (uint32_t)((gi % kAcc) * 128);
                float r2a = 0.f, r2b = 0.f;
#pragma unroll
                for (int cb = 0; cb < 4; cb++) {
                    float x[32];
                    tmem_ld32(tb + 32 * cb, x);
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const uint4 v = lds_v4(vt + opnd_off(ln, 4 * cb + c));
                        float f[8];
                        unpack8(v, f);
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            r2a = fmaf(x[8 * c + e], f[e], r2a);
                            r2b = fmaf(x[8 * c + e + 1], f[e + 1], r2b);
                        }
                    }
                }
                const int kl = t * kTk + ln;
                if (k0 + kl < k1) pout[kl] = r2a + r2b;
            }
            release(gi);
            // every warp of the set has read the V tile: free its ring stage
            asm volatile("bar.sync %0, 128;" ::"r"(2 + set) : "memory");
            if ((w & 3) == 2 && lane == 0 && good) mbar_arrive(&S.empty[s]);
        };

        // ---------------- stage A: row statistics of row ln (base-2 logits)
        const int jr = ln >> 2;
        const int lim = N - W + jr;                // last key window row jr sees
        float m = -INFINITY, sum = 0.f;
        auto stat_job = [&](int gi, int t) {
            if (acquire(gi)) {
                const uint32_t tb = lane_base + (uint32_t)((gi % kAcc) * 128);
                const int kbase = k0 + t * kTk;
                const bool interior = kbase + kTk <= k1 && kbase + kTk - 1 <= N - W;
#pragma unroll
                for (int cb = 0; cb < 4; cb++) {
                    float x[32];
                    tmem_ld32(tb + 32 * cb, x);
                    if (!interior) {
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            const int key = kbase + 32 * cb + i;
                            if (key >= k1 || key > lim) x[i] = -INFINITY;
                        }
                    }
                    float mx = x[0];
#pragma unroll
                    for (int i = 1; i < 32; i++) mx = fmaxf(mx, x[i]);
                    if (mx != -INFINITY) {
                        const float mn = fmaxf(m, mx * cs);
                        float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            e0 += ex2_approx(fmaf(x[i], cs, -mn));
                            e1 += ex2_approx(fmaf(x[i + 1], cs, -mn));
                            e2 += ex2_approx(fmaf(x[i + 2], cs, -mn));
                            e3 += ex2_approx(fmaf(x[i + 3], cs, -mn));
                        }
                        sum = sum * ex2_approx(m - mn) + ((e0 + e1) + (e2 + e3));
                        m = mn;
                    }
                }
            }
            release(gi);
        };
        const int ga = jobs_stage_a(nt, [&](int gi, int kind, int t) {
            if ((t & 1) != set) return;
            if (kind == kStat) stat_job(gi, t);
            else val_job(gi, t);
        });
        // this set's partial statistics of row ln -> global, then the cluster
        // barrier publishes them to the other CTAs of the (layer, KV head)
        a.stats[(((size_t)lg * kCS + cr) * 2 + set) * kRows + ln] = make_float2(m, sum);
        cluster_arrive();
        cluster_wait();
        if (set == 0) {
            const float2 *st = a.stats + (size_t)lg * kCS * 2 * kRows + ln;
            float M = -INFINITY;
            for (int c = 0; c < 2 * kCS; c++) M = fmaxf(M, __ldcg(st + (size_t)c * kRows).x);
            float Z = 0.f;
            for (int c = 0; c < 2 * kCS; c++) {
                const float2 v = __ldcg(st + (size_t)c * kRows);
                if (v.x != -INFINITY) Z += v.y * ex2_approx(v.x - M);
            }
            // rows past the window (zero queries) and empty rows contribute 0
            const bool live = jr < W && M != -INFINITY && Z > 0.f;
            S.rs[ln] = live ? make_float2(M, 1.f / Z) : make_float2(0.f, 0.f);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");

        // ---------------- stage B: column norms, p = c r
        const float4 *rs4 = reinterpret_cast<const float4 *>(S.rs);
        auto norm_job = [&](int gi, int t) {
            if (acquire(gi)) {
                const uint32_t tb = lane_base + (uint32_t)((gi % kAcc) * 128);
                const int kl = t * kTk + ln;
                const int jmin = k0 + kl - (N - W);     // window rows j < jmin do not see the key
                float c2a = 0.f, c2b = 0.f;
#pragma unroll
                for (int cb = 0; cb < 4; cb++) {
                    float x[32];
                    tmem_ld32(tb + 32 * cb, x);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        const float4 A = rs4[16 * cb + 2 * jj], B = rs4[16 * cb + 2 * jj + 1];
                        float sh = ex2_approx(fmaf(x[4 * jj], cs, -A.x)) * A.y;
                        sh = fmaf(ex2_approx(fmaf(x[4 * jj + 1], cs, -A.z)), A.w, sh);
                        sh = fmaf(ex2_approx(fmaf(x[4 * jj + 2], cs, -B.x)), B.y, sh);
                        sh = fmaf(ex2_approx(fmaf(x[4 * jj + 3], cs, -B.z)), B.w, sh);
                        sh = (8 * cb + jj >= jmin) ? sh : 0.f;
                        if (jj & 1) c2b = fmaf(sh, sh, c2b);
                        else c2a = fmaf(sh, sh, c2a);
                    }
                }
                if (k0 + kl < k1) {
                    const float r2 = pout[kl];
                    const float pv = sqrtf((c2a + c2b) * (1.f / (kPG * kPG))) * sqrtf(fmaxf(r2, 0.f));
                    pout[kl] = pv;
                    lsum += (double)pv;
                }
            }
            release(gi);
        };
        jobs_stage_b(nt, ga, [&](int gi, int kind, int t) {
            if ((t & 1) != set) return;
            if (kind == kNorm) norm_job(gi, t);
            else val_job(gi, t);
        });
        if (!good) atomicExch(&S.bad, 1);
    }
    __syncthreads();
    if (w == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // the layer's partial sum of p
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) lsum += __shfl_xor_sync(kFull, lsum, msk);
    if (lane == 0) S.red[w] = lsum;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
        for (int j = 0; j < kPThreads / 32; j++) s += S.red[j];
        atomicAdd(&a.layer_sum[l], s);
        if (S.bad) a.layer_sum[l] = __longlong_as_double(0x7ff8000000000000ll);   // NaN: timed out
    }
}

// --------------------------------------------------------------- operands
// Per (layer, KV head): the 128 window rows (row 4 j + h = query head h of
// the group at window position j; zero past the window) and the three bf16
// terms of the Gram matrix (hi + mid + lo carries its fp32 value), each a
// 128 x 128 K-major tile in the layout of a 128-byte-swizzled TMA load.
__global__ void __launch_bounds__(256) pack_kernel(const uint16_t *q, const float *gram,
                                                   unsigned char *pack, int Hq, int Hkv, int W)
{
    const int lg = blockIdx.x, l = lg / Hkv, g = lg % Hkv;
    unsigned char *dst = pack + (size_t)lg * kPackBytes;
    for (int e = threadIdx.x; e < kRows * 16; e += blockDim.x) {
        const int r = e >> 4, c = e & 15, j = r >> 2, h = r & 3;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j < W) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(
                q + (((size_t)l * Hq + (size_t)g * kPG + h) * W + j) * kD + 8 * c);
            v = make_uint4(src[0], src[1], src[2], src[3]);
        }
        *reinterpret_cast<uint4 *>(dst + opnd_off(r, c)) = v;
    }
    const float *G0 = gram + (size_t)lg * kD * kD;
    for (int e = threadIdx.x; e < kD * 16; e += blockDim.x) {
        const int b = e >> 4, c = e & 15;
        float x[8];
        const float4 lo = *reinterpret_cast<const float4 *>(G0 + (size_t)b * kD + 8 * c);
        const float4 hi = *reinterpret_cast<const float4 *>(G0 + (size_t)b * kD + 8 * c + 4);
        x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
        x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
        uint32_t t[3][4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            float x0 = x[i], x1 = x[i + 1];
#pragma unroll
            for (int sp = 0; sp < 3; sp++) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                t[sp][i >> 1] = (uint32_t)__bfloat16_as_ushort(h0) |
                                ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                x0 -= __bfloat162float(h0);
                x1 -= __bfloat162float(h1);
            }
        }
#pragma unroll
        for (int sp = 0; sp < 3; sp++)
            *reinterpret_cast<uint4 *>(dst + (size_t)(1 + sp) * kOp + opnd_off(b, c)) =
                make_uint4(t[sp][0], t[sp][1], t[sp][2], t[sp][3]);
    }
}

// --------------------------------------------------------------- Gram
// One CTA per (layer, KV head); thread (ta, tb) owns the 8 x 8 block of the
// Gram matrix at rows 8 ta, columns 8 tb.  Columns of W_g are taken 32 at a
// time; W_g entries are fp32 sums of the group's bf16 W_O entries.
__global__ void __launch_bounds__(256) gram_kernel(const uint16_t *W, float *Gram, int Hq, int Hkv,
                                                   int D)
{
    __shared__ float Wc[kD][33];
    const int lg = blockIdx.x, l = lg / Hkv, g = lg % Hkv;
    const int G = Hq / Hkv;
    const int tid = threadIdx.x, ta = tid >> 4, tb = tid & 15;
    double acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[i][j] = 0.0;
    const uint16_t *Wl = W + (size_t)l * Hq * kD * D;
    for (int c0 = 0; c0 < D; c0 += 32) {
        __syncthreads();
        for (int e = tid; e < kD * 32; e += blockDim.x) {
            const int row = e >> 5, col = e & 31;
            float s = 0.f;
            if (c0 + col < D)
                for (int h = g * G; h < (g + 1) * G; h++)
                    s += bf2f(Wl[((size_t)h * kD + row) * D + c0 + col]);
            Wc[row][col] = s;
        }
        __syncthreads();
        for (int cc = 0; cc < 32; cc++) {
            double wa[8], wb[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                wa[i] = (double)Wc[8 * ta + i][cc];
                wb[i] = (double)Wc[8 * tb + i][cc];
            }
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = fma(wa[i], wb[j], acc[i][j]);
        }
    }
    float *Gm = Gram + (size_t)lg * kD * kD;
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) Gm[(8 * ta + i) * kD + 8 * tb + j] = (float)acc[i][j];
}

// --------------------------------------------------------------- top-K
struct TopkState {
    uint32_t prefix, mask;
    int64_t rank;          // rank still to place inside the current prefix
    int64_t below;         // keys strictly below the final threshold
    uint32_t thr;
    int64_t need;          // elements taken from the tie group
};

constexpr int kTkBlock = 1024;
constexpr int kTkPer = 4;                 // elements per thread
constexpr int kTkSpan = kTkBlock * kTkPer;

// order key: ascending key = descending score
__device__ __forceinline__ uint32_t desc_key(float s) { return ~float_key(s); }

__global__ void normalize_kernel(float *s, const double *layer_sum, int64_t per_layer, int64_t M,
                                 int normalize)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M || !normalize) return;
    const double z = layer_sum[i / per_layer];
    s[i] = z > 0.0 ? (float)((double)s[i] / z) : 0.f;
}

__global__ void topk_hist_kernel(const float *s, int64_t M, const TopkState *st, int shift,
                                 unsigned *hist)
{
    __shared__ unsigned h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const uint32_t prefix = st->prefix, mask = st->mask;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < M;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t k = desc_key(s[i]);
        if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&hist[i], h[i]);
}

__global__ void topk_pick_kernel(TopkState *st, unsigned *hist, int shift, int64_t rank0)
{
    if (threadIdx.x != 0) return;
    if (shift == 24) {
        st->rank = rank0;
    }
    int64_t rank = st->rank, cum = 0;
    int b = 0;
    for (; b < 255; b++) {
        if (cum + (int64_t)hist[b] > rank) break;
        cum += hist[b];
    }
    st->prefix |= (uint32_t)b << shift;
    st->mask |= 255u << shift;
    st->rank = rank - cum;
    for (int i = 0; i < 256; i++) hist[i] = 0;
    if (shift == 0) {
        st->thr = st->prefix;
        st->below = rank0 - st->rank;
        st->need = st->rank + 1;
    }
}

// per block: elements below the threshold and equal to it
__global__ void __launch_bounds__(kTkBlock) topk_count_kernel(const float *s, int64_t M,
                                                               const TopkState *st, int *lt,
                                                               int *eq)
{
    __shared__ int scan[40];
    const uint32_t thr = st->thr;
    int nlt = 0, neq = 0;
    const int64_t base = (int64_t)blockIdx.x * kTkSpan;
    for (int k = 0; k < kTkPer; k++) {
        const int64_t i = base + (int64_t)k * kTkBlock + threadIdx.x;
        if (i < M) {
            const uint32_t key = desc_key(s[i]);
            nlt += key < thr;
            neq += key == thr;
        }
    }
    int tlt, teq;
    block_exscan(nlt, scan, &tlt);
    block_exscan(neq, scan, &teq);
    if (threadIdx.x == 0) {
        lt[blockIdx.x] = tlt;
        eq[blockIdx.x] = teq;
    }
}

// one block: offsets of the tie group and of the kept elements per block
__global__ void __launch_bounds__(kTkBlock) topk_scan_kernel(const int *lt, const int *eq, int nblk,
                                                              const TopkState *st, int64_t *eq_off,
                                                              int64_t *keep_off)
{
    __shared__ int scan[40];
    __shared__ int64_t carry[2];
    if (threadIdx.x == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    const int64_t need = st->need;
    for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {
        const int b = b0 + threadIdx.x;
        const int e = b < nblk ? eq[b] : 0;
        int te;
        const int ex = block_exscan(e, scan, &te);
        const int64_t eoff = carry[0] + ex;
        const int64_t take = b < nblk ? max((int64_t)0, min((int64_t)e, need - eoff)) : 0;
        const int kept = b < nblk ? lt[b] + (int)take : 0;
        int tk;
        const int kx = block_exscan(kept, scan, &tk);
        if (b < nblk) {
            eq_off[b] = eoff;
            keep_off[b] = carry[1] + kx;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            carry[0] += te;
            carry[1] += tk;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kTkBlock) topk_write_kernel(const float *s, int64_t M, int N,
                                                               const TopkState *st,
                                                               const int64_t *eq_off,
                                                               const int64_t *keep_off,
                                                               uint8_t *keep, int *counts,
                                                               int64_t *idx)
{
    __shared__ int scan[40];
    const uint32_t thr = st->thr;
    const int64_t need = st->need;
    int64_t eo = eq_off[blockIdx.x], ko = keep_off[blockIdx.x];
    const int64_t base = (int64_t)blockIdx.x * kTkSpan;
    for (int k = 0; k < kTkPer; k++) {
        const int64_t i = base + (int64_t)k * kTkBlock + threadIdx.x;
        uint32_t key = 0xffffffffu;
        const bool in = i < M;
        if (in) key = desc_key(s[i]);
        const int iseq = in && key == thr;
        int teq;
        const int er = block_exscan(iseq, scan, &teq);
        const int kp = in && (key < thr || (iseq && eo + er < need));
        int tkp;
        const int kr = block_exscan(kp, scan, &tkp);
        if (in) keep[i] = (uint8_t)kp;
        if (kp) {
            if (idx) idx[ko + kr] = i;
            if (counts) atomicAdd(&counts[i / N], 1);
        }
        eo += teq;
        ko += tkp;
    }
}

struct PfWs {
    float *p;
    double *layer_sum;
    unsigned char *pack;
    float2 *stats;
    TopkState *st;
    unsigned *hist;
    int *lt, *eq;
    int64_t *eq_off, *keep_off;
    size_t bytes;
};

PfWs pf_layout(int NL, int Hkv, int N, void *base)
{
    PfWs w{};
    char *b = static_cast<char *>(base);
    size_t off = 0;
    const int64_t M = (int64_t)NL * Hkv * N;
    const int64_t nblk = (M + kTkSpan - 1) / kTkSpan;
    auto take = [&](size_t n) {
        char *p = b ? b + off : nullptr;
        off += align_up(n);
        return p;
    };
    w.p = reinterpret_cast<float *>(take((size_t)M * 4));
    w.layer_sum = reinterpret_cast<double *>(take((size_t)NL * 8));
    w.pack = reinterpret_cast<unsigned char *>(take((size_t)NL * Hkv * kPackBytes));
    w.stats = reinterpret_cast<float2 *>(take((size_t)NL * Hkv * kCS * 2 * kRows * sizeof(float2)));
    w.st = reinterpret_cast<TopkState *>(take(sizeof(TopkState)));
    w.hist = reinterpret_cast<unsigned *>(take(256 * 4));
    w.lt = reinterpret_cast<int *>(take((size_t)nblk * 4));
    w.eq = reinterpret_cast<int *>(take((size_t)nblk * 4));
    w.eq_off = reinterpret_cast<int64_t *>(take((size_t)nblk * 8));
    w.keep_off = reinterpret_cast<int64_t *>(take((size_t)nblk * 8));
    w.bytes = off;
    return w;
}

}  // namespace
}  // namespace kvc

using namespace kvc;

#define PF_CHECK(cond, code, ...)      \
    do {                               \
        if (!(cond)) {                 \
            set_error(__VA_ARGS__);    \
            return (code);             \
        }                              \
    } while (0)

static kvc_status pf_cuda(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return KVC_OK;
    set_error("%s: %s", what, cudaGetErrorString(e));
    return KVC_ERR_CUDA;
}

extern "C" {

kvc_status kvc_prefill_prepare(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t D,
                               const uint16_t *W_O, float *Gram, void *stream)
{
    PF_CHECK(NL >= 1 && Hq >= 1 && Hkv >= 1 && D >= 1, KVC_ERR_INVALID_ARG,
             "kvc_prefill_prepare: NL, Hq, Hkv, D must be >= 1");
    PF_CHECK(d == kD, KVC_ERR_UNSUPPORTED, "kvc_prefill_prepare: d = %d unsupported", d);
    PF_CHECK(Hq % Hkv == 0, KVC_ERR_INVALID_ARG, "kvc_prefill_prepare: Hq %% Hkv != 0");
    PF_CHECK(W_O && Gram, KVC_ERR_INVALID_ARG, "kvc_prefill_prepare: NULL pointer");
    gram_kernel<<<NL * Hkv, 256, 0, static_cast<cudaStream_t>(stream)>>>(W_O, Gram, Hq, Hkv, D);
    return pf_cuda(cudaGetLastError(), "kvc_prefill_prepare launch");
}

size_t kvc_prefill_workspace_size(int32_t NL, int32_t Hkv, int32_t N, int64_t B_total)
{
    (void)B_total;
    if (NL < 1 || Hkv < 1 || N < 1) return 0;
    return pf_layout(NL, Hkv, N, nullptr).bytes;
}

kvc_status kvc_prefill_score(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t N,
                             int32_t w, int64_t B_total, int32_t normalize, const uint16_t *q_win,
                             const uint16_t *K, const uint16_t *V, const float *Gram,
                             float *scores, uint8_t *keep, int32_t *counts, int64_t *idx,
                             void *ws, size_t ws_bytes, void *stream)
{
    PF_CHECK(NL >= 1 && Hkv >= 1 && N >= 1 && w >= 1, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: NL, Hkv, N, w must be >= 1");
    PF_CHECK(d == kD, KVC_ERR_UNSUPPORTED, "kvc_prefill_score: d = %d unsupported", d);
    PF_CHECK(Hq == kPG * Hkv, KVC_ERR_UNSUPPORTED,
             "kvc_prefill_score: only 4 query heads per KV head are supported (Hq = %d, Hkv = %d)",
             Hq, Hkv);
    PF_CHECK(w <= 32 && w <= N, KVC_ERR_UNSUPPORTED, "kvc_prefill_score: window w = %d must be <= 32 and <= N", w);
    const int64_t M = (int64_t)NL * Hkv * N;
    PF_CHECK(B_total >= 0 && B_total <= M, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: B_total = %lld outside [0, %lld]", (long long)B_total, (long long)M);
    const int per_cta = ((N + kCS - 1) / kCS + kTk - 1) / kTk * kTk;
    PF_CHECK(q_win && K && V && Gram && keep, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: q_win, K, V, Gram and keep are required");
    PF_CHECK(((uintptr_t)K & 15u) == 0 && ((uintptr_t)V & 15u) == 0 && ((uintptr_t)Gram & 15u) == 0 &&
                 ((uintptr_t)q_win & 3u) == 0,
             KVC_ERR_INVALID_ARG, "kvc_prefill_score: K, V, Gram must be 16-byte aligned, q_win 4-byte");
    PfWs pw = pf_layout(NL, Hkv, N, nullptr);
    PF_CHECK(ws != nullptr && ws_bytes >= pw.bytes && ((uintptr_t)ws & 255u) == 0, KVC_ERR_WORKSPACE,
             "kvc_prefill_score: workspace of %zu bytes (256-byte aligned) required", pw.bytes);
    pw = pf_layout(NL, Hkv, N, ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *pbuf = scores ? scores : pw.p;

    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)NL * Hkv * N;
    PF_CHECK(rows + kTk < (1ull << 31), KVC_ERR_UNSUPPORTED, "kvc_prefill_score: too many rows");
    PF_CHECK(make_row_map(&tmK, K, rows, kTk) && make_row_map(&tmV, V, rows, kTk), KVC_ERR_CUDA,
             "kvc_prefill_score: tensor map encoding failed");
    kvc_status s = pf_cuda(cudaMemsetAsync(pw.layer_sum, 0, (size_t)NL * 8, st), "memset");
    if (s != KVC_OK) return s;
    s = pf_cuda(cudaMemsetAsync(pw.st, 0, sizeof(TopkState), st), "memset");
    if (s != KVC_OK) return s;
    s = pf_cuda(cudaMemsetAsync(pw.hist, 0, 256 * 4, st), "memset");
    if (s != KVC_OK) return s;
    if (counts) {
        s = pf_cuda(cudaMemsetAsync(counts, 0, (size_t)NL * Hkv * 4, st), "memset");
        if (s != KVC_OK) return s;
    }

    pack_kernel<<<NL * Hkv, 256, 0, st>>>(q_win, Gram, pw.pack, Hq, Hkv, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score pack launch");
    ScoreArgs a{pw.pack, pbuf, pw.stats, pw.layer_sum, NL, Hkv, N, w, per_cta,
                (float)(1.4426950408889634 / sqrt((double)kD))};
    e = cudaFuncSetAttribute(prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPDyn);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NL * Hkv * kCS);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPDyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, prefill_score_kernel, a, tmK, tmV);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score launch");

    normalize_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(pbuf, pw.layer_sum, (int64_t)Hkv * N,
                                                                  M, normalize);
    if ((e = cudaGetLastError()) != cudaSuccess) return pf_cuda(e, "normalize launch");
    const int nblk = (int)((M + kTkSpan - 1) / kTkSpan);
    if (B_total == 0) {
        s = pf_cuda(cudaMemsetAsync(keep, 0, (size_t)M, st), "memset");
        return s;
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
        topk_hist_kernel<<<min(nblk * 4, 4 * 152), 512, 0, st>>>(pbuf, M, pw.st, shift, pw.hist);
        topk_pick_kernel<<<1, 32, 0, st>>>(pw.st, pw.hist, shift, B_total - 1);
    }
    topk_count_kernel<<<nblk, kTkBlock, 0, st>>>(pbuf, M, pw.st, pw.lt, pw.eq);
    topk_scan_kernel<<<1, kTkBlock, 0, st>>>(pw.lt, pw.eq, nblk, pw.st, pw.eq_off, pw.keep_off);
    topk_write_kernel<<<nblk, kTkBlock, 0, st>>>(pbuf, M, N, pw.st, pw.eq_off, pw.keep_off, keep,
                                                 counts, idx);
    return pf_cuda(cudaGetLastError(), "kvc_prefill_score top-K launch");
}

}  // extern "C"
