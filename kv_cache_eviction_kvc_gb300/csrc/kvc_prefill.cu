// kvc_prefill.cu -- LaProx prefill scorer (sm_103a).
//
//   gram_kernel        W_g = sum of the group's W_O slices; Gram = W_g W_g^T
//                      (fp64 accumulation, once per weight set)
//   prefill_score      one cluster of kCS CTAs per (layer, KV head):
//                        phase 0  row max / sum of the window logits
//                                 (q K^T on tensor cores), merged over the
//                                 cluster through distributed shared memory
//                        phase 1  group-mean attention column norms
//                                 c_i = ||A_bar[:, i]||_2
//                        phase 2  r_i = sqrt(v_i^T Gram v_i) on tensor cores
//                                 (Gram split into three bf16 terms)
//                        p_i = c_i r_i; per-layer sums (fp64)
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

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int kPG = 4;               // query heads per KV head (the supported GQA group)
constexpr int kRows = 128;           // window rows: row r = 4 j + h (j = window query, h = head)
constexpr int kPCW = 8;              // consumer warps: 16 rows each
constexpr int kPThreads = (kPCW + 1) * 32;
constexpr int kCS = 8;               // CTAs per (layer, KV head)
constexpr int kTk = 64;              // keys per ring stage
constexpr int kPBox = kTk * 128;     // bytes of one box (64 keys x 64 dims)
constexpr int kPStage = 2 * kPBox;   // 16 KB: 64 keys x 128 dims
constexpr int kPStages = 4;
constexpr int kMaxKeysCTA = 4096;

__device__ __forceinline__ uint32_t psw(int r, int j) { return sw_off_t<kTk>(r, j); }

struct ScoreArgs {
    const uint16_t *q;     // [NL][Hq][w][d]
    const float *gram;     // [NL][Hkv][d][d]
    float *p;              // [NL][Hkv][N]  indicator p = c r
    double *layer_sum;     // [NL]
    int NL, Hq, Hkv, N, w, per_cta;
};

struct PfSmem {
    uint64_t full[kPStages];
    uint64_t empty[kPStages];
    float pm[kRows], pl[kRows];      // this CTA's row max / sum (read by the cluster)
    float c2[kMaxKeysCTA];           // sum_j A_bar[j, i]^2
    float r2[kMaxKeysCTA];           // v_i^T Gram v_i
    double red[kPThreads / 32];
    int bad;
};

__global__ void __launch_bounds__(kPThreads, 1)
prefill_score_kernel(ScoreArgs a, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int cr = (int)cluster.block_rank();
    const int lg = blockIdx.x / kCS;
    const int l = lg / a.Hkv, g = lg % a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;

    __shared__ PfSmem S;
    extern __shared__ __align__(128) unsigned char dyn[];
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_s = smem_u32(ring);

    const int N = a.N, W = a.w;
    const int k0 = min(N, cr * a.per_cta), k1 = min(N, k0 + a.per_cta);
    const int nk = k1 - k0;
    const int ntile = (nk + kTk - 1) / kTk;
    const float rs = rsqrtf((float)kD);

    for (int i = tid; i < kMaxKeysCTA; i += blockDim.x) {
        S.c2[i] = 0.f;
        S.r2[i] = 0.f;
    }
    if (tid == 0) {
        S.bad = 0;
        for (int j = 0; j < kPStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], kPCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (w == kPCW) {
        // ------------------------------------------------ producer warp
        // K tiles (phase 0), K tiles again (phase 1, mostly from L2), V tiles
        const int row0 = (int)((size_t)lg * N + k0);
        bool ok = true;
        int gi = 0;
        auto issue = [&](const CUtensorMap *map) {
            for (int t = 0; t < ntile && ok; t++, gi++) {
                const int stage = gi % kPStages;
                const uint32_t ph = (uint32_t)(gi / kPStages) & 1u;
                if (!mbar_wait(&S.empty[stage], ph ^ 1u)) { ok = false; break; }
                mbar_expect_tx(&S.full[stage], (uint32_t)kPStage);
                unsigned char *dst = ring + (size_t)stage * kPStage;
                tma_2d(dst, map, 0, row0 + t * kTk, &S.full[stage]);
                tma_2d(dst + kPBox, map, 64, row0 + t * kTk, &S.full[stage]);
            }
        };
        if (lane == 0) issue(&tmK);
        __syncwarp();
        cluster_arrive();                 // phase-0 barrier: arrive now, wait after issuing
        if (lane == 0) {
            issue(&tmK);
            issue(&tmV);
            if (!ok) {
                atomicExch(&S.bad, 1);
                for (int j = max(0, gi - kPStages); j < gi; j++)
                    mbar_wait(&S.full[j % kPStages], (uint32_t)(j / kPStages) & 1u);
            }
        }
        __syncwarp();
        cluster_wait();
    } else {
        // ------------------------------------------------ consumers
        // rows of this lane: r1 = 16 w + gq and r2 = r1 + 8 (same head, window + 2)
        const int r1 = 16 * w + gq;
        const int j1 = r1 >> 2, j2 = j1 + 2, hh = r1 & 3;
        const int lim1 = N - W + j1, lim2 = N - W + j2;     // last visible key of each row
        const bool v1 = j1 < W, v2 = j2 < W;
        uint32_t qa[8][4];
        {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q);
            const size_t hq = (size_t)l * a.Hq + (size_t)g * kPG + hh;
            const size_t b1 = ((hq * W + j1) * kD) >> 1, b2 = ((hq * W + j2) * kD) >> 1;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                qa[ks][0] = v1 ? q32[b1 + 8 * ks + tq] : 0u;
                qa[ks][1] = v2 ? q32[b2 + 8 * ks + tq] : 0u;
                qa[ks][2] = v1 ? q32[b1 + 8 * ks + 4 + tq] : 0u;
                qa[ks][3] = v2 ? q32[b2 + 8 * ks + 4 + tq] : 0u;
            }
        }
        bool good = true;
        int gi = 0;
        // S (16 rows x 64 keys) of one tile on tensor cores
        auto qk_tile = [&](uint32_t so, float (&Sf)[8][4]) {
#pragma unroll
            for (int n = 0; n < 8; n++) Sf[n][0] = Sf[n][1] = Sf[n][2] = Sf[n][3] = 0.f;
            const int mi = lane >> 3;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
#pragma unroll
                for (int np = 0; np < 4; np++) {
                    const int lrow = 16 * np + ((mi >> 1) << 3) + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(ring_s + so + psw(lrow, 2 * ks + (mi & 1)), b0, b1, b2, b3);
                    mma16816(Sf[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma16816(Sf[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
            }
        };
        auto acquire = [&](int &stage, uint32_t &so) {
            stage = gi % kPStages;
            const uint32_t ph = (uint32_t)(gi / kPStages) & 1u;
            if (good && !mbar_wait(&S.full[stage], ph)) good = false;
            so = (uint32_t)stage * kPStage;
        };
        auto release = [&](int stage) {
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.empty[stage]);
            gi++;
        };

        // ---------------- phase 0: row max and sum
        float m1 = -INFINITY, s1 = 0.f, m2 = -INFINITY, s2 = 0.f;
        for (int t = 0; t < ntile; t++) {
            int stage;
            uint32_t so;
            acquire(stage, so);
            if (good) {
                float Sf[8][4];
                qk_tile(so, Sf);
                float x[8][4];
                float tm1 = -INFINITY, tm2 = -INFINITY;
#pragma unroll
                for (int n = 0; n < 8; n++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int key = k0 + t * kTk + 8 * n + 2 * tq + e;
                        const bool ok = key < k1;
                        x[n][e] = (ok && v1 && key <= lim1) ? Sf[n][e] * rs : -INFINITY;
                        x[n][2 + e] = (ok && v2 && key <= lim2) ? Sf[n][2 + e] * rs : -INFINITY;
                        tm1 = fmaxf(tm1, x[n][e]);
                        tm2 = fmaxf(tm2, x[n][2 + e]);
                    }
                const float n1m = fmaxf(m1, tm1), n2m = fmaxf(m2, tm2);
                if (n1m != -INFINITY) {
                    float acc = (m1 == -INFINITY) ? 0.f : s1 * expf(m1 - n1m);
#pragma unroll
                    for (int n = 0; n < 8; n++)
#pragma unroll
                        for (int e = 0; e < 2; e++) acc += expf(x[n][e] - n1m);
                    s1 = acc;
                    m1 = n1m;
                }
                if (n2m != -INFINITY) {
                    float acc = (m2 == -INFINITY) ? 0.f : s2 * expf(m2 - n2m);
#pragma unroll
                    for (int n = 0; n < 8; n++)
#pragma unroll
                        for (int e = 0; e < 2; e++) acc += expf(x[n][2 + e] - n2m);
                    s2 = acc;
                    m2 = n2m;
                }
            }
            release(stage);
        }
        // merge over the 4 lanes sharing the rows
#pragma unroll
        for (int msk = 1; msk <= 2; msk <<= 1) {
            const float om1 = __shfl_xor_sync(kFull, m1, msk), os1 = __shfl_xor_sync(kFull, s1, msk);
            const float om2 = __shfl_xor_sync(kFull, m2, msk), os2 = __shfl_xor_sync(kFull, s2, msk);
            const float nm1 = fmaxf(m1, om1), nm2 = fmaxf(m2, om2);
            s1 = (nm1 == -INFINITY) ? 0.f
                                    : ((m1 == -INFINITY ? 0.f : s1 * expf(m1 - nm1)) +
                                       (om1 == -INFINITY ? 0.f : os1 * expf(om1 - nm1)));
            s2 = (nm2 == -INFINITY) ? 0.f
                                    : ((m2 == -INFINITY ? 0.f : s2 * expf(m2 - nm2)) +
                                       (om2 == -INFINITY ? 0.f : os2 * expf(om2 - nm2)));
            m1 = nm1;
            m2 = nm2;
        }
        if (tq == 0) {
            S.pm[r1] = m1; S.pl[r1] = s1;
            S.pm[r1 + 8] = m2; S.pl[r1 + 8] = s2;
        }
        cluster_arrive();
        cluster_wait();
        // cluster-wide row statistics of this lane's two rows
        float M1 = -INFINITY, M2 = -INFINITY;
        for (int q = 0; q < kCS; q++) {
            PfSmem *R = cluster.map_shared_rank(&S, q);
            M1 = fmaxf(M1, R->pm[r1]);
            M2 = fmaxf(M2, R->pm[r1 + 8]);
        }
        float Z1 = 0.f, Z2 = 0.f;
        for (int q = 0; q < kCS; q++) {
            PfSmem *R = cluster.map_shared_rank(&S, q);
            if (R->pm[r1] != -INFINITY) Z1 += R->pl[r1] * expf(R->pm[r1] - M1);
            if (R->pm[r1 + 8] != -INFINITY) Z2 += R->pl[r1 + 8] * expf(R->pm[r1 + 8] - M2);
        }
        const float iz1 = Z1 > 0.f ? 1.f / Z1 : 0.f, iz2 = Z2 > 0.f ? 1.f / Z2 : 0.f;

        // ---------------- phase 1: group-mean column norms
        for (int t = 0; t < ntile; t++) {
            int stage;
            uint32_t so;
            acquire(stage, so);
            if (good) {
                float Sf[8][4];
                qk_tile(so, Sf);
#pragma unroll
                for (int n = 0; n < 8; n++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int key = k0 + t * kTk + 8 * n + 2 * tq + e;
                        const bool ok = key < k1;
                        float pa = (ok && v1 && key <= lim1) ? expf(Sf[n][e] * rs - M1) * iz1 : 0.f;
                        float pb = (ok && v2 && key <= lim2) ? expf(Sf[n][2 + e] * rs - M2) * iz2 : 0.f;
                        // sum over the 4 heads of the window row (lane bits 2-3)
                        pa += __shfl_xor_sync(kFull, pa, 4);
                        pa += __shfl_xor_sync(kFull, pa, 8);
                        pb += __shfl_xor_sync(kFull, pb, 4);
                        pb += __shfl_xor_sync(kFull, pb, 8);
                        pa *= 1.f / kPG;
                        pb *= 1.f / kPG;
                        float sq = pa * pa + pb * pb;
                        sq += __shfl_xor_sync(kFull, sq, 16);   // the warp's 4 window rows
                        if (gq == 0 && ok) atomicAdd(&S.c2[key - k0], sq);
                    }
            }
            release(stage);
        }

        // ---------------- phase 2: r_i^2 = v_i^T Gram v_i
        // warp w owns Gram rows b = 16 w .. 16 w + 15; A = Gram (b x a, three
        // bf16 terms), B = V^T (a x keys): T^T[b][key] = sum_a Gram[b][a] v[key][a]
        uint32_t ga[3][8][4];
        {
            const float *G0 = a.gram + (size_t)lg * kD * kD;
            const int b1 = 16 * w + gq, b2 = b1 + 8;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                const int c0 = 16 * ks + 2 * tq;
                const float vals[4][2] = {{G0[b1 * kD + c0], G0[b1 * kD + c0 + 1]},
                                          {G0[b2 * kD + c0], G0[b2 * kD + c0 + 1]},
                                          {G0[b1 * kD + c0 + 8], G0[b1 * kD + c0 + 9]},
                                          {G0[b2 * kD + c0 + 8], G0[b2 * kD + c0 + 9]}};
#pragma unroll
                for (int rg = 0; rg < 4; rg++) {
                    uint16_t t0[3], t1[3];
                    float x0 = vals[rg][0], x1 = vals[rg][1];
#pragma unroll
                    for (int sp = 0; sp < 3; sp++) {
                        const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                        t0[sp] = __bfloat16_as_ushort(h0);
                        t1[sp] = __bfloat16_as_ushort(h1);
                        x0 -= __bfloat162float(h0);
                        x1 -= __bfloat162float(h1);
                    }
#pragma unroll
                    for (int sp = 0; sp < 3; sp++)
                        ga[sp][ks][rg] = (uint32_t)t0[sp] | ((uint32_t)t1[sp] << 16);
                }
            }
        }
        const int b1 = 16 * w + gq;
        for (int t = 0; t < ntile; t++) {
            int stage;
            uint32_t so;
            acquire(stage, so);
            if (good) {
                float T[8][4];
#pragma unroll
                for (int n = 0; n < 8; n++) T[n][0] = T[n][1] = T[n][2] = T[n][3] = 0.f;
                const int mi = lane >> 3;
#pragma unroll
                for (int ks = 0; ks < 8; ks++) {
#pragma unroll
                    for (int np = 0; np < 4; np++) {
                        const int lrow = 16 * np + ((mi >> 1) << 3) + (lane & 7);
                        uint32_t b0, bb1, b2, b3;
                        ldsm_x4(ring_s + so + psw(lrow, 2 * ks + (mi & 1)), b0, bb1, b2, b3);
#pragma unroll
                        for (int sp = 0; sp < 3; sp++) {
                            mma16816(T[2 * np], ga[sp][ks][0], ga[sp][ks][1], ga[sp][ks][2],
                                     ga[sp][ks][3], b0, bb1);
                            mma16816(T[2 * np + 1], ga[sp][ks][0], ga[sp][ks][1], ga[sp][ks][2],
                                     ga[sp][ks][3], b2, b3);
                        }
                    }
                }
                // r^2 partial = sum over this lane's b rows of T^T[b][key] v[key][b]
                const unsigned char *tile = ring + so;
#pragma unroll
                for (int n = 0; n < 8; n++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int krow = 8 * n + 2 * tq + e;
                        const uint16_t va = *reinterpret_cast<const uint16_t *>(
                            tile + psw(krow, b1 >> 3) + (b1 & 7) * 2);
                        const uint16_t vb = *reinterpret_cast<const uint16_t *>(
                            tile + psw(krow, (b1 + 8) >> 3) + ((b1 + 8) & 7) * 2);
                        float part = T[n][e] * bf2f(va) + T[n][2 + e] * bf2f(vb);
                        part += __shfl_xor_sync(kFull, part, 4);
                        part += __shfl_xor_sync(kFull, part, 8);
                        part += __shfl_xor_sync(kFull, part, 16);
                        const int key = k0 + t * kTk + krow;
                        if (gq == 0 && key < k1) atomicAdd(&S.r2[krow + t * kTk], part);
                    }
            }
            release(stage);
        }
        if (!good) atomicExch(&S.bad, 1);
    }
    __syncthreads();
    // ---------------- p = c r and the layer's partial sum
    double part = 0.0;
    float *pout = a.p + (size_t)lg * N + k0;
    for (int i = tid; i < nk; i += blockDim.x) {
        const float c = sqrtf(S.c2[i]);
        const float r = sqrtf(fmaxf(S.r2[i], 0.f));
        const float pv = c * r;
        pout[i] = pv;
        part += (double)pv;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) part += __shfl_xor_sync(kFull, part, m);
    if (lane == 0) S.red[w] = part;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
        for (int j = 0; j < kPThreads / 32; j++) s += S.red[j];
        atomicAdd(&a.layer_sum[l], s);
        if (S.bad) a.layer_sum[l] = __longlong_as_double(0x7ff8000000000000ll);   // NaN: timed out
    }
    cluster_arrive();              // no CTA leaves while another may read its partials
    cluster_wait();
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
    PF_CHECK(per_cta <= kMaxKeysCTA, KVC_ERR_UNSUPPORTED,
             "kvc_prefill_score: N = %d too long (at most %d)", N, kCS * kMaxKeysCTA);
    PF_CHECK(q_win && K && V && Gram && keep, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: q_win, K, V, Gram and keep are required");
    PF_CHECK(((uintptr_t)K & 15u) == 0 && ((uintptr_t)V & 15u) == 0 && ((uintptr_t)q_win & 3u) == 0,
             KVC_ERR_INVALID_ARG, "kvc_prefill_score: K, V must be 16-byte aligned");
    PfWs pw = pf_layout(NL, Hkv, N, nullptr);
    PF_CHECK(ws != nullptr && ws_bytes >= pw.bytes && ((uintptr_t)ws & 255u) == 0, KVC_ERR_WORKSPACE,
             "kvc_prefill_score: workspace of %zu bytes (256-byte aligned) required", pw.bytes);
    pw = pf_layout(NL, Hkv, N, ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *pbuf = scores ? scores : pw.p;

    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)NL * Hkv * N;
    PF_CHECK(rows < (1ull << 31), KVC_ERR_UNSUPPORTED, "kvc_prefill_score: too many rows");
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

    ScoreArgs a{q_win, Gram, pbuf, pw.layer_sum, NL, Hq, Hkv, N, w, per_cta};
    const size_t dyn = 1024 + (size_t)kPStages * kPStage;
    cudaError_t e = cudaFuncSetAttribute(prefill_score_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NL * Hkv * kCS);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = dyn;
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
