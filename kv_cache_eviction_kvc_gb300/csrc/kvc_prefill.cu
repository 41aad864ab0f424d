// kvc_prefill.cu -- LaProx prefill scorer (sm_103a).
//
//   factor_kernel      W_g = sum of the group's W_O slices; Gram = W_g W_g^T
//                      in fp64 and its pivoted Cholesky factor R (R^T R =
//                      Gram), once per weight set
//   pack_kernel        per (layer, KV head): the window queries and R split
//                      into three bf16 terms, laid out as the scorer's
//                      shared-memory tensor-core operands
//   prefill_val        r_i^2 = ||(V W_g)[i, :]||^2 = sum_b T[i][b]^2 with
//                      T = V R^T (keys x dims, R as three bf16 terms);
//                      persistent, 128-key tiles scheduled dynamically
//   prefill_attn       persistent 8-CTA clusters looping over (layer, KV head)
//                      items, 128-key tiles per CTA:
//                        stat   S = Q K^T (rows x keys): row max / sum of the
//                               window logits, merged over the cluster
//                        norm   S^T = K Q^T (keys x rows): group-mean
//                               attention column norms c_i = ||A_bar[:, i]||_2
//                      the column norms c_i (combine_kernel then writes
//                      p_i = c_i r_i and the per-layer sums of p, fp64);
//                      optionally the weighted column sum
//                      S_i = sum_j roww_j A_bar[j, i] (SnapKV's accumulated
//                      window attention, KeepKV's windowed EMA init)
//                      Both kernels: every contraction on tcgen05 (128 x 128
//                      x 128 bf16, fp32 accumulators in tensor memory), a TMA
//                      producer warp, one MMA-issuing thread, epilogue warps
//                      reading the accumulators by lane quarter.  They run
//                      side by side: the attention clusters on the caller's
//                      stream, the value norms on a library stream (behind a
//                      short pause_kernel, so that the clusters are placed
//                      first) taking the SMs the clusters leave free.
//   select             s = p / layer sum; three-pass radix select of the
//                      B_total largest (ties to the smaller flat index); keep
//                      mask, per-(layer, KV head) counts, ascending kept
//                      indices
//
// Method: LaProx key designs 1-3 and its GQA group-mean paragraph; the
// observation window of the last w prompt queries (SnapKV protocol, as used in
// MomentKV's experimental setup).
#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>
#include <cstddef>
#include <mutex>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_tma.cuh"
#include "kvc_umma.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int kPG = 4;               // query heads per KV head (the supported GQA group)
constexpr int kRows = 128;           // window rows: row r = 4 j + h (j = window query, h = head)
constexpr int kCS = 8;               // CTAs per (layer, KV head) in the attention kernel
constexpr int kTk = 128;             // keys per tile
constexpr int kOp = 2 * kUmmaBox;    // 32 KB: one 128 x 128 bf16 operand
constexpr int kAcc = 4;              // tensor-memory accumulators of 128 fp32 columns
constexpr int kPackBytes = 4 * kOp;  // [Q][R hi][R mid][R lo]
constexpr uint32_t kIdesc = umma_idesc_bf16(128, 128);

// attention kernel: [Q (three buffers) | ring of K tiles]
constexpr int kAQ = 3;
constexpr int kAStages = 4;
constexpr int kALead = 4;            // statistics jobs of a block before its first norm job
constexpr int kASets = 2;            // epilogue sets: tile t goes to set t % kASets
constexpr int kAEpiWarps = 4 * kASets;   // four warps per set, one per tensor-memory lane quarter
constexpr int kAThreads = (2 + kAEpiWarps) * 32;
constexpr size_t kADyn = 1024 + (size_t)kAQ * kOp + (size_t)kAStages * kOp;
// value-norm kernel: [R x 3 | ring of V tiles]
constexpr int kVStages = 4;
constexpr int kVThreads = (2 + 4 + 1) * 32;   // producer, MMA, 4 epilogue, scheduler
constexpr size_t kVDyn = 1024 + (size_t)3 * kOp + (size_t)kVStages * kOp;

// Byte offset of 16-byte chunk c (0..15) of row r (0..127) in an operand tile.
__host__ __device__ __forceinline__ uint32_t opnd_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kUmmaBox + (r << 7) + (((c & 7) ^ (r & 7)) << 4));
}

struct Ring {
    // shared by the producer, the MMA issuer and the epilogue: job gi uses
    // ring stage gi % stages and accumulator gi % kAcc
    static __device__ __forceinline__ uint32_t stage_parity(int gi, int stages)
    {
        return (uint32_t)(gi / stages) & 1u;
    }
    static __device__ __forceinline__ uint32_t acc_parity(int gi) { return (uint32_t)(gi / kAcc) & 1u; }
};

// =============================================================== attention
// Persistent: gridDim.x / kCS clusters of kCS CTAs; cluster c takes the
// (layer, KV head) items c, c + nclu, ... (item p of the cluster); within an
// item CTA cr owns keys [cr per_cta, (cr + 1) per_cta).  Per item, stat(t)
// for t = 0..nt-1 (S = Q K_t^T, rows x keys: row max / sum) and norm(t) for
// t = nt-1..0 (S^T = K_t Q^T, keys x rows: column norms).  The items are
// software-pipelined: block p runs stat(p) and then norm(p - 1), so the
// cluster-wide merge of item p - 1's statistics is hidden behind a whole
// statistics pass.  Q of item p lives in buffer p % 3.
// Output: the column norms c_i = ||A_bar[:, i]||_2 (combine_kernel then
// forms p_i = c_i r_i with r_i from the value-norm kernel, which runs beside
// this one), and/or the weighted column sums.
struct AttnArgs {
    const unsigned char *pack;   // [NL][Hkv][kPackBytes] from pack_kernel
    float *c;                    // [NL][Hkv][N]: column norms c (want_c)
    float2 *stats;               // [NL][Hkv][kCS][kASets][kRows] partial (max, sum) per row
    double *layer_sum;           // [NL]: NaN on a timed-out wait
    float *colsum;               // [NL][Hkv][N]: sum_j roww_j A_bar[j, i], or NULL
    int Hkv, N, w, per_cta, nitem;
    int want_c;                  // LaProx's attention column norms
    float cs;                    // log2(e) / sqrt(d): logits in base-2 units
    float roww[32];              // window row weights of colsum
};

struct AttnSmem {
    uint64_t full[kAStages];
    uint64_t empty[kAStages];
    uint64_t accf[kAcc];         // accumulator ready (MMA commit)
    uint64_t acce[kAcc];         // accumulator drained (4 epilogue warps)
    uint64_t qfull[kAQ];         // Q buffer loaded
    uint64_t qfree[kAQ];         // every MMA reading the Q buffer completed
    uint64_t ready[2];           // the cluster's partial statistics of an item are published
    uint64_t fin;                // every MMA of the CTA completed
    __align__(16) float rm[kRows];    // per row: minus the cluster max (base 2); read as float4
    __align__(16) float rz[kRows];    // per row: 1 / cluster sum; read as float4
    float roww[32];              // colsum weights per window row
    uint32_t tmem;
    int bad;
};
static_assert(offsetof(AttnSmem, rm) % 16 == 0 && offsetof(AttnSmem, rz) % 16 == 0,
              "rm and rz are read as float4");

// Two fp32 lanes per instruction (Blackwell's packed f32x2 arithmetic): each
// lane is rounded exactly as the scalar fma / mul / add would round it.
__device__ __forceinline__ uint64_t f2pk(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2up(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint64_t ex2_2(uint64_t t)
{
    const float2 v = f2up(t);
    return f2pk(ex2_approx(v.x), ex2_approx(v.y));
}

// Statistics of one window row over a 128-key tile (x: logits, masked keys
// at -inf): the running base-2 max m and sum of 2^(x cs - m).
__device__ __forceinline__ void row_stats(const float (&x)[128], float cs, float &m, float &sum)
{
    float mx[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        float a = fmax3(x[32 * k], x[32 * k + 1], x[32 * k + 2]);
#pragma unroll
        for (int i = 3; i < 31; i += 2) a = fmax3(a, x[32 * k + i], x[32 * k + i + 1]);
        mx[k] = fmaxf(a, x[32 * k + 31]);
    }
    const float tm = fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], mx[3]);
    if (tm == -INFINITY) return;
    const float mn = fmaxf(m, tm * cs);
    const uint64_t cs2 = f2pk(cs, cs), nm2 = f2pk(-mn, -mn);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 64; i++)
        acc[i & 3] = add2(acc[i & 3], ex2_2(fma2(f2pk(x[2 * i], x[2 * i + 1]), cs2, nm2)));
    const float2 a = f2up(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
    sum = sum * ex2_approx(m - mn) + (a.x + a.y);
    m = mn;
}

// Column sums of one key over the 128 window rows (x[4 j + h]: window query
// j, head h): sum_j sh_j^2 and sum_j roww_j sh_j with sh_j the group sum of
// the probabilities 2^(x cs - M) / Z.  MASK: rows j < jmin do not see the key.
template <bool MASK, bool COLSUM>
__device__ __forceinline__ void key_norms(const float (&x)[128], float cs, const float *rm,
                                          const float *rz, const float *roww, int jmin,
                                          float &c2s, float &cws)
{
    const float4 *rm4 = reinterpret_cast<const float4 *>(rm);
    const float4 *rz4 = reinterpret_cast<const float4 *>(rz);
    const uint64_t cs2 = f2pk(cs, cs);
    float c2[4] = {0.f, 0.f, 0.f, 0.f};
    float cw[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; j++) {
        const float4 A = rm4[j], Z = rz4[j];
        const uint64_t e01 = ex2_2(fma2(f2pk(x[4 * j], x[4 * j + 1]), cs2, f2pk(A.x, A.y)));
        const uint64_t e23 = ex2_2(fma2(f2pk(x[4 * j + 2], x[4 * j + 3]), cs2, f2pk(A.z, A.w)));
        const float2 pr = f2up(fma2(e23, f2pk(Z.z, Z.w), mul2(e01, f2pk(Z.x, Z.y))));
        float sh = pr.x + pr.y;
        if (MASK) sh = (j >= jmin) ? sh : 0.f;
        c2[j & 3] = fmaf(sh, sh, c2[j & 3]);
        if (COLSUM) cw[j & 3] = fmaf(roww[j], sh, cw[j & 3]);
    }
    c2s = (c2[0] + c2[1]) + (c2[2] + c2[3]);
    cws = (cw[0] + cw[1]) + (cw[2] + cw[3]);
}

__global__ void __launch_bounds__(kAThreads, 1)
prefill_attn_kernel(AttnArgs a, const __grid_constant__ CUtensorMap tmK)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int cr = (int)cluster.block_rank();
    const int cid = blockIdx.x / kCS, nclu = gridDim.x / kCS;
    const int nmine = cid < a.nitem ? (a.nitem - cid + nclu - 1) / nclu : 0;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

    __shared__ __align__(16) AttnSmem S;
    extern __shared__ __align__(1024) unsigned char dyn[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    unsigned char *ring = sm + kAQ * kOp;      // [Q x kAQ | ring]
    const uint32_t q_s = smem_u32(sm), ring_s = smem_u32(ring);

    const int N = a.N, W = a.w;
    const int k0 = min(N, cr * a.per_cta), k1 = min(N, k0 + a.per_cta);
    const int nt = (k1 - k0 + kTk - 1) / kTk;
    // first job of block p (block 0: nt jobs, blocks 1..nmine-1: 2 nt, block nmine: nt)
    auto block_base = [nt](int p) { return p == 0 ? 0 : (2 * p - 1) * nt; };
    // Jobs of block p in order: kALead statistics jobs of item p, then (where
    // item p - 1 exists) mid() -- the point where its merged statistics are
    // needed -- and its column-norm jobs alternating with the remaining
    // statistics jobs: HBM-bound and exponential-bound work overlap.
    auto for_block = [nt, nmine, &block_base](int p, auto &&stat, auto &&norm, auto &&mid) {
        const int ns = p < nmine ? nt : 0, nn = p >= 1 ? nt : 0;
        int gi = block_base(p), is = 0, in = 0;
        for (; is < min(ns, kALead); is++) stat(gi++, is);
        if (nn) mid();
        while (is < ns || in < nn) {
            if (in < nn) norm(gi++, nt - 1 - in++);
            if (is < ns) stat(gi++, is++);
        }
    };
    auto none = [] {};

    if (tid < 32) S.roww[tid] = a.roww[tid];
    if (tid == 0) {
        S.bad = 0;
        for (int j = 0; j < kAStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], 1);
        }
        for (int j = 0; j < kAcc; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], 4);
        }
        for (int j = 0; j < kAQ; j++) {
            mbar_init(&S.qfull[j], 1);
            mbar_init(&S.qfree[j], 1);
        }
        for (int j = 0; j < 2; j++) mbar_init(&S.ready[j], kCS);
        mbar_init(&S.fin, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 1) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    // peers arrive on this CTA's barriers: all of them are initialized first
    cluster_arrive();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (w == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0, qloads = 0;
            // each K tile is read twice: kept in L2 until its second read
            const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_first();
            auto load = [&](int gi, int lg, int t, uint64_t pol) {
                const int s = gi % kAStages;
                if (!mbar_wait(&S.empty[s], Ring::stage_parity(gi, kAStages) ^ 1u)) {
                    ok = false;
                    return;
                }
                mbar_expect_tx(&S.full[s], (uint32_t)kOp);
                unsigned char *dst = ring + (size_t)s * kOp;
                const int row = lg * N + k0 + t * kTk;
                tma_2d_hint(dst, &tmK, 0, row, &S.full[s], pol);
                tma_2d_hint(dst + kUmmaBox, &tmK, 64, row, &S.full[s], pol);
                issued = gi + 1;
            };
            for (int p = 0; p <= nmine && ok; p++) {
                if (p < nmine) {
                    const int lg = cid + p * nclu, qb = p % kAQ;
                    // buffer qb held Q of item p - kAQ: free once its column norms completed
                    if (p >= kAQ && !mbar_wait(&S.qfree[qb], (uint32_t)(p / kAQ - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&S.qfull[qb], (uint32_t)kOp);
                    bulk_g2s(sm + qb * kOp, a.pack + (size_t)lg * kPackBytes, kOp, &S.qfull[qb]);
                    qloads = p + 1;
                }
                const int lgs = cid + p * nclu, lgn = cid + (p - 1) * nclu;
                for_block(p, [&](int gi, int t) { if (ok) load(gi, lgs, t, keep); },
                          [&](int gi, int t) { if (ok) load(gi, lgn, t, once); }, none);
            }
            if (!ok) {
                // let the copies in flight land before the CTA may exit
                atomicExch(&S.bad, 1);
                for (int j = max(0, qloads - kAQ); j < qloads; j++)
                    mbar_wait(&S.qfull[j % kAQ], (uint32_t)(j / kAQ) & 1u);
                for (int j = max(0, issued - kAStages); j < issued; j++)
                    mbar_wait(&S.full[j % kAStages], Ring::stage_parity(j, kAStages));
            }
        }
        __syncwarp();
    } else if (w == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            // one job: 8 MMAs of 128 x 128 x 16 into accumulator gi % kAcc;
            // stat: A = Q (rows), B = K tile (keys); norm: the transpose
            auto mma = [&](int gi, uint32_t qa, bool stat) {
                const int s = gi % kAStages, b = gi % kAcc;
                if (!mbar_wait(&S.full[s], Ring::stage_parity(gi, kAStages)) ||
                    !mbar_wait(&S.acce[b], Ring::acc_parity(gi) ^ 1u)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * 128);
                const uint32_t tile = ring_s + (uint32_t)(s * kOp);
                const uint64_t dq = umma_sdesc(qa), dt = umma_sdesc(tile);
                const uint64_t dA = stat ? dq : dt, dB = stat ? dt : dq;
#pragma unroll
                for (int ks = 0; ks < 8; ks++)
                    umma_bf16(d, umma_sdesc_step(dA, ks), umma_sdesc_step(dB, ks), kIdesc, ks > 0);
                umma_commit(&S.accf[b]);
                umma_commit(&S.empty[s]);     // the tile is free once its MMAs completed
            };
            for (int p = 0; p <= nmine && ok; p++) {
                if (p < nmine && !mbar_wait(&S.qfull[p % kAQ], (uint32_t)(p / kAQ) & 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t qs = q_s + (uint32_t)((p % kAQ) * kOp);
                const uint32_t qn = q_s + (uint32_t)(((p + kAQ - 1) % kAQ) * kOp);
                for_block(p, [&](int gi, int) { if (ok) mma(gi, qs, true); },
                          [&](int gi, int) { if (ok) mma(gi, qn, false); }, none);
                if (p >= 1) umma_commit(&S.qfree[(p - 1) % kAQ]);    // item p - 1's Q buffer
            }
            umma_commit(&S.fin);
            if (!mbar_wait(&S.fin, 0)) ok = false;
            if (!ok) atomicExch(&S.bad, 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps
        const int set = (w - 2) >> 2;              // tiles t with t % kASets == set
        const int qd = w & 3;                      // tensor-memory lane quarter
        const int ln = 32 * qd + lane;             // row (stat) or tile key (norm)
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const float cs = a.cs;
        const int jr = ln >> 2;
        const int lim = N - W + jr;                // last key window row jr sees
        bool good = true;

        // wait for accumulator gi (uniform over the warp)
        auto acquire = [&](int gi) {
            bool ok = good && mbar_wait(&S.accf[gi % kAcc], Ring::acc_parity(gi));
            good = __all_sync(kFull, ok);
            if (good) tc_fence_after();
            return good;
        };
        auto release = [&](int gi) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.acce[gi % kAcc]);
        };

        for (int p = 0; p <= nmine; p++) {
            const int lgs = cid + p * nclu, q = p - 1, lgn = cid + q * nclu;
            float m = -INFINITY, sum = 0.f;        // statistics of row ln of item p (base-2 logits)
            // ---------------- statistics job: tile t of item p
            auto stat = [&](int gi, int t) {
                if (t % kASets != set) return;
                if (acquire(gi)) {
                    const uint32_t tb = lane_base + (uint32_t)((gi % kAcc) * 128);
                    const int kbase = k0 + t * kTk;
                    const bool interior = kbase + kTk <= k1 && kbase + kTk - 1 <= N - W;
                    float x[128];
                    tmem_ld128(tb, x);
                    release(gi);                  // the accumulator is drained into registers
                    if (!interior) {
#pragma unroll
                        for (int i = 0; i < 128; i++) {
                            const int key = kbase + i;
                            if (key >= k1 || key > lim) x[i] = -INFINITY;
                        }
                    }
                    row_stats(x, cs, m, sum);
                } else {
                    release(gi);
                }
            };
            // ---------------- merged statistics of item p - 1 (needed by its norm jobs)
            auto mid = [&] {
                if (set == 0) {
                    bool ok = good && mbar_wait_cluster(&S.ready[q & 1], (uint32_t)(q >> 1) & 1u);
                    good = __all_sync(kFull, ok);
                    const float2 *st = a.stats + (size_t)lgn * kCS * kASets * kRows + ln;
                    float2 v[kASets * kCS];
#pragma unroll
                    for (int c = 0; c < kASets * kCS; c++) v[c] = __ldcg(st + (size_t)c * kRows);
                    float M = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kASets * kCS; c++) M = fmaxf(M, v[c].x);
                    float Z = 0.f;
#pragma unroll
                    for (int c = 0; c < kASets * kCS; c++)
                        if (v[c].x != -INFINITY) Z += v[c].y * ex2_approx(v[c].x - M);
                    // rows past the window (zero queries) and empty rows contribute 0
                    const bool live = jr < W && M != -INFINITY && Z > 0.f;
                    S.rm[ln] = live ? -M : 0.f;
                    S.rz[ln] = live ? 1.f / Z : 0.f;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kAEpiWarps * 32) : "memory");
            };
            // ---------------- column-norm job: tile t of item p - 1
            auto norm = [&](int gi, int t) {
                if (t % kASets != set) return;
                const int kl = t * kTk + ln;
                const size_t o = (size_t)lgn * N + k0 + kl;
                if (acquire(gi)) {
                    const uint32_t tb = lane_base + (uint32_t)((gi % kAcc) * 128);
                    const int jmin = k0 + kl - (N - W);     // window rows j < jmin do not see the key
                    float x[128];
                    tmem_ld128(tb, x);
                    release(gi);                  // the accumulator is drained into registers
                    float c2 = 0.f, cw = 0.f;     // cw: weighted column sum (times G)
                    const bool mask = __any_sync(kFull, jmin > 0);
                    if (a.colsum) {
                        if (mask) key_norms<true, true>(x, cs, S.rm, S.rz, S.roww, jmin, c2, cw);
                        else key_norms<false, true>(x, cs, S.rm, S.rz, S.roww, jmin, c2, cw);
                    } else {
                        if (mask) key_norms<true, false>(x, cs, S.rm, S.rz, S.roww, jmin, c2, cw);
                        else key_norms<false, false>(x, cs, S.rm, S.rz, S.roww, jmin, c2, cw);
                    }
                    if (k0 + kl < k1) {
                        if (a.want_c) a.c[o] = sqrtf(c2 * (1.f / (kPG * kPG)));
                        if (a.colsum) a.colsum[o] = cw * (1.f / kPG);
                    }
                } else {
                    release(gi);
                }
            };
            for_block(p, stat, norm, mid);
            if (p < nmine) {
                // publish this set's partial statistics of row ln; one thread
                // then tells every CTA of the cluster (release at cluster scope)
                a.stats[(((size_t)lgs * kCS + cr) * kASets + set) * kRows + ln] = make_float2(m, sum);
                __threadfence();
                asm volatile("bar.sync 1, %0;" ::"n"(kAEpiWarps * 32) : "memory");
                if (tid == 64)
                    for (int c = 0; c < kCS; c++) mbar_arrive_remote(&S.ready[p & 1], (uint32_t)c);
            }
        }
        if (!good) atomicExch(&S.bad, 1);
    }
    __syncthreads();
    if (w == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && S.bad)
        for (int p = 0; p < nmine; p++)    // NaN: a wait timed out
            a.layer_sum[(cid + p * nclu) / a.Hkv] = __longlong_as_double(0x7ff8000000000000ll);
    // no CTA leaves while a peer may still arrive on its barriers
    cluster_arrive();
    cluster_wait();
}

// =============================================================== value norms
// Persistent, dynamically scheduled: the producer of each CTA opens a
// (layer, KV head) item from a global counter and takes chunks of kVChunk of
// its key tiles from the item's own counter until the item runs dry, then
// opens the next; once every item is open it helps with whatever tiles are
// left.  Chunks reach the MMA issuer and the epilogue through a small
// shared-memory queue; R is reloaded only where the item changes.  Per tile: T = V_t R^T (keys x dims; R as three
// bf16 terms accumulated into one fp32 accumulator), r^2 = sum_b T[i][b]^2.
constexpr int kVChunk = 4;           // tiles per chunk
constexpr int kVQueue = 3;           // chunks posted ahead of the epilogue

struct ValArgs {
    const unsigned char *pack;   // [NL][Hkv][kPackBytes]
    float *r2;                   // [NL][Hkv][N]
    double *layer_sum;           // [NL]: NaN on a timed-out wait
    int *item_next;              // next unopened item (zero before the launch)
    int *tile_next;              // [NL Hkv] next free tile of each item (zero before the launch)
    int NL, N, ntl;              // ntl = tiles per (layer, KV head)
    int nitem;                   // NL Hkv
};

struct ValSmem {
    uint64_t full[kVStages];
    uint64_t empty[kVStages];
    uint64_t accf[kAcc];
    uint64_t acce[kAcc];
    uint64_t qfull[kVQueue];     // chunk posted by the producer
    uint64_t qfree[kVQueue];     // chunk finished by the epilogue (4 warps)
    uint64_t rfull, rfree;       // R loaded / every MMA reading it completed
    uint64_t fin;
    long long chunk[kVQueue];    // first tile of the chunk, -1: no more work
    uint32_t tmem;
    int bad;
};

__global__ void __launch_bounds__(kVThreads, 1)
prefill_val_kernel(ValArgs a, const __grid_constant__ CUtensorMap tmV)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int N = a.N, ntl = a.ntl;

    __shared__ __align__(16) ValSmem S;
    extern __shared__ __align__(1024) unsigned char dyn[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    unsigned char *ring = sm + 3 * kOp;
    const uint32_t r_s = smem_u32(sm), ring_s = smem_u32(ring);

    if (tid == 0) {
        S.bad = 0;
        for (int j = 0; j < kVStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], 1);
        }
        for (int j = 0; j < kAcc; j++) {
            mbar_init(&S.accf[j], 1);
            mbar_init(&S.acce[j], 4);
        }
        for (int j = 0; j < kVQueue; j++) {
            mbar_init(&S.qfull[j], 1);
            mbar_init(&S.qfree[j], 4);
        }
        mbar_init(&S.rfull, 1);
        mbar_init(&S.rfree, 1);
        mbar_init(&S.fin, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (w == 1) tmem_alloc(&S.tmem, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;

    // chunk k of this CTA: wait until posted, return its first tile (-1: done)
    auto take = [&](int k, bool &ok) -> long long {
        const int slot = k % kVQueue;
        if (!ok || !mbar_wait(&S.qfull[slot], (uint32_t)(k / kVQueue) & 1u)) {
            ok = false;
            return -1;
        }
        return S.chunk[slot];
    };

    if (w == 6) {
        // ------------------------------------------------ scheduler (whole warp)
        int item = -1;
        for (int k = 0;; k++) {
            // next chunk: global index of its first tile, -1 when no tile is left
            long long c0 = -2;
            if (lane == 0) {
                for (;;) {
                    if (item >= 0) {
                        const int c = atomicAdd(&a.tile_next[item], kVChunk);
                        if (c < ntl) {
                            c0 = (long long)item * ntl + c;
                            break;
                        }
                    }
                    const int nx = atomicAdd(a.item_next, 1);
                    if (nx >= a.nitem) break;       // every item is open: help below
                    item = nx;
                }
            }
            c0 = __shfl_sync(kFull, c0, 0);
            item = __shfl_sync(kFull, item, 0);
            if (c0 == -2) {
                // take tiles left in any item: 32 counters per round, in parallel
                c0 = -1;
                const int from = max(item, 0);
                for (int base = 0; base < a.nitem && c0 < 0; base += 32) {
                    const int cand = (from + 1 + base + lane) % a.nitem;
                    const bool has = base + lane < a.nitem &&
                                     *(volatile int *)&a.tile_next[cand] < ntl;
                    unsigned m = __ballot_sync(kFull, has);
                    while (m != 0u && c0 < 0) {
                        const int src = __ffs(m) - 1;
                        m &= m - 1u;
                        const int cc = __shfl_sync(kFull, cand, src);
                        long long got = -1;
                        if (lane == 0) {
                            const int c = atomicAdd(&a.tile_next[cc], kVChunk);
                            if (c < ntl) got = (long long)cc * ntl + c;
                        }
                        got = __shfl_sync(kFull, got, 0);
                        if (got >= 0) {
                            c0 = got;
                            item = cc;
                        }
                    }
                }
            }
            int ok = 1;
            if (lane == 0) {
                const int slot = k % kVQueue;
                if (mbar_wait(&S.qfree[slot], ((uint32_t)(k / kVQueue) & 1u) ^ 1u)) {
                    S.chunk[slot] = c0;
                    mbar_arrive(&S.qfull[slot]);
                } else {
                    // nobody reads the queue any more: the others time out
                    atomicExch(&S.bad, 1);
                    ok = 0;
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok || c0 < 0) break;
        }
    } else if (w == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0, rloads = 0, cur_lg = -1;
            const uint64_t once = l2_policy_evict_first();
            int j = 0;
            for (int k = 0; ok; k++) {
                const long long c0 = take(k, ok);
                if (c0 < 0) break;
                const int lg = (int)c0 / ntl, t0 = (int)c0 - lg * ntl, t1 = min(ntl, t0 + kVChunk);
                for (int t = t0; t < t1 && ok; t++, j++) {
                    if (lg != cur_lg) {
                        // R of (layer, KV head) lg, once the MMAs reading the previous R are done
                        if (rloads > 0 && !mbar_wait(&S.rfree, (uint32_t)(rloads - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(&S.rfull, (uint32_t)(3 * kOp));
                        const unsigned char *src = a.pack + (size_t)lg * kPackBytes + kOp;
                        for (int q = 0; q < 3; q++) bulk_g2s(sm + q * kOp, src + q * kOp, kOp, &S.rfull);
                        rloads++;
                        cur_lg = lg;
                    }
                    const int s = j % kVStages;
                    if (!mbar_wait(&S.empty[s], Ring::stage_parity(j, kVStages) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&S.full[s], (uint32_t)kOp);
                    unsigned char *dst = ring + (size_t)s * kOp;
                    const int row = lg * N + t * kTk;
                    tma_2d_hint(dst, &tmV, 0, row, &S.full[s], once);
                    tma_2d_hint(dst + kUmmaBox, &tmV, 64, row, &S.full[s], once);
                    issued = j + 1;
                }
            }
            if (!ok) {
                atomicExch(&S.bad, 1);
                if (rloads > 0) mbar_wait(&S.rfull, (uint32_t)(rloads - 1) & 1u);
                for (int q = max(0, issued - kVStages); q < issued; q++)
                    mbar_wait(&S.full[q % kVStages], Ring::stage_parity(q, kVStages));
            }
        }
    } else if (w == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            int j = 0, rloads = 0, cur_lg = -1;
            for (int k = 0; ok; k++) {
                const long long c0 = take(k, ok);
                if (c0 < 0) break;
                const int lg = (int)c0 / ntl, t0 = (int)c0 - lg * ntl, t1 = min(ntl, t0 + kVChunk);
                for (int t = t0; t < t1; t++, j++) {
                    if (lg != cur_lg) {
                        if (rloads > 0) umma_commit(&S.rfree);   // the previous R is free once these complete
                        if (!mbar_wait(&S.rfull, (uint32_t)rloads & 1u)) {
                            ok = false;
                            break;
                        }
                        rloads++;
                        cur_lg = lg;
                    }
                    const int s = j % kVStages, b = j % kAcc;
                    if (!mbar_wait(&S.full[s], Ring::stage_parity(j, kVStages)) ||
                        !mbar_wait(&S.acce[b], Ring::acc_parity(j) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(b * 128);
                    const uint32_t tile = ring_s + (uint32_t)(s * kOp);
                    const uint64_t dv = umma_sdesc(tile);
#pragma unroll
                    for (int sp = 0; sp < 3; sp++) {
                        const uint64_t dr = umma_sdesc(r_s + (uint32_t)(sp * kOp));
#pragma unroll
                        for (int ks = 0; ks < 8; ks++)
                            umma_bf16(d, umma_sdesc_step(dv, ks), umma_sdesc_step(dr, ks), kIdesc,
                                      sp > 0 || ks > 0);
                    }
                    umma_commit(&S.accf[b]);
                    umma_commit(&S.empty[s]);
                }
            }
            umma_commit(&S.fin);
            if (!mbar_wait(&S.fin, 0)) ok = false;
            if (!ok) atomicExch(&S.bad, 1);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int qd = w & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        bool good = true;
        int j = 0;
        for (int k = 0; good; k++) {
            bool ok = good;
            const long long c0 = take(k, ok);
            good = __all_sync(kFull, ok);
            if (!good || c0 < 0) break;
            const int lg = (int)c0 / ntl, t0 = (int)c0 - lg * ntl, t1 = min(ntl, t0 + kVChunk);
            for (int t = t0; t < t1; t++, j++) {
                const int b = j % kAcc;
                ok = good && mbar_wait(&S.accf[b], Ring::acc_parity(j));
                good = __all_sync(kFull, ok);
                if (good) {
                    tc_fence_after();
                    float x[128];
                    tmem_ld128(lane_base + (uint32_t)(b * 128), x);
                    float r2[8];
#pragma unroll
                    for (int q = 0; q < 8; q++) r2[q] = x[q] * x[q];
#pragma unroll
                    for (int e = 8; e < 128; e++) r2[e & 7] = fmaf(x[e], x[e], r2[e & 7]);
                    const int key = t * kTk + 32 * qd + lane;
                    if (key < N)
                        a.r2[(size_t)lg * N + key] =
                            ((r2[0] + r2[1]) + (r2[2] + r2[3])) + ((r2[4] + r2[5]) + (r2[6] + r2[7]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && good) mbar_arrive(&S.acce[b]);
            }
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.qfree[k % kVQueue]);
        }
        if (!good) atomicExch(&S.bad, 1);
    }
    __syncthreads();
    if (w == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && S.bad)
        for (int l = 0; l < a.NL; l++)     // NaN: a wait timed out
            a.layer_sum[l] = __longlong_as_double(0x7ff8000000000000ll);
}

// --------------------------------------------------------------- operands
// Per (layer, KV head): the 128 window rows (row 4 j + h = query head h of
// the group at window position j; zero past the window) and the three bf16
// terms of the factor R (hi + mid + lo carries its fp32 value), each a
// 128 x 128 K-major tile in the layout of a 128-byte-swizzled TMA load.
__global__ void __launch_bounds__(256) pack_kernel(const uint16_t *q, const float *R,
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
    if (R == nullptr) return;                // window attention only: no value-norm factor
    const float *G0 = R + (size_t)lg * kD * kD;
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

// --------------------------------------------------------------- factor
// One CTA per (layer, KV head).  Phase 1: Gram = W_g W_g^T in fp64, thread
// (ta, tb) owning the 8 x 8 block at rows 8 ta, columns 8 tb, the columns of
// W_g (fp32 sums of the group's bf16 W_O entries) taken 32 at a time.
// Phase 2: pivoted Cholesky of Gram in fp64 (outer-product form, the largest
// remaining diagonal as pivot; stops when that falls to d * eps * the largest
// diagonal, the rest of the factor being zero).  Step k gives the column l_k
// of F with F F^T = Gram, written as row k of R = F^T, so that
// ||v W_g||^2 = v Gram v^T = ||R v^T||^2.
constexpr size_t kFacSmem = (size_t)kD * kD * 8 + (size_t)kD * 8;

__global__ void __launch_bounds__(256) factor_kernel(const uint16_t *W, float *R, int Hq, int Hkv,
                                                     int D)
{
    extern __shared__ __align__(16) unsigned char fsm[];
    double *A = reinterpret_cast<double *>(fsm);     // Gram, then its Schur complements
    double *lk = A + kD * kD;                         // current factor column
    __shared__ float Wc[kD][33];
    __shared__ int done[kD];
    __shared__ int piv;
    __shared__ double pd, tol;
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
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) A[(8 * ta + i) * kD + 8 * tb + j] = acc[i][j];
    if (tid < kD) done[tid] = 0;
    __syncthreads();

    float *Rg = R + (size_t)lg * kD * kD;
    bool live = true;
    for (int k = 0; k < kD; k++) {
        if (tid < 32) {
            // largest remaining diagonal (ties to the smaller index)
            double best = -1.0;
            int bi = kD;
            for (int i = tid; i < kD; i += 32)
                if (!done[i] && A[i * kD + i] > best) { best = A[i * kD + i]; bi = i; }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                const double ob = __shfl_xor_sync(kFull, best, m);
                const int oi = __shfl_xor_sync(kFull, bi, m);
                if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
            }
            if (tid == 0) {
                piv = bi;
                pd = best;
                if (k == 0) tol = (double)kD * 2.220446049250313e-16 * fmax(best, 0.0);
            }
        }
        __syncthreads();
        const int p = piv;
        live = live && pd > tol && p < kD;
        const double inv = live ? 1.0 / sqrt(pd) : 0.0;
        if (tid < kD) {
            const double v = (live && !done[tid]) ? A[tid * kD + p] * inv : 0.0;
            lk[tid] = v;
            Rg[(size_t)k * kD + tid] = (float)v;
        }
        __syncthreads();
        if (tid == 0 && p < kD) done[p] = 1;
        if (live)
            for (int e = tid; e < kD * kD; e += blockDim.x) {
                const double li = lk[e >> 7];
                if (li != 0.0) A[e] = fma(-li, lk[e & (kD - 1)], A[e]);
            }
        __syncthreads();
    }
}

// --------------------------------------------------------------- top-K
// Radix select of the B_total largest scores over an order key that ascends
// as the score descends: three passes over the 32-bit key (bits 31-20, 19-8,
// 7-0).  Pass k histograms the keys that match the digits picked so far; the
// last block of the pass to finish picks the next digit (the bin holding
// the element of the wanted rank) for the next pass.
struct SelState {
    int d[3];              // digits picked by passes 1-3
    long long r[3];        // rank of the wanted element inside the picked bin
    unsigned done[3];      // blocks finished per pass
    uint32_t thr;          // order key of the B_total-th largest score
    long long need;        // elements taken from the group of keys equal to thr
};

constexpr int kTkBlock = 1024;
constexpr int kTkPer = 4;                 // elements per thread
constexpr int kTkSpan = kTkBlock * kTkPer;
constexpr int kH1 = 4096, kH2 = 4096, kH3 = 256;

// order key: ascending key = descending score
__device__ __forceinline__ uint32_t desc_key(float s) { return ~float_key(s); }

// LaProx's indicator p_i = c_i r_i, written over the column norms c, and the
// per-layer sums of p (fp32 within a thread, fp64 across threads).  Grid
// (blocks per layer, NL); block b of layer l strides over the layer's Hkv N
// scores.
constexpr int kCbBlock = 256;
constexpr unsigned kPauseNs = 10000;   // head start of the attention kernel over the value norms
__global__ void __launch_bounds__(kCbBlock) combine_kernel(float *p, const float *r2,
                                                           double *layer_sum, int per_layer)
{
    const int l = blockIdx.y, lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    float *pl = p + (size_t)l * per_layer;
    const float *rl = r2 + (size_t)l * per_layer;
    float part = 0.f;
#pragma unroll 4
    for (int i = blockIdx.x * kCbBlock + threadIdx.x; i < per_layer; i += gridDim.x * kCbBlock) {
        const float v = pl[i] * sqrtf(rl[i]);
        pl[i] = v;
        part += v;
    }
    double d = (double)part;
#pragma unroll
    for (int msk = 16; msk > 0; msk >>= 1) d += __shfl_xor_sync(kFull, d, msk);
    __shared__ double wsum[kCbBlock / 32];
    if (lane == 0) wsum[wp] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int k = 0; k < kCbBlock / 32; k++) t += wsum[k];
        if (t != 0.0) atomicAdd(&layer_sum[l], t);
    }
}

// A pause of about ns nanoseconds (one warp, no shared memory, at most ~1 ms
// whatever the clock does), queued ahead of the value-norm launch so that the
// attention kernel's clusters, made eligible at the same moment, are placed
// first; the value-norm CTAs then start on the SMs the clusters leave free.
__global__ void pause_kernel(unsigned ns)
{
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (int i = 0; i < 4096; i++) {
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 >= ns) break;
        __nanosleep(256);
    }
}

// inv[l] = 1 / (sum of p over layer l), 0 for an all-zero layer
__global__ void layer_inv_kernel(const double *layer_sum, float *inv, int NL)
{
    for (int l = threadIdx.x; l < NL; l += blockDim.x) {
        const double z = layer_sum[l];
        inv[l] = z > 0.0 ? (float)(1.0 / z) : (z == 0.0 ? 0.f : __int_as_float(0x7fc00000));
    }
}

// Bin of a histogram (n bins, ascending order key) holding the element of
// 0-based rank `rank`, and that element's rank inside the bin; whole block.
// kGlobal: the histogram is in global memory (other blocks' atomics, read
// through L2); otherwise in this block's shared memory.
template <bool kGlobal = true>
__device__ void block_pick(const unsigned *hist, int n, long long rank, int *scan, int *bin_out,
                           long long *rin_out)
{
    auto ld = [&](int b) -> unsigned { return kGlobal ? __ldcg(hist + b) : hist[b]; };
    __shared__ int sb;
    __shared__ long long sr;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int b0 = threadIdx.x * per;
    if (threadIdx.x == 0) {
        sb = 0;
        sr = 0;
    }
    int loc = 0;
    for (int k = 0; k < per; k++)
        if (b0 + k < n) loc += (int)ld(b0 + k);
    int total;
    const int ex = block_exscan(loc, scan, &total);
    if (ex <= rank && rank < (long long)ex + loc) {
        long long cum = ex;
        for (int k = 0; k < per; k++) {
            const long long h = ld(b0 + k);
            if (cum + h > rank) {
                sb = b0 + k;
                sr = rank - cum;
                break;
            }
            cum += h;
        }
    }
    __syncthreads();
    *bin_out = sb;
    *rin_out = sr;
    __syncthreads();
}

// warp-aggregated shared-memory histogram increment (bin < 0: no element);
// every lane of the warp calls it
__device__ __forceinline__ void hist_add(unsigned *h, int bin)
{
    const unsigned same = __match_any_sync(kFull, bin);
    if (bin >= 0 && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&h[bin], (unsigned)__popc(same));
}

// Pass kPass of the select.  Pass 1 also normalizes in place (s = p inv[l]).
template <int kPass>
__global__ void __launch_bounds__(kTkBlock) sel_pass_kernel(float *s, int M, const float *inv,
                                                              int per_layer, int normalize,
                                                              unsigned *hist, long long rank0,
                                                              SelState *ss)
{
    constexpr int NB = kPass == 3 ? kH3 : kH1;
    __shared__ unsigned h[NB];
    __shared__ int scan[40];
    __shared__ int last;
    const uint32_t pre = kPass == 1 ? 0u
                       : kPass == 2 ? (uint32_t)ss->d[0]
                                    : (((uint32_t)ss->d[0] << 12) | (uint32_t)ss->d[1]);
    for (int i = threadIdx.x; i < NB; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long base = (long long)blockIdx.x * blockDim.x; base < M; base += 4 * stride) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {        // four loads in flight
            const long long i = base + u * stride + threadIdx.x;
            v[u] = i < M ? s[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const long long i = base + u * stride + threadIdx.x;
            int bin = -1;
            if (i < M) {
                if (kPass == 1 && normalize) {
                    v[u] *= inv[(int)i / per_layer];
                    s[i] = v[u];
                }
                const uint32_t k = desc_key(v[u]);
                if (kPass == 1) bin = (int)(k >> 20);
                else if (kPass == 2) { if ((k >> 20) == pre) bin = (int)((k >> 8) & (kH2 - 1)); }
                else if ((k >> 8) == pre) bin = (int)(k & (kH3 - 1));
            }
            hist_add(h, bin);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NB; i += blockDim.x)
        if (h[i]) atomicAdd(&hist[i], h[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(&ss->done[kPass - 1], 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    // the last block: every block's counts are in; pick this pass's digit
    __threadfence();
    int d;
    long long r;
    block_pick(hist, NB, kPass == 1 ? rank0 : ss->r[kPass - 2], scan, &d, &r);
    if (threadIdx.x == 0) {
        ss->d[kPass - 1] = d;
        ss->r[kPass - 1] = r;
        if (kPass == 3) {
            ss->thr = ((uint32_t)ss->d[0] << 20) | ((uint32_t)ss->d[1] << 8) | (uint32_t)d;
            ss->need = r + 1;
        }
    }
}

// per block of kTkSpan elements (4 consecutive per thread): elements below
// the threshold key and equal to it
__global__ void __launch_bounds__(kTkBlock) topk_count_kernel(const float *s, int M,
                                                               const SelState *ss, int *lt, int *eq)
{
    __shared__ int scan[40];
    const uint32_t thr = ss->thr;
    const long long i0 = (long long)blockIdx.x * kTkSpan + kTkPer * threadIdx.x;
    int nlt = 0, neq = 0;
#pragma unroll
    for (int u = 0; u < kTkPer; u++)
        if (i0 + u < M) {
            const uint32_t key = desc_key(s[i0 + u]);
            nlt += key < thr;
            neq += key == thr;
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
                                                              const SelState *ss, int64_t *eq_off,
                                                              int64_t *keep_off)
{
    __shared__ int scan[40];
    __shared__ int64_t carry[2];
    if (threadIdx.x == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    const int64_t need = ss->need;
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

// keep mask, per-(layer, KV head) counts and ascending kept indices; equal
// keys are kept in flat order up to `need`
__global__ void __launch_bounds__(kTkBlock) topk_write_kernel(const float *s, int M, int N,
                                                               const SelState *ss,
                                                               const int64_t *eq_off,
                                                               const int64_t *keep_off,
                                                               uint8_t *keep, int *counts,
                                                               int64_t *idx)
{
    __shared__ int scan[40];
    const uint32_t thr = ss->thr;
    const int64_t need = ss->need;
    const long long i0 = (long long)blockIdx.x * kTkSpan + kTkPer * threadIdx.x;
    uint32_t key[kTkPer];
    int neq = 0;
#pragma unroll
    for (int u = 0; u < kTkPer; u++) {
        key[u] = i0 + u < M ? desc_key(s[i0 + u]) : 0xffffffffu;
        neq += i0 + u < M && key[u] == thr;
    }
    int teq;
    int64_t er = eq_off[blockIdx.x] + block_exscan(neq, scan, &teq);   // tie rank of my first equal key
    bool kp[kTkPer];
    int nk = 0;
#pragma unroll
    for (int u = 0; u < kTkPer; u++) {
        const bool in = i0 + u < M;
        const bool iseq = in && key[u] == thr;
        kp[u] = in && (key[u] < thr || (iseq && er < need));
        er += iseq;
        nk += kp[u];
    }
    int tk;
    int64_t ko = keep_off[blockIdx.x] + block_exscan(nk, scan, &tk);
#pragma unroll
    for (int u = 0; u < kTkPer; u++) {
        if (i0 + u < M) keep[i0 + u] = (uint8_t)kp[u];
        if (kp[u]) {
            if (idx) idx[ko++] = i0 + u;
            if (counts) atomicAdd(&counts[(i0 + u) / N], 1);
        }
    }
}

// Segmented selection for the LaProx allocation ablation: one block per
// segment (a layer for head-flatten only, a (layer, KV head) for the uniform
// allocation) keeps its kseg largest scores.  The same three radix passes
// as the global select, on shared-memory histograms (pass 1 also
// normalizes in place), then one ordered pass over the segment: equal keys
// are kept in flat order (tie rank carried across chunks) and the kept flat
// indices land in ascending order in idx[segment * kseg ...].
constexpr int kSegMaxHeads = 64;          // KV heads a layer segment may span
__global__ void __launch_bounds__(kTkBlock) seg_select_kernel(float *s, int N, int seg_len, int kseg,
                                                               int per_layer, const float *inv,
                                                               int normalize, uint8_t *keep,
                                                               int *counts, int64_t *idx)
{
    __shared__ unsigned h[kH1];
    __shared__ int scan[40];
    __shared__ int cnt[kSegMaxHeads];
    __shared__ long long carry[2];
    const int q = blockIdx.x, tid = threadIdx.x;
    const int64_t base = (int64_t)q * seg_len;
    float *sg = s + base;
    const float sc = normalize ? inv[(int)(base / per_layer)] : 1.f;
    const int head0 = (int)(base / N), nheads = seg_len / N;
    for (int i = tid; i < kSegMaxHeads; i += blockDim.x) cnt[i] = 0;
    if (kseg == 0) {                         // nothing kept: scale and clear only
        for (int i = tid; i < seg_len; i += blockDim.x) {
            if (normalize) sg[i] *= sc;
            keep[base + i] = 0;
        }
        __syncthreads();
        if (counts)
            for (int g = tid; g < nheads; g += blockDim.x) counts[head0 + g] = 0;
        return;
    }
    uint32_t pre = 0;                        // digits picked so far
    long long rank = kseg - 1;               // 0-based rank of the kseg-th largest
    for (int pass = 1; pass <= 3; pass++) {
        const int NB = pass == 3 ? kH3 : kH1;
        for (int i = tid; i < NB; i += blockDim.x) h[i] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < seg_len; i0 += 4 * kTkBlock) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {        // four loads in flight
                const int i = i0 + u * kTkBlock + tid;
                v[u] = i < seg_len ? sg[i] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int i = i0 + u * kTkBlock + tid;
                int bin = -1;
                if (i < seg_len) {
                    if (pass == 1 && normalize) {
                        v[u] *= sc;
                        sg[i] = v[u];
                    }
                    const uint32_t k = desc_key(v[u]);
                    if (pass == 1) bin = (int)(k >> 20);
                    else if (pass == 2) { if ((k >> 20) == pre) bin = (int)((k >> 8) & (kH2 - 1)); }
                    else if ((k >> 8) == pre) bin = (int)(k & (kH3 - 1));
                }
                hist_add(h, bin);
            }
        }
        __syncthreads();
        int d;
        long long r;
        block_pick<false>(h, NB, rank, scan, &d, &r);
        rank = r;
        pre = pass == 3 ? ((pre << 8) | (uint32_t)d) : ((pre << 12) | (uint32_t)d);
    }
    const uint32_t thr = pre;                // order key of the kseg-th largest score
    const long long need = rank + 1;         // keys equal to thr that are kept
    if (tid == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    for (int c0 = 0; c0 < seg_len; c0 += kTkSpan) {
        const int i0 = c0 + kTkPer * tid;
        uint32_t key[kTkPer];
        int neq = 0;
#pragma unroll
        for (int u = 0; u < kTkPer; u++) {
            key[u] = i0 + u < seg_len ? desc_key(sg[i0 + u]) : 0xffffffffu;
            neq += i0 + u < seg_len && key[u] == thr;
        }
        int teq;
        long long er = carry[0] + block_exscan(neq, scan, &teq);
        bool kp[kTkPer];
        int nk = 0;
#pragma unroll
        for (int u = 0; u < kTkPer; u++) {
            const bool in = i0 + u < seg_len;
            const bool iseq = in && key[u] == thr;
            kp[u] = in && (key[u] < thr || (iseq && er < need));
            er += iseq;
            nk += kp[u];
        }
        int tk;
        long long ko = carry[1] + block_exscan(nk, scan, &tk);
#pragma unroll
        for (int u = 0; u < kTkPer; u++) {
            if (i0 + u < seg_len) keep[base + i0 + u] = (uint8_t)kp[u];
            if (kp[u]) {
                if (idx && ko < kseg) idx[(int64_t)q * kseg + ko] = base + i0 + u;
                ko++;
                atomicAdd(&cnt[(i0 + u) / N], 1);
            }
        }
        __syncthreads();
        if (tid == 0) {
            carry[0] += teq;
            carry[1] += tk;
        }
        __syncthreads();
    }
    if (counts)
        for (int g = tid; g < nheads; g += blockDim.x) counts[head0 + g] = cnt[g];
}

// SnapKV's scores under MomentKV's prefill protocol: each block of `pool`
// consecutive positions of a (layer, KV head) takes the mean of its tokens'
// accumulated window attention, and position 0 (the attention sink) scores
// +infinity when sink != 0.  One thread per token.
__global__ void snapkv_pool_kernel(const float *acc, float *s, int N, int pool, int sink,
                                   int64_t M)
{
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= M) return;
    const int i = (int)(e % N);
    const int64_t row = e - i;
    const int b0 = i - i % pool, b1 = min(N, b0 + pool);
    float m = 0.f;
    for (int j = b0; j < b1; j++) m += acc[row + j];
    m /= (float)(b1 - b0);
    s[e] = (sink && i == 0) ? __int_as_float(0x7f800000) : m;
}

struct PfWs {
    float *p;
    double *layer_sum;
    float *inv;
    float *r2;
    int *counter;                // [0]: next unopened item, [1 + i]: next tile of item i
    unsigned char *pack;
    float2 *stats;
    SelState *st;
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
    w.inv = reinterpret_cast<float *>(take((size_t)NL * 4));
    w.r2 = reinterpret_cast<float *>(take((size_t)M * 4));
    w.counter = reinterpret_cast<int *>(take((size_t)(NL * Hkv + 1) * 4));
    w.pack = reinterpret_cast<unsigned char *>(take((size_t)NL * Hkv * kPackBytes));
    w.stats = reinterpret_cast<float2 *>(take((size_t)NL * Hkv * kCS * kASets * kRows * sizeof(float2)));
    w.st = reinterpret_cast<SelState *>(take(sizeof(SelState)));
    w.hist = reinterpret_cast<unsigned *>(take((size_t)(kH1 + kH2 + kH3) * 4));
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

// Identity of the calling thread's current context (cuCtxGetId, through the
// runtime's driver entry points): unique for the process's lifetime, so a
// context made after a device reset, or another context made current, gets
// an id of its own.  0 when the entry points are unavailable.
static unsigned long long current_context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur && get_id && get_cur(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// One library-owned stream per (context, device), created on first use at
// the lowest priority, non-blocking and never destroyed, for work that runs
// beside the caller's stream; it joins the caller's stream through events,
// so a stream capture follows it.  Keyed on the context id, a stream made in
// a context that has since been destroyed is never handed out again.
static cudaError_t side_stream(int dev, cudaStream_t *out)
{
    struct Entry {
        unsigned long long ctx;
        int dev;
        cudaStream_t s;
    };
    constexpr int kMax = 64;
    static Entry tab[kMax] = {};
    static int used = 0, next = 0;
    static std::mutex mu;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; i++)
        if (tab[i].ctx == ctx && tab[i].dev == dev) {
            *out = tab[i].s;
            return cudaSuccess;
        }
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e != cudaSuccess) return e;
    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, lo);
    if (e != cudaSuccess) return e;
    // a full table forgets its oldest entry (the stream stays valid)
    const int slot = used < kMax ? used++ : (next++ % kMax);
    tab[slot] = Entry{ctx, dev, s};
    *out = s;
    return cudaSuccess;
}

// Two events for a fork and a join, destroyed with the call (a recorded
// event's resources are released once it completes).
struct EventPair {
    cudaEvent_t a = nullptr, b = nullptr;
    cudaError_t create()
    {
        cudaError_t e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
        return e;
    }
    ~EventPair()
    {
        if (a) cudaEventDestroy(a);
        if (b) cudaEventDestroy(b);
    }
};

// The persistent attention kernel: as many 8-CTA clusters as the GPU holds
// at once, each looping over (layer, KV head) items.
static cudaError_t launch_attn(const AttnArgs &aa, const CUtensorMap &tmK, int nitem, int nsm,
                               cudaStream_t st, int priority = 0)
{
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kADyn);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kAThreads);
    cfg.dynamicSmemBytes = kADyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributePriority;
    attr[1].val.priority = priority;
    cfg.attrs = attr;
    cfg.numAttrs = 1;            // the occupancy query sees the cluster shape only
    cfg.gridDim = dim3(kCS * std::min(nitem, std::max(1, nsm / kCS)));
    int nclu = 0;
    if (cudaOccupancyMaxActiveClusters(&nclu, prefill_attn_kernel, &cfg) != cudaSuccess || nclu < 1)
        nclu = std::max(1, nsm / (2 * kCS));
    (void)cudaGetLastError();
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(kCS * std::min(nitem, nclu));
    return cudaLaunchKernelEx(&cfg, prefill_attn_kernel, aa, tmK);
}

// Window attention shared by kvc_prefill_window_attention and
// kvc_prefill_snapkv: checks, pack (window queries only) and the attention
// kernel writing the weighted column sums into S.
static kvc_status window_colsum(const char *who, int32_t NL, int32_t Hq, int32_t Hkv, int32_t d,
                                int32_t N, int32_t w, const float *row_weight,
                                const uint16_t *q_win, const uint16_t *K, float *S, void *ws,
                                size_t ws_bytes, cudaStream_t st)
{
    PF_CHECK(NL >= 1 && Hkv >= 1 && N >= 1 && w >= 1, KVC_ERR_INVALID_ARG,
             "%s: NL, Hkv, N, w must be >= 1", who);
    PF_CHECK(d == kD, KVC_ERR_UNSUPPORTED, "%s: d = %d unsupported", who, d);
    PF_CHECK(Hq == kPG * Hkv, KVC_ERR_UNSUPPORTED,
             "%s: only 4 query heads per KV head are supported (Hq = %d, Hkv = %d)", who, Hq, Hkv);
    PF_CHECK(w <= 32 && w <= N, KVC_ERR_UNSUPPORTED, "%s: window w = %d must be <= 32 and <= N",
             who, w);
    PF_CHECK(q_win && K && S && row_weight, KVC_ERR_INVALID_ARG,
             "%s: q_win, K, the row weights and the output are required", who);
    PF_CHECK(((uintptr_t)K & 15u) == 0 && ((uintptr_t)q_win & 3u) == 0, KVC_ERR_INVALID_ARG,
             "%s: K must be 16-byte aligned, q_win 4-byte", who);
    PfWs pw = pf_layout(NL, Hkv, N, nullptr);
    PF_CHECK(ws != nullptr && ws_bytes >= pw.bytes && ((uintptr_t)ws & 255u) == 0, KVC_ERR_WORKSPACE,
             "%s: workspace of %zu bytes (256-byte aligned) required", who, pw.bytes);
    pw = pf_layout(NL, Hkv, N, ws);
    const uint64_t rows = (uint64_t)NL * Hkv * N;
    PF_CHECK(rows + kTk < (1ull << 31), KVC_ERR_UNSUPPORTED, "%s: too many rows", who);
    CUtensorMap tmK;
    PF_CHECK(make_row_map(&tmK, K, rows, kTk), KVC_ERR_CUDA, "%s: tensor map encoding failed", who);
    int dev = 0, nsm = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return pf_cuda(e, who);
    kvc_status s = pf_cuda(cudaMemsetAsync(pw.layer_sum, 0, (size_t)NL * 8, st), "memset");
    if (s != KVC_OK) return s;
    pack_kernel<<<NL * Hkv, 256, 0, st>>>(q_win, nullptr, pw.pack, Hq, Hkv, w);
    if ((e = cudaGetLastError()) != cudaSuccess) return pf_cuda(e, who);
    const int per_cta = ((N + kCS - 1) / kCS + kTk - 1) / kTk * kTk;
    AttnArgs aa{pw.pack, nullptr, pw.stats, pw.layer_sum, S, Hkv, N, w, per_cta, NL * Hkv, 0,
                (float)(1.4426950408889634 / sqrt((double)kD)), {}};
    for (int j = 0; j < 32; j++) aa.roww[j] = j < w ? row_weight[j] : 0.f;
    return pf_cuda(launch_attn(aa, tmK, NL * Hkv, nsm, st), who);
}

extern "C" {

kvc_status kvc_prefill_prepare(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t D,
                               const uint16_t *W_O, float *R, void *stream)
{
    PF_CHECK(NL >= 1 && Hq >= 1 && Hkv >= 1 && D >= 1, KVC_ERR_INVALID_ARG,
             "kvc_prefill_prepare: NL, Hq, Hkv, D must be >= 1");
    PF_CHECK(d == kD, KVC_ERR_UNSUPPORTED, "kvc_prefill_prepare: d = %d unsupported", d);
    PF_CHECK(Hq % Hkv == 0, KVC_ERR_INVALID_ARG, "kvc_prefill_prepare: Hq %% Hkv != 0");
    PF_CHECK(W_O && R, KVC_ERR_INVALID_ARG, "kvc_prefill_prepare: NULL pointer");
    cudaError_t e = cudaFuncSetAttribute(factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFacSmem);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_prepare attribute");
    factor_kernel<<<NL * Hkv, 256, kFacSmem, static_cast<cudaStream_t>(stream)>>>(W_O, R, Hq, Hkv, D);
    return pf_cuda(cudaGetLastError(), "kvc_prefill_prepare launch");
}

size_t kvc_prefill_workspace_size(int32_t NL, int32_t Hkv, int32_t N, int64_t B_total)
{
    (void)B_total;
    if (NL < 1 || Hkv < 1 || N < 1) return 0;
    return pf_layout(NL, Hkv, N, nullptr).bytes;
}

kvc_status kvc_prefill_score(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t N,
                             int32_t w, int64_t B_total, int32_t normalize, int32_t alloc,
                             const uint16_t *q_win,
                             const uint16_t *K, const uint16_t *V, const float *R,
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
    PF_CHECK(alloc >= KVC_ALLOC_GLOBAL && alloc <= KVC_ALLOC_HEAD, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: alloc = %d unknown", alloc);
    const int64_t nseg = alloc == KVC_ALLOC_GLOBAL ? 1 : alloc == KVC_ALLOC_LAYER ? NL : (int64_t)NL * Hkv;
    PF_CHECK(B_total % nseg == 0, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: B_total = %lld is not a multiple of the %lld segments",
             (long long)B_total, (long long)nseg);
    PF_CHECK(alloc != KVC_ALLOC_LAYER || Hkv <= kSegMaxHeads, KVC_ERR_UNSUPPORTED,
             "kvc_prefill_score: per-layer allocation supports up to %d KV heads", kSegMaxHeads);
    const int per_cta = ((N + kCS - 1) / kCS + kTk - 1) / kTk * kTk;
    PF_CHECK(q_win && K && V && R && keep, KVC_ERR_INVALID_ARG,
             "kvc_prefill_score: q_win, K, V, R and keep are required");
    PF_CHECK(((uintptr_t)K & 15u) == 0 && ((uintptr_t)V & 15u) == 0 && ((uintptr_t)R & 15u) == 0 &&
                 ((uintptr_t)q_win & 3u) == 0,
             KVC_ERR_INVALID_ARG, "kvc_prefill_score: K, V, R must be 16-byte aligned, q_win 4-byte");
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
    s = pf_cuda(cudaMemsetAsync(pw.st, 0, sizeof(SelState), st), "memset");
    if (s != KVC_OK) return s;
    s = pf_cuda(cudaMemsetAsync(pw.hist, 0, (size_t)(kH1 + kH2 + kH3) * 4, st), "memset");
    if (s != KVC_OK) return s;
    s = pf_cuda(cudaMemsetAsync(pw.counter, 0, (size_t)(NL * Hkv + 1) * 4, st), "memset");
    if (s != KVC_OK) return s;
    if (counts) {
        s = pf_cuda(cudaMemsetAsync(counts, 0, (size_t)NL * Hkv * 4, st), "memset");
        if (s != KVC_OK) return s;
    }

    pack_kernel<<<NL * Hkv, 256, 0, st>>>(q_win, R, pw.pack, Hq, Hkv, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score pack launch");
    // The value norms r^2 (a library stream) and the attention column norms c
    // (the caller's stream) run side by side: the attention kernel's
    // clusters cannot fill every SM, and the value-norm CTAs take the SMs
    // left over, then the rest once the clusters finish.  Then p = c r with
    // the per-layer sums.
    const int ntl = (N + kTk - 1) / kTk;
    const long long total = (long long)NL * Hkv * ntl;
    int dev = 0, nsm = 0, prio_lo = 0, prio_hi = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi)) != cudaSuccess)
        return pf_cuda(e, "kvc_prefill_score device query");
    e = cudaFuncSetAttribute(prefill_val_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kVDyn);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score attribute");
    cudaStream_t aux = nullptr;
    if ((e = side_stream(dev, &aux)) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score stream");
    EventPair ev;
    if ((e = ev.create()) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score event");
    const int nitem = NL * Hkv;
    // the attention kernel is enqueued first and at the higher priority, so
    // its clusters are placed before the value-norm CTAs take SMs
    if ((e = cudaEventRecord(ev.a, st)) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score record");
    AttnArgs aa{pw.pack, pbuf, pw.stats, pw.layer_sum, nullptr, Hkv, N, w, per_cta, nitem, 1,
                (float)(1.4426950408889634 / sqrt((double)kD)), {}};
    e = launch_attn(aa, tmK, nitem, nsm, st, prio_hi);
    if (e != cudaSuccess) return pf_cuda(e, "kvc_prefill_score attention launch");
    if ((e = cudaStreamWaitEvent(aux, ev.a, 0)) != cudaSuccess)
        return pf_cuda(e, "kvc_prefill_score stream wait");
    pause_kernel<<<1, 32, 0, aux>>>(kPauseNs);
    ValArgs va{pw.pack, pw.r2, pw.layer_sum, pw.counter, pw.counter + 1, NL, N, ntl, nitem};
    prefill_val_kernel<<<(unsigned)std::min<long long>((total + kVChunk - 1) / kVChunk, nsm), kVThreads,
                         kVDyn, aux>>>(va, tmV);
    if ((e = cudaGetLastError()) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score value launch");
    if ((e = cudaEventRecord(ev.b, aux)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, ev.b, 0)) != cudaSuccess)
        return pf_cuda(e, "kvc_prefill_score stream join");
    const int per_layer_i = Hkv * N;
    combine_kernel<<<dim3((unsigned)std::min(64, (per_layer_i + kCbBlock * 32 - 1) / (kCbBlock * 32)),
                          (unsigned)NL),
                     kCbBlock, 0, st>>>(pbuf, pw.r2, pw.layer_sum, per_layer_i);
    if ((e = cudaGetLastError()) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score combine launch");
    const int64_t per_layer = (int64_t)Hkv * N;

    // radix select of the B_total largest s (pass 1 also normalizes in place)
    if (normalize) layer_inv_kernel<<<1, 256, 0, st>>>(pw.layer_sum, pw.inv, NL);
    if (alloc != KVC_ALLOC_GLOBAL) {
        const int seg_len = (int)(M / nseg);
        seg_select_kernel<<<(unsigned)nseg, kTkBlock, 0, st>>>(pbuf, N, seg_len, (int)(B_total / nseg),
                                                              (int)per_layer, pw.inv, normalize, keep,
                                                              counts, idx);
        return pf_cuda(cudaGetLastError(), "kvc_prefill_score segmented select launch");
    }
    const int sel_grid = (int)std::min<int64_t>((M + kTkBlock - 1) / kTkBlock, 2 * (int64_t)nsm);
    unsigned *h1 = pw.hist, *h2 = h1 + kH1, *h3 = h2 + kH2;
    const long long rank0 = B_total > 0 ? B_total - 1 : 0;
    sel_pass_kernel<1><<<sel_grid, kTkBlock, 0, st>>>(pbuf, (int)M, pw.inv, (int)per_layer, normalize, h1,
                                                      rank0, pw.st);
    if ((e = cudaGetLastError()) != cudaSuccess) return pf_cuda(e, "kvc_prefill_score select launch");
    if (B_total == 0) {
        s = pf_cuda(cudaMemsetAsync(keep, 0, (size_t)M, st), "memset");
        return s;
    }
    sel_pass_kernel<2><<<sel_grid, kTkBlock, 0, st>>>(pbuf, (int)M, pw.inv, (int)per_layer, 0, h2, rank0,
                                                      pw.st);
    sel_pass_kernel<3><<<sel_grid, kTkBlock, 0, st>>>(pbuf, (int)M, pw.inv, (int)per_layer, 0, h3, rank0,
                                                      pw.st);
    const int nblk = (int)((M + kTkSpan - 1) / kTkSpan);
    topk_count_kernel<<<nblk, kTkBlock, 0, st>>>(pbuf, (int)M, pw.st, pw.lt, pw.eq);
    topk_scan_kernel<<<1, kTkBlock, 0, st>>>(pw.lt, pw.eq, nblk, pw.st, pw.eq_off, pw.keep_off);
    topk_write_kernel<<<nblk, kTkBlock, 0, st>>>(pbuf, (int)M, N, pw.st, pw.eq_off, pw.keep_off, keep,
                                                 counts, idx);
    return pf_cuda(cudaGetLastError(), "kvc_prefill_score top-K launch");
}

kvc_status kvc_prefill_window_attention(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t N,
                                        int32_t w, const float *row_weight, const uint16_t *q_win,
                                        const uint16_t *K, float *S, void *ws, size_t ws_bytes,
                                        void *stream)
{
    return window_colsum("kvc_prefill_window_attention", NL, Hq, Hkv, d, N, w, row_weight, q_win,
                         K, S, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

kvc_status kvc_prefill_snapkv(int32_t NL, int32_t Hq, int32_t Hkv, int32_t d, int32_t N, int32_t w,
                              int64_t B_total, int32_t pool, int32_t sink, const uint16_t *q_win,
                              const uint16_t *K, float *scores, uint8_t *keep, int32_t *counts,
                              int64_t *idx, void *ws, size_t ws_bytes, void *stream)
{
    const char *who = "kvc_prefill_snapkv";
    PF_CHECK(NL >= 1 && Hkv >= 1 && N >= 1, KVC_ERR_INVALID_ARG, "%s: NL, Hkv, N must be >= 1", who);
    const int64_t M = (int64_t)NL * Hkv * N;
    PF_CHECK(B_total >= 0 && B_total <= M && B_total % NL == 0, KVC_ERR_INVALID_ARG,
             "%s: B_total = %lld must be a multiple of NL = %d in [0, %lld]", who,
             (long long)B_total, NL, (long long)M);
    PF_CHECK(pool >= 1 && pool <= 64, KVC_ERR_INVALID_ARG, "%s: pool = %d outside [1, 64]", who, pool);
    PF_CHECK(Hkv <= kSegMaxHeads, KVC_ERR_UNSUPPORTED,
             "%s: per-layer allocation supports up to %d KV heads", who, kSegMaxHeads);
    PF_CHECK(keep != nullptr, KVC_ERR_INVALID_ARG, "%s: keep is required", who);
    PF_CHECK(M < (1ll << 31), KVC_ERR_UNSUPPORTED, "%s: too many tokens", who);
    float ones[32];
    for (int j = 0; j < 32; j++) ones[j] = 1.f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // accumulated window attention into the workspace's score buffer
    PfWs pw = pf_layout(NL, Hkv, N, ws);
    kvc_status s = window_colsum(who, NL, Hq, Hkv, d, N, w, ones, q_win, K, pw.p, ws, ws_bytes, st);
    if (s != KVC_OK) return s;
    float *sc = scores ? scores : pw.r2;
    snapkv_pool_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(pw.p, sc, N, pool, sink, M);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return pf_cuda(e, who);
    // each layer keeps B_total / NL over its heads and tokens
    seg_select_kernel<<<(unsigned)NL, kTkBlock, 0, st>>>(sc, N, (int)(M / NL), (int)(B_total / NL),
                                                          (int)(M / NL), pw.inv, 0, keep, counts, idx);
    return pf_cuda(cudaGetLastError(), "kvc_prefill_snapkv select launch");
}

}  // extern "C"
