// kvc_fused.cu -- the steady-state decode step in one cluster kernel.
//
// Steady state: every unit enters with len = L, appends one token and evicts
// one slot.  One thread-block cluster of CS CTAs serves one unit; CTA r owns
// the slot range [r*chunk, min(L, (r+1)*chunk)).  Shared-memory partials are
// merged across the cluster through distributed shared memory; there is no
// global-memory round trip and no wait on another CTA other than the
// hardware cluster barrier.
//
// Non-refresh step (InertiaKV-Lazy): utilities are stale, so the victim is
// known before attention: it is the next entry of the victim queue written at
// the last refresh (the T lowest (utility, position) pairs of that step, in
// order), or, when the queue is not valid, the lowest scored slot.  The new
// token takes the victim's slot directly, so the pass over the L slots is
// already the retained set: f_R and Z_R come out directly.
//
// Refresh step: the pass covers the L slots plus the new token (a virtual
// slot L).  Head-mean probabilities (InertiaKV sec 3.1 eq 1) update the
// utilities (eqs 2-4); the T lowest pairs are selected; the first is the
// victim and the rest form the queue.  The victim's share is removed from the
// merged output by the eviction-error identity (KeepKV eq 3); when its mass
// exceeds 1/2 in some head the retained output is recomputed instead.
//
// Both: the victim is folded into the moments (West's weighted incremental
// update of the mean / covariance form), and the normalization correction of
// MomentKV sec 4.2 eq 12 (with eq 9 and App. C.2) gives the output.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cuda_bf16.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_tma.cuh"

namespace cg = cooperative_groups;

namespace kvc {

constexpr int kFusedMaxChunk = 4096;   // slots per CTA
constexpr int kFusedMaxCS = 8;         // CTAs per cluster
constexpr int kMaxQueue = kPendStride - 2;
constexpr int kNC = 4;                 // consumer warps
constexpr int kWarps = kNC + 2;        // + one producer warp + one moment-fold warp
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 64;              // slots per ring stage: 16 per consumer warp
constexpr int kBoxBytes = kTile * 128; // one box: 64 rows x 64 bf16, 128B-swizzled
constexpr int kTileBytes = 2 * kBoxBytes;
constexpr int kStages = 4;

__device__ __forceinline__ uint32_t sw_off(int r, int j) { return sw_off_t<kTile>(r, j); }
__device__ __forceinline__ void consumer_sync() { named_sync<kNC * 32>(); }

struct FusedArgs {
    const uint16_t *q, *k_new, *v_new;
    uint16_t *K, *V;
    int32_t *votes, *pos;
    double *util;
    int32_t *len;
    float *mn, *mu_k, *mu_v, *C;
    float *o;
    double *probs;
    int32_t *evict_idx, *evict_pos, *n_evict;
    int32_t *pend, *status;
    const int32_t *budget;      // per-unit budgets (NULL: L for every unit)
    const float *rr;            // moment-informed rule: ||r|| per slot ([U][cap], the new token at L)
    int cap, L, T, rule, correction, t, new_pos, kmax, chunk;
    float alpha;
    int merge;                  // KeepKV merge mode: attend over L + 1, append at L
    int R;                      // merge mode: the last R positions are never partners
};

struct Cand {
    uint64_t key;
    int32_t pos;
    int32_t slot;
};

__device__ __forceinline__ bool cand_less(const Cand &a, const Cand &b)
{
    return a.key < b.key || (a.key == b.key && a.pos < b.pos);
}

__device__ __forceinline__ Cand shfl_cand(const Cand &c, int m)
{
    Cand o;
    o.key = __shfl_xor_sync(kFull, (unsigned long long)c.key, m);
    o.pos = __shfl_xor_sync(kFull, c.pos, m);
    o.slot = __shfl_xor_sync(kFull, c.slot, m);
    return o;
}

template <int G>
struct FusedSmem {
    uint64_t full[kStages];     // ring: stage filled (producer -> consumers)
    uint64_t empty[kStages];    // ring: stage drained (consumers -> producer)
    uint64_t vready;            // late victim: every CTA's candidate published
    float qs[G][kD];            // q / sqrt(d), fp32
    float red[kWarps][G];
    float pM[G], pl[G];         // this CTA's partial max / sum
    float po[G][kD];            // this CTA's partial unnormalized output
    float gM[G], gl[G];         // merged
    float fR[G][kD];
    float lzR[G];
    float mass[G];
    float ae[G];                // exp(x_e - M) of the victim (refresh)
    double igl[G];              // (1/G) / merged sum (refresh)
    float igl32[G];
    float pk[kD], pv[kD];       // victim key / value as published by its owner
    float pvp;                  // (never modified after publication)
    int32_t pvpos;
    float ae_pub[G];
    float vk[kD], vv[kD];       // local copies (become the deltas of the fold)
    float vp;                   // victim vote
    int32_t vpos;               // victim position
    float mk0[kD], mv0[kD];     // moments as they were on entry
    float n0;
    float muk[kD], muv[kD];
    float cq[G][kD];
    float zq[G];                // q_h . mu_k' / sqrt(d) after the fold
    float wR[G];
    double vm;                  // utility of the new token (refresh, last CTA)
    Cand cand[kMaxQueue];
    int ncand;
    Cand bc[kWarps];
    Cand zc[kNC];               // merge mode, lazy: each consumer warp's best partner
    Cand zbest;                 // this CTA's best partner (key: cosine, then older position)
    float zred[kWarps][2];
    float zcoef[4];
    int victim;                 // slot index of the victim (L = the new token)
    int qvalid;
    int direct;
    int bad;                    // a ring wait timed out
};

// Stream the rows of this CTA's slots (8 lanes per row, lane c holding the
// 16-byte chunks c and 8 + c), keeping kPrefetch iterations of loads in
// flight per warp so that enough bytes are outstanding to cover HBM latency.
// body(li, i, isnew, ok, r0, r1) consumes one row; the new token (virtual
// slot L, or the victim's slot on a lazy step) is read from `newrow`.
constexpr int kPrefetch = 3;

template <typename Body>
__device__ __forceinline__ void stream_rows(const uint16_t *rows, const uint16_t *newrow, int s0,
                                            int nloc, int L, int victim, int w, int nw, int grp,
                                            int c, Body body)
{
    const int first = w * 4, stride = nw * 4;
    const int niter = nloc > first ? (nloc - first + stride - 1) / stride : 0;   // uniform per warp
    uint4 rb[kPrefetch][2];
    auto issue = [&](int it, uint4 *dst) {
        const int li = first + it * stride + grp;
        const int i = s0 + li;
        if (it < niter && li < nloc) {
            const bool isnew = (i == L || i == victim);
            if (isnew) {
                dst[0] = *reinterpret_cast<const uint4 *>(newrow + 8 * c);
                dst[1] = *reinterpret_cast<const uint4 *>(newrow + 64 + 8 * c);
            } else {
                const uint16_t *r = rows + (size_t)i * kD;
                dst[0] = ldg_nc_v4(r + 8 * c);
                dst[1] = ldg_nc_v4(r + 64 + 8 * c);
            }
        } else {
            dst[0] = make_uint4(0, 0, 0, 0);
            dst[1] = make_uint4(0, 0, 0, 0);
        }
    };
#pragma unroll
    for (int p = 0; p < kPrefetch; p++) issue(p, rb[p]);
    for (int it = 0; it < niter; it += kPrefetch) {
#pragma unroll
        for (int p = 0; p < kPrefetch; p++) {
            if (it + p < niter) {
                const uint4 c0 = rb[p][0], c1 = rb[p][1];
                issue(it + p + kPrefetch, rb[p]);
                const int li = first + (it + p) * stride + grp;
                const int i = s0 + li;
                const bool ok = li < nloc;
                body(li, i, ok && (i == L || i == victim), ok, c0, c1);
            }
        }
    }
}

// ZS: merge mode with the partner search in pass 1 (G = 2 or 4); the
// other instances carry none of its code.
template <int G, bool ZS>
__global__ void __launch_bounds__(kThreads, 2)
fused_step_kernel(FusedArgs a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int CS = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    const int u = blockIdx.x / CS;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int grp = lane >> 3, c = lane & 7;

    __shared__ FusedSmem<G> S;
    extern __shared__ __align__(128) unsigned char dyn[];
    const int ch = a.chunk;
    // [ring: kStages x 8 KB][logits G x (ch + 1)]; the refresh-step selection
    // arrays reuse the ring once both passes have drained it
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));       // swizzle atoms
    float *xsb = reinterpret_cast<float *>(ring + (size_t)kStages * kTileBytes);   // [G][ch + 1]
    double *msm = reinterpret_cast<double *>(ring);
    int32_t *possm = reinterpret_cast<int32_t *>(ring + align_up((size_t)(ch + 1) * 8));
    unsigned char *chosen = ring + align_up((size_t)(ch + 1) * 8) + align_up((size_t)(ch + 1) * 4);
    auto XS = [&](int h, int li) -> float & { return xsb[h * (ch + 1) + li]; };

    // this unit's budget (the grid is laid out for the largest, a.L)
    int L = a.L;
    bool bad_budget = false;
    if (a.budget) {
        const int b = a.budget[u];
        if (b >= 1 && b <= a.L) L = b;
        else bad_budget = true;
    }
    const bool refresh = is_refresh(a.t, a.T);
    const size_t ubase = (size_t)u * a.cap;
    const int s0 = min(L, r * ch), s1 = min(L, s0 + ch);
    const int ntile = (s1 - s0 + kTile - 1) / kTile;

    // The ring starts before anything else: the first kStages K tiles of this
    // CTA's range depend on nothing but the geometry, so they are in flight
    // while the step's scalars, q and the moments are read.
    if (tid == 0) {
        for (int j = 0; j < kStages; j++) {
            mbar_init(&S.full[j], 1);
            mbar_init(&S.empty[j], kNC);
        }
        mbar_init(&S.vready, CS);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int pre = min(kStages, ntile);    // K tiles issued up front (stages 0..pre-1)
    if (w == kNC && lane == 0) {
        const int row0 = (int)(ubase + s0);
        for (int g = 0; g < pre; g++) {
            mbar_expect_tx(&S.full[g], (uint32_t)kTileBytes);
            unsigned char *dst = ring + (size_t)g * kTileBytes;
            tma_2d(dst, &tmK, 0, row0 + g * kTile, &S.full[g]);
            tma_2d(dst + kBoxBytes, &tmK, 64, row0 + g * kTile, &S.full[g]);
        }
    }
    const int n_old = a.len[u];
    if (n_old != L || bad_budget) {        // uniform over the cluster
        if (r == 0 && tid == 0) {
            record_status(a.status, KVC_ERR_SHAPE);
            a.n_evict[u] = 0;
        }
        if (w == kNC && lane == 0)         // the copies land before the CTA leaves
            for (int g = 0; g < pre; g++) mbar_wait(&S.full[g], 0);
        return;
    }
    // Lazy steps take the victim from the refresh step's queue when it has
    // an entry for this step (never in merge mode: a merge raises the
    // partner's utility).  Otherwise the victim is found "late": the fold
    // warp takes the argmin over the stale utilities during pass 1, and pass
    // 2 leaves the victim out (merge mode keeps it).
    int victim = -1;
    bool late = false;
    // merge mode, lazy step, victim known up front: the partner search runs
    // in pass 1 and the merge in the epilogue (no separate merge pass)
    bool zl = false;
    if (!refresh) {
        // last refresh step (step 1 alone for a Score-Free run, T = 0) and
        // this step's place in its queue
        const int tr = a.T > 0 ? a.t - ((a.t - 1) % a.T) : 1;
        const int idx = a.t - tr;
        const int32_t *pq = a.pend + (size_t)u * kPendStride;
        if (!a.merge && pq[0] == tr && pq[1] >= idx) {
            victim = pq[2 + idx - 1];
            if (victim < 0 || victim >= L) victim = -1;
        } else if (ZS && pq[0] == tr) {
            // merge mode: a merge only raises the partner's utility, so the
            // lowest (utility, position) pair among the queued slots is the
            // unit's lowest while it is not above the queue's threshold (the
            // last pair queued at the refresh step: every slot left out was
            // above it then and can only have risen; slots refilled by a new
            // token since are unscored).  Every CTA reads the same entries.
            // lane j of every warp takes entry j (the loads of all entries
            // are in flight together), then a warp minimum
            const int cnt = min(pq[1], kMaxQueue - 3);
            Cand b{~0ull, 0x7fffffff, -1};
            for (int j = lane; j < cnt; j += 32) {
                const int sl = pq[2 + j];
                if (sl < 0 || sl >= L) continue;
                const uint64_t ub = (uint64_t)__double_as_longlong(a.util[ubase + sl]);
                if ((ub & 0x7fffffffffffffffull) == 0x7ff0000000000000ull) continue;
                const Cand cd{double_key(__longlong_as_double((long long)ub)), a.pos[ubase + sl], sl};
                if (cand_less(cd, b)) b = cd;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                const Cand o = shfl_cand(b, m);
                if (cand_less(o, b)) b = o;
            }
            const Cand th{((uint64_t)(uint32_t)pq[kPendStride - 3] << 32) | (uint32_t)pq[kPendStride - 2],
                          pq[kPendStride - 1], 0};
            if (b.slot >= 0 && !cand_less(th, b)) {
                victim = b.slot;
                zl = true;
            }
        }
        late = victim < 0;                  // uniform over the cluster
    }
    // the new token is a separate (virtual) slot L on refresh steps, on late
    // lazy steps and in merge mode; otherwise it replaces the victim's row
    const bool has_new = (refresh || a.merge || late) && (r == CS - 1);
    const int nloc = (s1 - s0) + (has_new ? 1 : 0);
    const float rs = rsqrtf((float)kD);
    const uint16_t *knew = a.k_new + (size_t)u * kD;
    const uint16_t *vnew = a.v_new + (size_t)u * kD;

    for (int e = tid; e < G * kD; e += blockDim.x)
        S.qs[e / kD][e % kD] = bf2f(a.q[(size_t)u * G * kD + e]) * rs;
    // the entry moments are read before the first cluster barrier; CTA 0
    // overwrites them only after several barriers
    for (int e = tid; e < kD; e += blockDim.x) {
        S.mk0[e] = a.mu_k[(size_t)u * kD + e];
        S.mv0[e] = a.mu_v[(size_t)u * kD + e];
    }
    if (tid == 0) {
        S.qvalid = 0; S.direct = 0; S.ncand = 0; S.bad = 0; S.n0 = a.mn[u];
    }
    __syncthreads();

    // every CTA's vready barrier is initialized before any remote arrival
    if (late) cluster.sync();

    // the late victim: the lowest candidate over the cluster's CTAs (each CTA
    // publishes its own before arriving on everyone's vready)
    auto late_victim = [&]() -> int {
        if (!mbar_wait_cluster(&S.vready, 0)) {
            atomicExch(&S.bad, 1);
            return -1;
        }
        Cand b{~0ull, 0x7fffffff, -1};
        for (int q = 0; q < CS; q++) {
            FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
            if (R->ncand > 0 && cand_less(R->cand[0], b)) b = R->cand[0];
        }
        return b.slot;
    };

    // ------------------------------------------------ passes 1 and 2 over the ring
    // The producer warp streams the K rows of [s0, s1), then the V rows, in
    // 64-slot tiles (two 128B-swizzled TMA boxes each) through the ring.  A
    // consumer warp owns 16 slots of a tile.  Pass 1: S = q K^T on tensor
    // cores (m16n8k16, the G query heads in rows 0..G-1 of A, exact bf16
    // products, fp32 accumulate); logits go to shared memory and the CTA max
    // is fixed.  Pass 2: O += P V with P = exp(x - max) split into bf16
    // hi + lo halves (two MMAs), so no online rescaling is needed.
    const uint16_t *Vu = a.V + ubase * kD;
    const int nrows = s1 - s0;
    const int gq = lane >> 2, tq = lane & 3;        // mma fragment coordinates
    const uint32_t ring_s = smem_u32(ring);
    float O[8][4];                                   // O^T fragments: dims 16 m + gq (+8), heads 2 tq (+1)
    float lsq = 0.f;                                 // sum of p for head gq (this lane's slots)
#pragma unroll
    for (int n = 0; n < 8; n++) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;

    // Moment fold of the victim (West's weighted incremental update of the
    // mean / covariance form): mu' = mu + (x - mu) p / n', C' = (n/n') C +
    // (p n / n'^2) dv dk^T with dk, dv taken against the old means; this
    // CTA updates its rows of C and forms C' q / sqrt(d) for them, and
    // q . mu_k' / sqrt(d) for the Jensen bound.  Run by the fold warp during
    // the passes on lazy steps (the victim is known up front), by the whole
    // CTA after the selection on refresh steps.
    const int rows = (kD + CS - 1) / CS;
    const int r0 = min(kD, r * rows), r1 = min(kD, r0 + rows);
    float *Cu = a.C + (size_t)u * kD * kD;
    auto fold = [&](int p, int np, bool block_sync) {
        auto psync = [&]() {
            if (block_sync) __syncthreads();
            else __syncwarp();
        };
        // merge mode folds nothing: the moments stay as they are and only
        // C q and q . mu_k are formed for the correction
        const bool upd = !a.merge;
        const float n0 = S.n0, pe = S.vp, n1 = n0 + pe, fw = upd ? pe / n1 : 0.f;
        for (int e = p; e < kD; e += np) {
            const float mk = S.mk0[e], mv = S.mv0[e];
            S.muk[e] = mk + (S.vk[e] - mk) * fw;
            S.muv[e] = mv + (S.vv[e] - mv) * fw;
            S.vk[e] -= mk;                  // delta k (old mean)
            S.vv[e] -= mv;                  // delta v
        }
        psync();
        const float sc_old = upd ? n0 / n1 : 1.f, sc_rank = upd ? pe * n0 / (n1 * n1) : 0.f;
        // participant -> (row, quarter of columns); the loop bound is uniform
        // so that every lane reaches the shuffles
        for (int rb = r0; rb < r1; rb += np >> 2) {
            const int rr = rb + (p >> 2);
            const bool valid = rr < r1;
            const int q4 = p & 3;
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; h++) acc[h] = 0.f;
            if (valid) {
                float *crow = Cu + (size_t)rr * kD + q4 * 32;
                const float dv = S.vv[rr] * sc_rank;
                float4 cv[8];
#pragma unroll
                for (int j = 0; j < 8; j++) cv[j] = *reinterpret_cast<float4 *>(crow + 4 * j);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float *dk = &S.vk[q4 * 32 + 4 * j];
                    cv[j].x = fmaf(cv[j].x, sc_old, dv * dk[0]);
                    cv[j].y = fmaf(cv[j].y, sc_old, dv * dk[1]);
                    cv[j].z = fmaf(cv[j].z, sc_old, dv * dk[2]);
                    cv[j].w = fmaf(cv[j].w, sc_old, dv * dk[3]);
                    if (upd) *reinterpret_cast<float4 *>(crow + 4 * j) = cv[j];
#pragma unroll
                    for (int h = 0; h < G; h++) {
                        const float *qq = &S.qs[h][q4 * 32 + 4 * j];
                        acc[h] = fmaf(cv[j].x, qq[0], acc[h]);
                        acc[h] = fmaf(cv[j].y, qq[1], acc[h]);
                        acc[h] = fmaf(cv[j].z, qq[2], acc[h]);
                        acc[h] = fmaf(cv[j].w, qq[3], acc[h]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < G; h++) {
                acc[h] += __shfl_xor_sync(kFull, acc[h], 1);
                acc[h] += __shfl_xor_sync(kFull, acc[h], 2);
                if (valid && q4 == 0) S.cq[h][rr] = acc[h];    // q already carries 1/sqrt(d)
            }
        }
        psync();
        const int pw = p >> 5, npw = np >> 5, pl = p & 31;
        for (int h = pw; h < G; h += npw) {
            float sacc = 0.f;
            for (int j = pl; j < kD; j += 32) sacc = fmaf(S.qs[h][j], S.muk[j], sacc);
            sacc = warp_sum(sacc);
            if (pl == 0) S.zq[h] = sacc;
        }
        psync();
    };

    // Refresh steps: the victim is only known after both passes, but the
    // costly part of its fold does not depend on it.  The fold warp, idle
    // during the passes, forms C q / sqrt(d) for the CTA's rows of C (two
    // rows per lane per round; q already carries 1/sqrt(d)), which brings
    // those rows into L2 for the write-back, and prefetches the utilities
    // and positions the epilogue reads.  The fold then enters C q as a
    // rank-one term (fold_cq below).
    auto refresh_prep = [&]() {
        const char *ub = reinterpret_cast<const char *>(a.util + ubase + s0);
        const char *pb = reinterpret_cast<const char *>(a.pos + ubase + s0);
        for (int o = lane * 128; o < (s1 - s0) * 8; o += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(ub + o));
        for (int o = lane * 128; o < (s1 - s0) * 4; o += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(pb + o));
        const int q4 = lane & 3;
        for (int rb = r0; rb < r1; rb += 16) {
            float4 cv[2][8];
            bool vr_[2];
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int rr = rb + 8 * k + (lane >> 2);
                vr_[k] = rr < r1;
#pragma unroll
                for (int j = 0; j < 8; j++)
                    cv[k][j] = vr_[k] ? *reinterpret_cast<const float4 *>(Cu + (size_t)rr * kD + q4 * 32 + 4 * j)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int rr = rb + 8 * k + (lane >> 2);
                float acc[G];
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float *qq = &S.qs[h][q4 * 32];
                    float s_ = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        s_ = fmaf(cv[k][j].x, qq[4 * j], s_);
                        s_ = fmaf(cv[k][j].y, qq[4 * j + 1], s_);
                        s_ = fmaf(cv[k][j].z, qq[4 * j + 2], s_);
                        s_ = fmaf(cv[k][j].w, qq[4 * j + 3], s_);
                    }
                    acc[h] = s_;
                }
#pragma unroll
                for (int h = 0; h < G; h++) {
                    acc[h] += __shfl_xor_sync(kFull, acc[h], 1);
                    acc[h] += __shfl_xor_sync(kFull, acc[h], 2);
                    if (vr_[k] && q4 == 0) S.cq[h][rr] = acc[h];
                }
            }
        }
    };
    // The fold of a refresh step given C q (from refresh_prep): the means,
    // the deltas dk, dv against the old means, and C' q = (n/n') C q +
    // (p n/n'^2) dv (dk . q); C itself is written back by write_back_C.
    auto fold_cq = [&](int p, int np) {
        const bool upd = !a.merge;
        const float n0 = S.n0, pe = S.vp, n1 = n0 + pe, fwt = upd ? pe / n1 : 0.f;
        for (int e = p; e < kD; e += np) {
            const float mk = S.mk0[e], mv = S.mv0[e];
            S.muk[e] = mk + (S.vk[e] - mk) * fwt;
            S.muv[e] = mv + (S.vv[e] - mv) * fwt;
            S.vk[e] -= mk;
            S.vv[e] -= mv;
        }
        __syncthreads();
        // dk . q and q . mu_k' per head: one warp per (head, quantity)
        const int pw = p >> 5, npw = np >> 5, pl = p & 31;
        for (int job = pw; job < 2 * G; job += npw) {
            const int h = job >> 1;
            const float *x = (job & 1) ? S.muk : S.vk;
            float acc = 0.f;
            for (int j = pl; j < kD; j += 32) acc = fmaf(S.qs[h][j], x[j], acc);
            acc = warp_sum(acc);
            if (pl == 0) {
                if (job & 1) S.zq[h] = acc;
                else S.mass[h] = acc;           // dk . q / sqrt(d) (mass is free by now)
            }
        }
        __syncthreads();
        if (upd) {
            const float sc_old = n0 / n1, sc_rank = pe * n0 / (n1 * n1);
            for (int e = p; e < G * (r1 - r0); e += np) {
                const int h = e / (r1 - r0), rr = r0 + e % (r1 - r0);
                S.cq[h][rr] = fmaf(sc_rank * S.vv[rr], S.mass[h], sc_old * S.cq[h][rr]);
            }
        }
        __syncthreads();
    };
    // C' = (n/n') C + (p n/n'^2) dv dk^T for the CTA's rows (L2-hot since
    // refresh_prep read them)
    auto write_back_C = [&]() {
        const float n0 = S.n0, pe = S.vp, n1 = n0 + pe;
        const float sc_old = n0 / n1, sc_rank = pe * n0 / (n1 * n1);
        // eight float4 per thread in flight before any is written back
        const int total = (r1 - r0) * (kD / 4);
        for (int e0 = tid; e0 < total; e0 += 8 * (int)blockDim.x) {
            float4 cv[8];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int e = e0 + k * (int)blockDim.x;
                cv[k] = e < total ? *reinterpret_cast<const float4 *>(Cu + (size_t)(r0 + e / (kD / 4)) * kD +
                                                                      (e % (kD / 4)) * 4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int e = e0 + k * (int)blockDim.x;
                if (e >= total) break;
                const int rr = r0 + e / (kD / 4), c4 = (e % (kD / 4)) * 4;
                const float dv = S.vv[rr] * sc_rank;
                float4 c = cv[k];
                c.x = fmaf(c.x, sc_old, dv * S.vk[c4]);
                c.y = fmaf(c.y, sc_old, dv * S.vk[c4 + 1]);
                c.z = fmaf(c.z, sc_old, dv * S.vk[c4 + 2]);
                c.w = fmaf(c.w, sc_old, dv * S.vk[c4 + 3]);
                *reinterpret_cast<float4 *>(Cu + (size_t)rr * kD + c4) = c;
            }
        }
    };

    if (w == kNC + 1) {
        // ---------------- late victim and moment fold (lazy steps), concurrent
        // with the passes
        if (late) {
            // eight slots per lane per round, every load issued before the
            // comparisons, so that the scan ends well inside pass 1
            constexpr int kScan = 8;
            Cand best{~0ull, 0x7fffffff, -1};
            for (int i0 = s0 + lane; i0 < s1; i0 += 32 * kScan) {
                double m[kScan];
                int32_t ps[kScan];
#pragma unroll
                for (int j = 0; j < kScan; j++) {
                    const int i = i0 + 32 * j;
                    m[j] = i < s1 ? a.util[ubase + i] : __longlong_as_double(0x7ff0000000000000ll);
                    ps[j] = i < s1 ? a.pos[ubase + i] : 0;
                }
#pragma unroll
                for (int j = 0; j < kScan; j++) {
                    if (isinf(m[j])) continue;
                    Cand cd{double_key(m[j]), ps[j], i0 + 32 * j};
                    if (cand_less(cd, best)) best = cd;
                }
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                Cand o = shfl_cand(best, m);
                if (cand_less(o, best)) best = o;
            }
            if (lane == 0) {
                S.cand[0] = best;
                S.ncand = best.slot >= 0 ? 1 : 0;
                for (int q = 0; q < CS; q++) mbar_arrive_remote(&S.vready, (uint32_t)q);
            }
            __syncwarp();
            victim = late_victim();
            if (lane == 0) S.victim = victim;
        }
        if (!refresh && victim >= 0) {
            const uint16_t *kr = a.K + (ubase + victim) * kD;
            const uint16_t *vr = a.V + (ubase + victim) * kD;
            for (int e = lane; e < kD; e += 32) {
                S.vk[e] = bf2f(kr[e]);
                S.vv[e] = bf2f(vr[e]);
            }
            if (lane == 0) {
                S.vp = a.merge ? 0.f : (a.votes ? (float)a.votes[ubase + victim] : 1.f);
                S.vpos = a.pos[ubase + victim];
            }
            __syncwarp();
            fold(lane, 32, false);
        } else if (refresh) {
            refresh_prep();
        }
    } else if (w == kNC) {
        // ---------------- producer
        if (lane == 0) {
            int g = pre;                    // the first pre K tiles are in flight already
            bool ok = true;
            const int row0 = (int)((size_t)u * a.cap + s0);
            for (int pass = 0; pass < 2 && ok; pass++) {
                const CUtensorMap *map = pass == 0 ? &tmK : &tmV;
                for (int t = pass == 0 ? pre : 0; t < ntile; t++, g++) {
                    const int stage = g % kStages;
                    const uint32_t ph = (uint32_t)(g / kStages) & 1u;
                    if (!mbar_wait(&S.empty[stage], ph ^ 1u)) { ok = false; break; }
                    mbar_expect_tx(&S.full[stage], (uint32_t)kTileBytes);
                    unsigned char *dst = ring + (size_t)stage * kTileBytes;
                    tma_2d(dst, map, 0, row0 + t * kTile, &S.full[stage]);
                    tma_2d(dst + kBoxBytes, map, 64, row0 + t * kTile, &S.full[stage]);
                }
            }
            if (!ok) {
                atomicExch(&S.bad, 1);
                for (int j = max(0, g - kStages); j < g; j++)   // let issued copies land
                    mbar_wait(&S.full[j % kStages], (uint32_t)(j / kStages) & 1u);
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers
        // q K^T as D[slot][head]: A = 16 K rows (ldmatrix from the swizzled
        // tile), B = q^T (16 dims x 8 heads, heads >= G zero).  P V as
        // O^T[dim][head]: A = V^T (ldmatrix.trans), B = P^T (16 slots x 8
        // heads, p split into bf16 hi + lo).  A lane (gq, tq) holds logits of
        // slots gq, gq + 8 for heads 2 tq, 2 tq + 1, and p of head gq.
        uint32_t qb[8][2];
        {
            // merge mode, lazy: column G carries the victim's key, so that
            // the same MMAs give k_e . k_j for the partner search
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(a.q + (size_t)u * G * kD);
            const uint32_t *ke32 = reinterpret_cast<const uint32_t *>(a.K + (ubase + (zl ? victim : 0)) * kD);
            const bool kecol = ZS && zl && gq == G;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                qb[ks][0] = gq < G ? q32[(gq * kD + 16 * ks + 2 * tq) >> 1]
                                   : (kecol ? ke32[(16 * ks + 2 * tq) >> 1] : 0u);
                qb[ks][1] = gq < G ? q32[(gq * kD + 16 * ks + 8 + 2 * tq) >> 1]
                                   : (kecol ? ke32[(16 * ks + 8 + 2 * tq) >> 1] : 0u);
            }
        }
        // partner search (merge mode, lazy): cosine of k_e with every slot
        // outside the last R positions, k_e . k_j / |k_j| (|k_e| > 0 is a
        // common factor); lanes tq = G / 2 hold column G
        const long long zlim = (long long)a.new_pos - a.R;
        unsigned long long zkey = 0ull;
        int zslot = -1;
        auto load_pos = [&](int t, int &p0, int &p1) {
            const int li = t * kTile + w * 16 + gq;
            p0 = li < nrows ? a.pos[ubase + s0 + li] : 0x7fffffff;
            p1 = li + 8 < nrows ? a.pos[ubase + s0 + li + 8] : 0x7fffffff;
        };
        int pn0 = 0x7fffffff, pn1 = 0x7fffffff;
        if (ZS && zl && ntile > 0) load_pos(0, pn0, pn1);
        const int rb = w * 16;                   // this warp's rows in a tile
        const int h0 = 2 * tq, h1 = 2 * tq + 1;  // heads of this lane's logits
        bool good = true;
        float mx0 = -INFINITY, mx1 = -INFINITY;  // max logit of heads h0, h1 over this lane's slots
        // Rows of this warp that must not be used as loaded: slots past the
        // CTA's range (zeroed) and, on a lazy step, the victim's slot (the new
        // token's row is written there; in merge mode the victim stays).
        // Generic writes into the ring are fenced against the next TMA write
        // of the stage.
        const int pvict = a.merge ? -1 : victim;
        auto patch = [&](uint32_t stage_off, int t, const uint16_t *newrow) -> bool {
            bool any = false;
            const int base_li = t * kTile + rb;
            if (base_li + 16 > nrows) {
                for (int e = lane; e < 16 * 16; e += 32) {
                    const int r = e >> 4, j = e & 15;
                    if (base_li + r >= nrows) {
                        *reinterpret_cast<uint4 *>(ring + stage_off + sw_off(rb + r, j)) = make_uint4(0, 0, 0, 0);
                        any = true;
                    }
                }
            }
            const int vr = pvict - s0 - t * kTile - rb;
            if (pvict >= 0 && vr >= 0 && vr < 16) {
                if (lane < 16)
                    *reinterpret_cast<uint4 *>(ring + stage_off + sw_off(rb + vr, lane)) =
                        *reinterpret_cast<const uint4 *>(newrow + 8 * lane);
                any = true;
            }
            any = __any_sync(kFull, any);
            if (any) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            return any;
        };
        int g = 0;
        // votes of this lane's two slots of a tile (gq, gq + 8), loaded one
        // tile ahead so that the loads are in flight during the previous tile
        auto load_votes = [&](int t, int &v0, int &v1) {
            const int li = t * kTile + rb + gq;
            v0 = li < nrows ? a.votes[ubase + s0 + li] : 1;
            v1 = li + 8 < nrows ? a.votes[ubase + s0 + li + 8] : 1;
        };
        int vn0 = 1, vn1 = 1;
        if (a.votes && ntile > 0) load_votes(0, vn0, vn1);
        // pass 1: logits
        for (int t = 0; t < ntile; t++, g++) {
            const int stage = g % kStages;
            const uint32_t ph = (uint32_t)(g / kStages) & 1u;
            const int vc[2] = {vn0, vn1};
            if (a.votes && t + 1 < ntile) load_votes(t + 1, vn0, vn1);
            const int pc[2] = {pn0, pn1};
            if (ZS && zl && t + 1 < ntile) load_pos(t + 1, pn0, pn1);
            if (good && !mbar_wait(&S.full[stage], ph)) good = false;
            if (good) {
                const uint32_t so = (uint32_t)stage * kTileBytes;
                patch(so, t, knew);
                float sacc[4] = {0.f, 0.f, 0.f, 0.f};
                // merge mode, lazy: the Gram blocks of the warp's 16 rows with
                // rows 0-7 and 8-15 (the A fragments are also the B fragments
                // of those rows), whose diagonals are |k_j|^2
                float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
                const int mi = lane >> 3;
                const int lrow = rb + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < 8; ks++) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(ring_s + so + sw_off(lrow, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                    mma16816(sacc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                    if (ZS && zl) {
                        mma16816(g0, a0, a1, a2, a3, a0, a2);
                        mma16816(g1, a0, a1, a2, a3, a1, a3);
                    }
                }
                if (ZS && zl) {
                    // |k|^2 of row gq sits in lane (gq, gq / 2) of g0, of row
                    // gq + 8 in the same lane of g1; bring both to this lane
                    const int src = 4 * gq + (gq >> 1);
                    const float d0 = (gq & 1) ? g0[1] : g0[0];
                    const float d1 = (gq & 1) ? g1[3] : g1[2];
                    const float sq0 = __shfl_sync(kFull, d0, src);
                    const float sq1 = __shfl_sync(kFull, d1, src);
                    if (2 * tq == G) {
#pragma unroll
                        for (int hf = 0; hf < 2; hf++) {
                            const int li = t * kTile + rb + gq + 8 * hf;
                            const int i = s0 + li;
                            const float ss = hf ? sq1 : sq0;
                            if (li < nrows && i != victim && (long long)pc[hf] <= zlim) {
                                const float sc = ss > 0.f ? sacc[2 * hf] * rsqrtf(ss) : 0.f;
                                const unsigned long long key =
                                    ((unsigned long long)float_key(sc) << 32) | (uint32_t)(0x7fffffff - pc[hf]);
                                if (key > zkey) {
                                    zkey = key;
                                    zslot = i;
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int hf = 0; hf < 2; hf++) {           // slot gq, then gq + 8
                    const int li = t * kTile + rb + gq + 8 * hf;
                    if (li < nrows) {
                        const bool isnew = (s0 + li == pvict);
                        const float lnp = (!isnew && a.votes) ? logf((float)vc[hf]) : 0.f;
                        if (h0 < G) {
                            const float x = sacc[2 * hf] * rs + lnp;
                            XS(h0, li) = x;
                            mx0 = fmaxf(mx0, x);
                        }
                        if (h1 < G) {
                            const float x = sacc[2 * hf + 1] * rs + lnp;
                            XS(h1, li) = x;
                            mx1 = fmaxf(mx1, x);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.empty[stage]);
        }
        if (ZS && zl) {
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                const unsigned long long ok = __shfl_xor_sync(kFull, zkey, m);
                const int os = __shfl_xor_sync(kFull, zslot, m);
                if (ok > zkey) {
                    zkey = ok;
                    zslot = os;
                }
            }
            if (lane == 0) S.zc[w] = Cand{zkey, 0, zslot};
        }
        // the virtual slot L (refresh steps): scalar dot products on warp 0
        float xv_new[G];
        if (has_new && w == 0) {
#pragma unroll
            for (int h = 0; h < G; h++) {
                float sacc = 0.f;
                for (int j = lane; j < kD; j += 32) sacc = fmaf(S.qs[h][j], bf2f(knew[j]), sacc);
                xv_new[h] = warp_sum(sacc);          // S.qs already carries 1/sqrt(d)
                if (lane == 0) XS(h, nrows) = xv_new[h];
            }
#pragma unroll
            for (int h = 0; h < G; h++) {
                if (h == h0) mx0 = fmaxf(mx0, xv_new[h]);
                if (h == h1) mx1 = fmaxf(mx1, xv_new[h]);
            }
        }
#pragma unroll
        for (int m = 4; m <= 16; m <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, m));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, m));
        }
        if (gq == 0) {
            if (h0 < G) S.red[w][h0] = mx0;
            if (h1 < G) S.red[w][h1] = mx1;
        }
        consumer_sync();
        float Mg = -INFINITY;                     // CTA max of head gq (the head of this lane's p)
        if (gq < G)
            for (int j = 0; j < kNC; j++) Mg = fmaxf(Mg, S.red[j][gq]);
        if (tid < G) {
            float v = S.red[0][tid];
            for (int j = 1; j < kNC; j++) v = fmaxf(v, S.red[j][tid]);
            S.pM[tid] = v;
        }
        consumer_sync();                          // S.red is reused below
        // a late victim leaves pass 2 (evict mode)
        int vmask = -1;
        if (late) {
            const int v = late_victim();
            if (!a.merge && v >= s0 && v < s1) vmask = v - s0;
        }
        // pass 2: O^T += V^T P^T
        for (int t = 0; t < ntile; t++, g++) {
            const int stage = g % kStages;
            const uint32_t ph = (uint32_t)(g / kStages) & 1u;
            if (good && !mbar_wait(&S.full[stage], ph)) good = false;
            if (good) {
                const uint32_t so = (uint32_t)stage * kTileBytes;
                patch(so, t, vnew);
                float pv[4];
                const int sl[4] = {2 * tq, 2 * tq + 1, 8 + 2 * tq, 9 + 2 * tq};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int li = t * kTile + rb + sl[e];
                    pv[e] = (gq < G && li < nrows && li != vmask) ? expf(XS(gq, li) - Mg) : 0.f;
                    lsq += pv[e];
                }
                uint16_t hi0, lo0, hi1, lo1, hi2, lo2, hi3, lo3;
                split_bf16(pv[0], hi0, lo0);
                split_bf16(pv[1], hi1, lo1);
                split_bf16(pv[2], hi2, lo2);
                split_bf16(pv[3], hi3, lo3);
                const uint32_t bh0 = (uint32_t)hi0 | ((uint32_t)hi1 << 16), bh1 = (uint32_t)hi2 | ((uint32_t)hi3 << 16);
                const uint32_t bl0 = (uint32_t)lo0 | ((uint32_t)lo1 << 16), bl1 = (uint32_t)lo2 | ((uint32_t)lo3 << 16);
                const int mi = lane >> 3;
                const int lrow = rb + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                for (int mt = 0; mt < 8; mt++) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(ring_s + so + sw_off(lrow, 2 * mt + (mi & 1)), a0, a1, a2, a3);
                    mma16816(O[mt], a0, a1, a2, a3, bh0, bh1);
                    mma16816(O[mt], a0, a1, a2, a3, bl0, bl1);
                }
            }
            __syncwarp();
            if (lane == 0 && good) mbar_arrive(&S.empty[stage]);
        }
        if (has_new && w == 0) {
            float pn0 = 0.f, pn1 = 0.f, pnq = 0.f;
            const float M0 = h0 < G ? S.pM[h0] : 0.f, M1 = h1 < G ? S.pM[h1] : 0.f;
#pragma unroll
            for (int h = 0; h < G; h++) {
                const float pe = expf(xv_new[h] - S.pM[h]);
                if (h == h0) pn0 = pe;
                if (h == h1) pn1 = pe;
                if (h == gq) pnq = pe;
            }
            (void)M0; (void)M1;
            if (tq == 0 && gq < G) lsq += pnq;
#pragma unroll
            for (int mt = 0; mt < 8; mt++) {
                const float va = bf2f(vnew[16 * mt + gq]), vb = bf2f(vnew[16 * mt + gq + 8]);
                O[mt][0] = fmaf(pn0, va, O[mt][0]);
                O[mt][1] = fmaf(pn1, va, O[mt][1]);
                O[mt][2] = fmaf(pn0, vb, O[mt][2]);
                O[mt][3] = fmaf(pn1, vb, O[mt][3]);
            }
        }
        if (!good) atomicExch(&S.bad, 1);
    }
    // reduce the p v partials of the consumer warps (O^T fragment layout:
    // lane (gq, tq) holds dims 16 m + gq and + 8 for heads 2 tq and 2 tq + 1)
    for (int e = tid; e < G * kD; e += blockDim.x) S.po[e / kD][e % kD] = 0.f;
    lsq += __shfl_xor_sync(kFull, lsq, 1);
    lsq += __shfl_xor_sync(kFull, lsq, 2);
    __syncthreads();
    if (w < kNC) {
        const int h0 = 2 * tq, h1 = 2 * tq + 1;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            if (h0 < G) {
                atomicAdd(&S.po[h0][16 * mt + gq], O[mt][0]);
                atomicAdd(&S.po[h0][16 * mt + gq + 8], O[mt][2]);
            }
            if (h1 < G) {
                atomicAdd(&S.po[h1][16 * mt + gq], O[mt][1]);
                atomicAdd(&S.po[h1][16 * mt + gq + 8], O[mt][3]);
            }
        }
        if (tq == 0 && gq < G) S.red[w][gq] = lsq;
    }
    __syncthreads();
    if (tid < G) {
        float l = 0.f;
        for (int j = 0; j < kNC; j++) l += S.red[j][tid];
        S.pl[tid] = l;
    }
    __syncthreads();

    // The rare direct recomputation of a refresh step (victim mass > 1/2)
    // re-reads V from global memory with CUDA cores: 8 lanes per slot, the
    // consumer warps only.
    auto pv_pass = [&](int skip, const float *Mref) {
        float accv[G][16], lsum[G];
#pragma unroll
        for (int h = 0; h < G; h++) {
            lsum[h] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) accv[h][j] = 0.f;
        }
        if (w < kNC) {
            float Mr[G];
#pragma unroll
            for (int h = 0; h < G; h++) Mr[h] = Mref[h];
            stream_rows(Vu, vnew, s0, nloc, L, victim, w, kNC, grp, c,
                        [&](int li, int i, bool isnew, bool ok, const uint4 &r0, const uint4 &r1) {
                (void)isnew;
                if (ok && i != skip) {
                    float vf[16];
                    unpack8(r0, vf);
                    unpack8(r1, vf + 8);
#pragma unroll
                    for (int h = 0; h < G; h++) {
                        const float p = expf(XS(h, li) - Mr[h]);
                        if (c == 0) lsum[h] += p;
#pragma unroll
                        for (int j = 0; j < 16; j++) accv[h][j] = fmaf(p, vf[j], accv[h][j]);
                    }
                }
            });
        }
#pragma unroll
        for (int h = 0; h < G; h++) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                accv[h][j] += __shfl_xor_sync(kFull, accv[h][j], 8);
                accv[h][j] += __shfl_xor_sync(kFull, accv[h][j], 16);
            }
            lsum[h] = warp_sum(lsum[h]);
        }
        for (int e = tid; e < G * kD; e += blockDim.x) S.po[e / kD][e % kD] = 0.f;
        __syncthreads();
        if (grp == 0 && w < kNC)
#pragma unroll
            for (int h = 0; h < G; h++)
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    atomicAdd(&S.po[h][8 * c + j], accv[h][j]);
                    atomicAdd(&S.po[h][64 + 8 * c + j], accv[h][8 + j]);
                }
        if (lane == 0)
#pragma unroll
            for (int h = 0; h < G; h++) S.red[w][h] = lsum[h];
        __syncthreads();
        if (tid < G) {
            float l = 0.f;
            for (int j = 0; j < kNC; j++) l += S.red[j][tid];
            S.pl[tid] = l;
        }
        __syncthreads();
    };

    if (ZS && zl && tid == 0) {
        Cand b{0ull, 0, -1};
        for (int j = 0; j < kNC; j++)
            if (S.zc[j].slot >= 0 && S.zc[j].key > b.key) b = S.zc[j];
        S.zbest = b;
    }
    // ------------------------------------------------ cluster merge
    cluster.sync();                                                    // partials visible
    auto merge = [&]() {
        if (tid < G) {
            const int h = tid;
            float M = -INFINITY;
            for (int q = 0; q < CS; q++) M = fmaxf(M, cluster.map_shared_rank(&S, q)->pM[h]);
            float l = 0.f;
            for (int q = 0; q < CS; q++) {
                FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
                if (R->pM[h] != -INFINITY) l += R->pl[h] * expf(R->pM[h] - M);
            }
            S.gM[h] = M;
            S.gl[h] = l;
        }
        __syncthreads();
        for (int e = tid; e < G * kD; e += blockDim.x) {
            const int h = e / kD, dd = e % kD;
            float v = 0.f;
            for (int q = 0; q < CS; q++) {
                FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
                if (R->pM[h] != -INFINITY) v += R->po[h][dd] * expf(R->pM[h] - S.gM[h]);
            }
            S.fR[h][dd] = v;                // unnormalized, relative to gM
        }
        __syncthreads();
    };
    merge();
    if (late) {
        victim = S.victim;
        if (victim < 0) {                       // no scored slot (or a timeout): refuse
            if (r == 0 && tid == 0) {
                record_status(a.status, S.bad ? KVC_ERR_TIMEOUT : KVC_ERR_INVALID_ARG);
                a.n_evict[u] = 0;
            }
            cluster.sync();                     // nobody reads this CTA's partials any more
            return;
        }
    }

    int vic_owner;
    if (refresh) {
        // -------------------------------------------- probabilities + utilities
        const double al = (double)a.alpha;
        if (tid < G) {
            // (1/G) / merged sum per head: one fp64 division per head; G is a
            // power of two, so the 1/G factor is exact
            S.igl[tid] = (1.0 / G) / (double)S.gl[tid];
            S.igl32[tid] = (float)S.igl[tid];
        }
        // the old utilities and the positions first, staged in shared
        // memory: eight slots per thread loaded into registers before any is
        // stored (the stores could alias the loads for all the compiler
        // knows, which would serialize them)
        for (int li0 = tid; li0 < nloc; li0 += 8 * (int)blockDim.x) {
            double mv8[8];
            int32_t pv8[8];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int li = li0 + k * (int)blockDim.x, i = s0 + li;
                const bool in = li < nloc, isv = in && i == L;
                mv8[k] = (in && !isv) ? a.util[ubase + i] : __longlong_as_double(0x7ff0000000000000ll);
                pv8[k] = (in && !isv) ? a.pos[ubase + i] : a.new_pos;
            }
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int li = li0 + k * (int)blockDim.x;
                if (li < nloc) {
                    msm[li] = mv8[k];
                    possm[li] = pv8[k];
                }
            }
        }
        __syncthreads();
        for (int li = tid; li < nloc; li += blockDim.x) {
            const int i = s0 + li;
            // head-mean probability.  While the largest head term is above
            // e^-60 the sum is far inside fp32's range (a term fp32 would
            // flush is below 1e-8 of it) and fp32 carries it to a few units
            // in the last place; below that the fp64 form keeps the range.
            float y[G], ymax = -INFINITY;
#pragma unroll
            for (int h = 0; h < G; h++) {
                y[h] = XS(h, li) - S.gM[h];
                ymax = fmaxf(ymax, y[h]);
            }
            double s;
            if (ymax > -60.f) {
                float s32 = 0.f;
#pragma unroll
                for (int h = 0; h < G; h++) s32 = fmaf(expf(y[h]), S.igl32[h], s32);
                s = (double)s32;
            } else {
                s = 0.0;
#pragma unroll
                for (int h = 0; h < G; h++) s = fma(exp_wide(y[h]), S.igl[h], s);
            }
            const bool isv = (i == L);
            const double m = msm[li];
            double mn;
            if (a.rule == KVC_RULE_MI) mn = s * (double)a.rr[ubase + i];   // MomentKV alpha ||r||
            else if (isinf(m)) mn = s;
            else if (a.rule == KVC_RULE_SINGLE) mn = s;
            else if (a.rule == KVC_RULE_CUMULATIVE) mn = m + s;
            else mn = al * m + (1.0 - al) * s;
            msm[li] = mn;
            chosen[li] = 0;
            if (!isv) a.util[ubase + i] = mn;
            else S.vm = mn;
            if (a.probs) a.probs[ubase + i] = s;
        }
        __syncthreads();
        // -------------------------------------------- local T lowest
        // Each warp finds the `want` lowest (utility, position) pairs among
        // its own slots (li = 32 w + lane + 32 kWarps j), with no block
        // barrier.  Every lane caches the two lowest of its own slots; a
        // round is a warp minimum by hardware reductions (key high word, key
        // low word, then position among equal keys), the winning lane
        // promotes its second entry and rescans only when it wins again.
        // Thread 0 then merges the sorted per-warp lists.
        // queue length: T (one victim per step until the next refresh); a
        // Score-Free run (T = 0, no later refresh) queues as many as fit.
        // Merge mode queues 2 T (a merge can lift a queued partner out of
        // the lowest) with the last pair as the queue's threshold; it is
        // used where the partner search can run in pass 1 (G = 2 or 4).
        const bool mq = ZS;
        const int Tq = a.merge ? (mq ? min(a.T > 0 ? 2 * a.T : kMaxQueue, kMaxQueue - 3) : 1)
                               : (a.T > 0 ? a.T : kMaxQueue);
        const int want = min(Tq, nloc);
        Cand *wl = reinterpret_cast<Cand *>(chosen + align_up((size_t)(ch + 1)));   // [kWarps][kMaxQueue]
        const Cand none{~0ull, 0x7fffffff, -1};
        Cand c1 = none, c2 = none;         // this lane's two lowest not yet taken
        auto lane_scan = [&]() {
            c1 = none;
            c2 = none;
            for (int li = w * 32 + lane; li < nloc; li += kWarps * 32) {
                if (chosen[li]) continue;
                const Cand cd{double_key(msm[li]), possm[li], s0 + li};
                if (cand_less(cd, c1)) {
                    c2 = c1;
                    c1 = cd;
                } else if (cand_less(cd, c2)) {
                    c2 = cd;
                }
            }
        };
        lane_scan();
        bool c2_valid = true;              // c2 is the true second of the remaining slots
        for (int rnd = 0; rnd < want; rnd++) {
            const uint32_t hi = (uint32_t)(c1.key >> 32), lo = (uint32_t)c1.key;
            const uint32_t mhi = __reduce_min_sync(kFull, hi);
            const uint32_t mlo = __reduce_min_sync(kFull, hi == mhi ? lo : 0xffffffffu);
            const bool tie = hi == mhi && lo == mlo;
            const uint32_t mpos = __reduce_min_sync(kFull, tie ? (uint32_t)c1.pos ^ 0x80000000u : 0xffffffffu);
            const bool win = tie && ((uint32_t)c1.pos ^ 0x80000000u) == mpos;
            const uint32_t wm = __ballot_sync(kFull, win && c1.slot >= 0);
            if (wm == 0u) {                 // nothing left in this warp
                if (lane == 0) wl[w * kMaxQueue + rnd] = none;
                continue;
            }
            const int src = __ffs(wm) - 1;
            Cand best;
            best.key = __shfl_sync(kFull, (unsigned long long)c1.key, src);
            best.pos = __shfl_sync(kFull, c1.pos, src);
            best.slot = __shfl_sync(kFull, c1.slot, src);
            if (lane == 0) wl[w * kMaxQueue + rnd] = best;
            if (lane == src) {
                chosen[best.slot - s0] = 1;
                if (c2_valid) {
                    c1 = c2;
                    c2 = none;
                    c2_valid = false;
                } else {
                    lane_scan();
                    c2_valid = true;
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            int ptr[kWarps];
            for (int q = 0; q < kWarps; q++) ptr[q] = 0;
            int nc = 0;
            for (; nc < want; nc++) {
                int bq = -1;
                Cand b{~0ull, 0x7fffffff, -1};
                for (int q = 0; q < kWarps; q++) {
                    if (ptr[q] >= want) continue;
                    const Cand cq = wl[q * kMaxQueue + ptr[q]];
                    if (cq.slot >= 0 && cand_less(cq, b)) {
                        b = cq;
                        bq = q;
                    }
                }
                if (bq < 0) break;
                ptr[bq]++;
                S.cand[nc] = b;
            }
            S.ncand = nc;
        }
        cluster.sync();                                                // candidates visible
        // every CTA merges the candidate lists the same way: one parallel
        // gather over distributed shared memory, then a local merge
        Cand *gc = wl + kWarps * kMaxQueue;                  // [CS][kMaxQueue]
        for (int e = tid; e < CS * Tq; e += blockDim.x) {
            const int q = e / Tq, jj = e % Tq;
            FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
            gc[q * kMaxQueue + jj] = jj < R->ncand ? R->cand[jj] : Cand{~0ull, 0x7fffffff, -1};
        }
        __syncthreads();
        if (tid == 0) {
            int ptr[kFusedMaxCS];
            for (int q = 0; q < CS; q++) ptr[q] = 0;
            Cand *sel = gc + kFusedMaxCS * kMaxQueue;       // [kMaxQueue]
            int nsel = 0;
            while (nsel < Tq) {
                int bq = -1;
                Cand b{~0ull, 0x7fffffff, -1};
                for (int q = 0; q < CS; q++) {
                    if (ptr[q] >= Tq) continue;
                    const Cand cq = gc[q * kMaxQueue + ptr[q]];
                    if (cq.slot >= 0 && cand_less(cq, b)) {
                        b = cq;
                        bq = q;
                    }
                }
                if (bq < 0) break;
                ptr[bq]++;
                sel[nsel++] = b;
            }
            S.victim = nsel > 0 ? sel[0].slot : -1;
            if (r == 0 && nsel > 0) {
                int32_t *pq = a.pend + (size_t)u * kPendStride;
                pq[0] = (a.merge && !mq) ? 0 : a.t;
                pq[1] = nsel - 1;
                for (int j = 1; j < nsel; j++)
                    pq[2 + j - 1] = sel[j].slot == L ? sel[0].slot : sel[j].slot;
                if (mq) {
                    // threshold: the last pair queued, or above everything
                    // when every scored slot is in the queue
                    const Cand th = nsel == Tq ? sel[nsel - 1] : Cand{~0ull, 0x7fffffff, -1};
                    pq[kPendStride - 3] = (int32_t)(uint32_t)(th.key >> 32);
                    pq[kPendStride - 2] = (int32_t)(uint32_t)th.key;
                    pq[kPendStride - 1] = th.pos;
                }
            }
        }
        __syncthreads();
        victim = S.victim;
        vic_owner = (victim == L) ? CS - 1 : victim / ch;
        // -------------------------------------------- victim data + identity
        if (r == vic_owner) {
            const int li = victim - s0;
            const bool isv = (victim == L);
            const uint16_t *kr = isv ? knew : a.K + (ubase + victim) * kD;
            const uint16_t *vr = isv ? vnew : a.V + (ubase + victim) * kD;
            for (int e = tid; e < kD; e += blockDim.x) {
                S.pk[e] = bf2f(kr[e]);
                S.pv[e] = bf2f(vr[e]);
            }
            if (tid < G) S.ae_pub[tid] = expf(XS(tid, li) - S.gM[tid]);
            if (tid == 0) {
                S.pvp = a.merge ? 0.f : ((isv || !a.votes) ? 1.f : (float)a.votes[ubase + victim]);
                S.pvpos = isv ? a.new_pos : possm[li];
            }
        }
        cluster.sync();                                                // victim visible
        FusedSmem<G> *O = cluster.map_shared_rank(&S, vic_owner);
        if (tid < G) {
            const float ae = O->ae_pub[tid];
            S.ae[tid] = ae;
            S.mass[tid] = ae / S.gl[tid];
            if (!a.merge && S.mass[tid] > 0.5f) atomicExch(&S.direct, 1);
        }
        for (int e = tid; e < kD; e += blockDim.x) {
            S.vk[e] = O->pk[e];
            S.vv[e] = O->pv[e];
        }
        if (tid == 0) { S.vp = O->pvp; S.vpos = O->pvpos; }
        __syncthreads();
        if (a.merge) {
            // nothing leaves the attention set: the output is the one over
            // every slot (the victim is merged after this kernel)
            for (int e = tid; e < G * kD; e += blockDim.x) S.fR[e / kD][e % kD] /= S.gl[e / kD];
            if (tid < G) S.lzR[tid] = S.gM[tid] + logf(S.gl[tid]);
            __syncthreads();
        } else if (!S.direct) {
            for (int e = tid; e < G * kD; e += blockDim.x) {
                const int h = e / kD, dd = e % kD;
                S.fR[h][dd] = (S.fR[h][dd] - S.ae[h] * S.vv[dd]) / (S.gl[h] - S.ae[h]);
            }
            if (tid < G) S.lzR[tid] = S.gM[tid] + logf(S.gl[tid] - S.ae[tid]);
            __syncthreads();
        } else {
            // recompute the retained output: the partial p v without the victim
            cluster.sync();                         // everyone is done reading partials
            pv_pass(victim, S.pM);
            cluster.sync();
            merge();
            for (int e = tid; e < G * kD; e += blockDim.x) S.fR[e / kD][e % kD] /= S.gl[e / kD];
            if (tid < G) S.lzR[tid] = S.gM[tid] + logf(S.gl[tid]);
            __syncthreads();
        }
    } else {
        vic_owner = victim / ch;
        for (int e = tid; e < G * kD; e += blockDim.x) S.fR[e / kD][e % kD] /= S.gl[e / kD];
        if (tid < G) S.lzR[tid] = S.gM[tid] + logf(S.gl[tid]);
        __syncthreads();
    }

    if (refresh) fold_cq(tid, blockDim.x);            // lazy steps folded during the passes
    const float n1 = S.n0 + S.vp;
    for (int h = tid; h < G; h += blockDim.x) {
        const float logZE = logf(n1) + S.zq[h];
        S.wR[h] = 1.f / (1.f + expf(logZE - S.lzR[h]));
    }
    __syncthreads();
    float *ou = a.o + (size_t)u * G * kD;
    for (int e = tid; e < G * (r1 - r0); e += blockDim.x) {
        const int h = e / (r1 - r0), dd = r0 + e % (r1 - r0);
        float val = S.fR[h][dd];
        if (a.correction != KVC_CORR_OFF) {
            const float fe = S.muv[dd] + (a.correction == KVC_CORR_FIRST_ORDER ? S.cq[h][dd] : 0.f);
            val = S.wR[h] * val + (1.f - S.wR[h]) * fe;
        }
        ou[(size_t)h * kD + dd] = val;
    }
    // merge mode, lazy step with the partner found in pass 1: KeepKV's
    // ZIP-merge (the weights w = p exp(x) of the group's mean logit, eqs
    // 10 and 12, the epsilon guard) of the victim into it on CTA 0, then the
    // new token takes the victim's slot: the unit keeps L slots and nothing
    // is left for the merge kernel (n_evict = 0).
    bool zdone = false;
    if (ZS && zl) {
        Cand b{0ull, 0, -1};
        for (int q = 0; q < CS; q++) {
            const Cand cq = cluster.map_shared_rank(&S, q)->zbest;
            if (cq.slot >= 0 && cq.key > b.key) b = cq;
        }
        const int cp = b.slot;
        zdone = cp >= 0;
        if (zdone && r == 0) {
            const int e = victim;
            float kef = 0.f, kcf = 0.f, vef = 0.f, vcf = 0.f;
            if (tid < kD) {
                kef = bf2f(a.K[(ubase + e) * kD + tid]);
                kcf = bf2f(a.K[(ubase + cp) * kD + tid]);
                vef = bf2f(a.V[(ubase + e) * kD + tid]);
                vcf = bf2f(a.V[(ubase + cp) * kD + tid]);
                float qbs = 0.f;                      // sum of the group's queries
                for (int h = 0; h < G; h++) qbs += bf2f(a.q[((size_t)u * G + h) * kD + tid]);
                const float se = warp_sum(qbs * kef), sc = warp_sum(qbs * kcf);
                if (lane == 0) {
                    S.zred[w][0] = se;
                    S.zred[w][1] = sc;
                }
            }
            __syncthreads();
            if (tid == 0) {
                const float scale = rsqrtf((float)kD) / (float)G;
                const float xe = (S.zred[0][0] + S.zred[1][0] + S.zred[2][0] + S.zred[3][0]) * scale;
                const float xc = (S.zred[0][1] + S.zred[1][1] + S.zred[2][1] + S.zred[3][1]) * scale;
                const float pe = a.votes ? (float)a.votes[ubase + e] : 1.f;
                const float pc = a.votes ? (float)a.votes[ubase + cp] : 1.f;
                const float m = fmaxf(xe, xc);
                const float we = pe * expf(xe - m), wc = pc * expf(xc - m), W = we + wc;
                const float le = we / W, lc = wc / W;
                const float xt = le * xe + lc * xc;
                const float ell = m + logf(W / (pe + pc));
                const bool guard = fabsf(xt) < (float)KVC_ZIP_EPS;
                S.zcoef[0] = le;
                S.zcoef[1] = lc;
                S.zcoef[2] = guard ? 0.f : ell / xt;
                S.zcoef[3] = guard ? 1.f : 0.f;
            }
            __syncthreads();
            if (tid < kD) {
                const float le = S.zcoef[0], lc = S.zcoef[1];
                const float kr = S.zcoef[3] != 0.f ? 0.5f * (kef + kcf) : (le * kef + lc * kcf) * S.zcoef[2];
                const float vr = le * vef + lc * vcf;
                a.K[(ubase + cp) * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(kr));
                a.V[(ubase + cp) * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(vr));
            }
            if (tid == kD) {
                if (a.votes) a.votes[ubase + cp] += a.votes[ubase + e];
                a.util[ubase + cp] += a.util[ubase + e];
            }
            __syncthreads();                          // the victim's rows were read
            uint16_t *kd = a.K + (ubase + e) * kD;
            uint16_t *vd = a.V + (ubase + e) * kD;
            if (tid < 32) {
                reinterpret_cast<uint2 *>(kd)[tid] = reinterpret_cast<const uint2 *>(knew)[tid];
                reinterpret_cast<uint2 *>(vd)[tid] = reinterpret_cast<const uint2 *>(vnew)[tid];
            } else if (tid == 32) {
                if (a.votes) a.votes[ubase + e] = 1;
                a.pos[ubase + e] = a.new_pos;
                a.util[ubase + e] = __longlong_as_double(0x7ff0000000000000ll);
            }
        }
    }
    if (!a.merge)
        for (int e = r0 + tid; e < r1; e += blockDim.x) a.mu_v[(size_t)u * kD + e] = S.muv[e];
    if (r == 0) {
        if (!a.merge)
            for (int e = tid; e < kD; e += blockDim.x) a.mu_k[(size_t)u * kD + e] = S.muk[e];
        if (tid == 0) {
            if (!a.merge) a.mn[u] = n1;
            a.n_evict[u] = zdone ? 0 : 1;
            if (a.evict_idx) a.evict_idx[(size_t)u * a.kmax] = victim;
            if (a.evict_pos) a.evict_pos[(size_t)u * a.kmax] = S.vpos;
        }
    }
    if (refresh && !a.merge) write_back_C();
    // ------------------------------------------------ the new token's slot
    if (a.merge && !zdone) {
        // appended at slot L; the merge that follows refills the victim's
        // slot from it and restores len = L
        if (r == CS - 1) {
            uint16_t *kd = a.K + (ubase + L) * kD;
            uint16_t *vd = a.V + (ubase + L) * kD;
            if (tid < 32) {
                reinterpret_cast<uint2 *>(kd)[tid] = reinterpret_cast<const uint2 *>(knew)[tid];
                reinterpret_cast<uint2 *>(vd)[tid] = reinterpret_cast<const uint2 *>(vnew)[tid];
            } else if (tid == 32) {
                if (a.votes) a.votes[ubase + L] = 1;
                a.pos[ubase + L] = a.new_pos;
                a.util[ubase + L] = refresh ? S.vm : __longlong_as_double(0x7ff0000000000000ll);
                a.len[u] = L + 1;
            }
        }
    } else if (victim != L && r == vic_owner) {
        uint16_t *kd = a.K + (ubase + victim) * kD;
        uint16_t *vd = a.V + (ubase + victim) * kD;
        if (tid < 32) {
            reinterpret_cast<uint2 *>(kd)[tid] = reinterpret_cast<const uint2 *>(knew)[tid];
            reinterpret_cast<uint2 *>(vd)[tid] = reinterpret_cast<const uint2 *>(vnew)[tid];
        } else if (tid == 32) {
            if (a.votes) a.votes[ubase + victim] = 1;
            a.pos[ubase + victim] = a.new_pos;
            a.util[ubase + victim] = refresh ? cluster.map_shared_rank(&S, CS - 1)->vm
                                             : __longlong_as_double(0x7ff0000000000000ll);
        }
    }
    if (tid == 0 && S.bad) record_status(a.status, KVC_ERR_TIMEOUT);
    cluster.sync();             // no CTA leaves while another may read its shared memory
}

template <int G>
static cudaError_t launch_fused_g(const FusedArgs &a0, int U, int CS, cudaStream_t st)
{
    FusedArgs a = a0;
    const size_t sel = align_up((size_t)(a.chunk + 1) * 8) + align_up((size_t)(a.chunk + 1) * 4) +
                       align_up((size_t)(a.chunk + 1)) +
                       (size_t)(kWarps + kFusedMaxCS + 1) * kMaxQueue * sizeof(Cand);
    if (sel > (size_t)kStages * kTileBytes) return cudaErrorNotSupported;
    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)U * (uint64_t)a.cap;
    if (rows >= (1ull << 31) || !make_row_map(&tmK, a.K, rows, kTile) || !make_row_map(&tmV, a.V, rows, kTile))
        return cudaErrorNotSupported;
    const size_t dyn = 1024 + (size_t)kStages * kTileBytes + align_up((size_t)G * (a.chunk + 1) * 4);
    // merge mode with G = 2 or 4 and R >= 1 searches the partner in pass 1
    auto kern = fused_step_kernel<G, false>;
    if constexpr (G == 2 || G == 4)
        if (a.merge && a.R >= 1) kern = fused_step_kernel<G, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    (void)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(U * CS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, tmK, tmV);
}

int fused_cluster_size(int U, int L)
{
    int cs = (L + 2047) / 2048;                        // about 1-2 K slots per CTA
    const int want = (4 * 152 + U - 1) / U;            // fill the SMs for small U
    cs = max(cs, min(want, (L + 31) / 32));
    cs = max(1, min(kFusedMaxCS, cs));
    return cs;
}

cudaError_t launch_fused_step(const kvc_params &p, int t, int new_pos, const uint16_t *q,
                              const uint16_t *k_new, const uint16_t *v_new, const kvc_cache &c,
                              const kvc_moments &m, float *o, double *probs, int kmax,
                              int32_t *evict_idx, int32_t *evict_pos, int32_t *n_evict,
                              const DecodeWs &ws, cudaStream_t st, const float *rr)
{
    if (p.rule == KVC_RULE_MI && (rr == nullptr || p.refresh_period != 1)) return cudaErrorNotSupported;
    if (p.refresh_period > kMaxQueue) return cudaErrorNotSupported;
    // merge mode: every unit must find a partner (positions are distinct, so
    // at most R of the other L slots are recent: R < L guarantees one), and
    // the victims must be published for the merge kernel
    if (p.merge && (p.merge_recent >= p.L || !evict_idx)) return cudaErrorNotSupported;
    const int CS = fused_cluster_size(p.U, p.L);
    const int chunk = (p.L + CS - 1) / CS;
    if (chunk > kFusedMaxChunk || p.L + 1 > p.cap) return cudaErrorNotSupported;
    FusedArgs a{q, k_new, v_new, c.K, c.V, c.votes, c.pos, c.util, c.len,
                m.n, m.mu_k, m.mu_v, m.C, o, probs, evict_idx, evict_pos, n_evict,
                ws.pend, ws.status, p.budget, rr, p.cap, p.L, p.refresh_period, p.rule,
                p.correction, t, new_pos, kmax, chunk, p.alpha, p.merge, p.merge_recent};
    switch (p.G) {
    case 1: return launch_fused_g<1>(a, p.U, CS, st);
    case 2: return launch_fused_g<2>(a, p.U, CS, st);
    case 4: return launch_fused_g<4>(a, p.U, CS, st);
    case 8: return launch_fused_g<8>(a, p.U, CS, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace kvc
