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
#include <math.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace cg = cooperative_groups;

namespace kvc {

constexpr int kFusedMaxChunk = 4096;   // slots per CTA
constexpr int kFusedMaxCS = 8;         // CTAs per cluster
constexpr int kMaxQueue = kPendStride - 2;

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
    int cap, L, T, rule, correction, t, new_pos, kmax, chunk;
    float alpha;
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
    float qs[G][kD];            // q / sqrt(d), fp32
    float red[8][G];
    float pM[G], pl[G];         // this CTA's partial max / sum
    float po[G][kD];            // this CTA's partial unnormalized output
    float gM[G], gl[G];         // merged
    float fR[G][kD];
    float lzR[G];
    float mass[G];
    float ae[G];                // exp(x_e - M) of the victim (refresh)
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
    float wR[G];
    double vm;                  // utility of the new token (refresh, last CTA)
    Cand cand[kMaxQueue];
    int ncand;
    Cand bc[8];
    int victim;                 // slot index of the victim (L = the new token)
    int qvalid;
    int direct;
};

template <int G>
__global__ void __launch_bounds__(256, 2) fused_step_kernel(FusedArgs a)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int CS = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    const int u = blockIdx.x / CS;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int grp = lane >> 3, c = lane & 7;

    __shared__ FusedSmem<G> S;
    extern __shared__ __align__(16) unsigned char dyn[];
    const int ch = a.chunk;
    float *xsb = reinterpret_cast<float *>(dyn);                       // [G][ch + 1]
    double *msm = reinterpret_cast<double *>(dyn + align_up((size_t)G * (ch + 1) * 4));
    int32_t *possm = reinterpret_cast<int32_t *>(reinterpret_cast<unsigned char *>(msm) +
                                                  align_up((size_t)(ch + 1) * 8));
    unsigned char *chosen = reinterpret_cast<unsigned char *>(possm) + align_up((size_t)(ch + 1) * 4);
    auto XS = [&](int h, int li) -> float & { return xsb[h * (ch + 1) + li]; };

    const int L = a.L;
    const bool refresh = is_refresh(a.t, a.T);
    const size_t ubase = (size_t)u * a.cap;
    const int n_old = a.len[u];
    if (n_old != L) {                      // uniform over the cluster
        if (r == 0 && tid == 0) {
            record_status(a.status, KVC_ERR_SHAPE);
            a.n_evict[u] = 0;
        }
        return;
    }
    const int s0 = min(L, r * ch), s1 = min(L, s0 + ch);
    const bool has_new = refresh && (r == CS - 1);
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
    if (tid == 0) { S.qvalid = 0; S.direct = 0; S.ncand = 0; S.n0 = a.mn[u]; }
    __syncthreads();

    // ------------------------------------------------ victim (non-refresh)
    int victim = -1;
    if (!refresh) {
        const int tr = a.t - ((a.t - 1) % a.T);      // last refresh step
        const int idx = a.t - tr;                      // 1 .. T-1
        const int32_t *pq = a.pend + (size_t)u * kPendStride;
        if (pq[0] == tr && pq[1] >= idx) {
            victim = pq[2 + idx - 1];
            if (victim < 0 || victim >= L) victim = -1;
        }
        if (victim < 0) {
            // lowest scored (utility, position) over the unit: per-CTA argmin
            Cand best{~0ull, 0x7fffffff, -1};
            for (int i = s0 + tid; i < s1; i += blockDim.x) {
                const double m = a.util[ubase + i];
                if (isinf(m)) continue;
                Cand cd{double_key(m), a.pos[ubase + i], i};
                if (cand_less(cd, best)) best = cd;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                Cand o = shfl_cand(best, m);
                if (cand_less(o, best)) best = o;
            }
            if (lane == 0) S.bc[w] = best;
            __syncthreads();
            if (tid == 0) {
                Cand b = S.bc[0];
                for (int j = 1; j < 8; j++)
                    if (cand_less(S.bc[j], b)) b = S.bc[j];
                S.cand[0] = b;
                S.ncand = b.slot >= 0 ? 1 : 0;
            }
            cluster.sync();
            Cand b{~0ull, 0x7fffffff, -1};
            for (int q = 0; q < CS; q++) {
                FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
                if (R->ncand > 0 && cand_less(R->cand[0], b)) b = R->cand[0];
            }
            victim = b.slot;
            cluster.sync();
            if (victim < 0) {                       // no scored slot: refuse
                if (r == 0 && tid == 0) {
                    record_status(a.status, KVC_ERR_INVALID_ARG);
                    a.n_evict[u] = 0;
                }
                return;
            }
        }
        // the owner publishes the victim's key / value / vote / position
        if (victim >= s0 && victim < s1) {
            const uint16_t *kr = a.K + (ubase + victim) * kD;
            const uint16_t *vr = a.V + (ubase + victim) * kD;
            for (int e = tid; e < kD; e += blockDim.x) {
                S.pk[e] = bf2f(kr[e]);
                S.pv[e] = bf2f(vr[e]);
            }
            if (tid == 0) {
                S.pvp = a.votes ? (float)a.votes[ubase + victim] : 1.f;
                S.pvpos = a.pos[ubase + victim];
            }
        }
    }

    // ------------------------------------------------ pass 1: logits
    float qf[G][16];
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int j = 0; j < 8; j++) {
            qf[h][j] = S.qs[h][8 * c + j];
            qf[h][8 + j] = S.qs[h][64 + 8 * c + j];
        }
    float mx[G];
#pragma unroll
    for (int h = 0; h < G; h++) mx[h] = -INFINITY;
    for (int base = w * 4; base < nloc; base += 32) {
        const int li = base + grp;
        const bool ok = li < nloc;
        const int i = s0 + li;                              // == L for the virtual slot
        const bool isnew = ok && (i == L || i == victim);
        float kf[16];
        if (ok) {
            const uint16_t *kr = isnew ? knew : a.K + (ubase + i) * kD;
            uint4 r0 = isnew ? *reinterpret_cast<const uint4 *>(kr + 8 * c) : ldg_nc_v4(kr + 8 * c);
            uint4 r1 = isnew ? *reinterpret_cast<const uint4 *>(kr + 64 + 8 * c)
                             : ldg_nc_v4(kr + 64 + 8 * c);
            unpack8(r0, kf);
            unpack8(r1, kf + 8);
        } else {
#pragma unroll
            for (int j = 0; j < 16; j++) kf[j] = 0.f;
        }
        float part[G];
#pragma unroll
        for (int h = 0; h < G; h++) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) acc = fmaf(qf[h][j], kf[j], acc);
            part[h] = acc;
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1)
#pragma unroll
            for (int h = 0; h < G; h++) part[h] += __shfl_xor_sync(kFull, part[h], m);
        if (ok) {
            const float lnp = (!isnew && a.votes) ? logf((float)a.votes[ubase + i]) : 0.f;
#pragma unroll
            for (int h = 0; h < G; h++) {
                const float x = part[h] + lnp;
                mx[h] = fmaxf(mx[h], x);
                if (c == h) XS(h, li) = x;
            }
        }
    }
#pragma unroll
    for (int h = 0; h < G; h++) {
        const float v = warp_max(mx[h]);
        if (lane == 0) S.red[w][h] = v;
    }
    __syncthreads();
    if (tid < G) {
        float v = S.red[0][tid];
        for (int j = 1; j < 8; j++) v = fmaxf(v, S.red[j][tid]);
        S.pM[tid] = v;
    }
    __syncthreads();

    // ------------------------------------------------ pass 2: p v
    auto pv_pass = [&](int skip, const float *Mref) {
        float acc[G][16], lsum[G], Mr[G];
#pragma unroll
        for (int h = 0; h < G; h++) {
            Mr[h] = Mref[h];
            lsum[h] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) acc[h][j] = 0.f;
        }
        for (int base = w * 4; base < nloc; base += 32) {
            const int li = base + grp;
            const int i = s0 + li;
            if (li < nloc && i != skip) {
                const bool isnew = (i == L || i == victim);
                const uint16_t *vr = isnew ? vnew : a.V + (ubase + i) * kD;
                uint4 r0 = isnew ? *reinterpret_cast<const uint4 *>(vr + 8 * c) : ldg_nc_v4(vr + 8 * c);
                uint4 r1 = isnew ? *reinterpret_cast<const uint4 *>(vr + 64 + 8 * c)
                                 : ldg_nc_v4(vr + 64 + 8 * c);
                float vf[16];
                unpack8(r0, vf);
                unpack8(r1, vf + 8);
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float p = expf(XS(h, li) - Mr[h]);
                    if (c == 0) lsum[h] += p;
#pragma unroll
                    for (int j = 0; j < 16; j++) acc[h][j] = fmaf(p, vf[j], acc[h][j]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < G; h++) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                acc[h][j] += __shfl_xor_sync(kFull, acc[h][j], 8);
                acc[h][j] += __shfl_xor_sync(kFull, acc[h][j], 16);
            }
            lsum[h] = warp_sum(lsum[h]);
        }
        for (int e = tid; e < G * kD; e += blockDim.x) S.po[e / kD][e % kD] = 0.f;
        __syncthreads();
        if (grp == 0)
#pragma unroll
            for (int h = 0; h < G; h++)
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    atomicAdd(&S.po[h][8 * c + j], acc[h][j]);
                    atomicAdd(&S.po[h][64 + 8 * c + j], acc[h][8 + j]);
                }
        if (lane == 0)
#pragma unroll
            for (int h = 0; h < G; h++) S.red[w][h] = lsum[h];
        __syncthreads();
        if (tid < G) {
            float l = 0.f;
            for (int j = 0; j < 8; j++) l += S.red[j][tid];
            S.pl[tid] = l;
        }
        __syncthreads();
    };
    pv_pass(-1, S.pM);

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

    int vic_owner;
    if (refresh) {
        // -------------------------------------------- probabilities + utilities
        const double al = (double)a.alpha;
        for (int li = tid; li < nloc; li += blockDim.x) {
            const int i = s0 + li;
            double s = 0.0;
#pragma unroll
            for (int h = 0; h < G; h++) s += exp_wide(XS(h, li) - S.gM[h]) / (double)S.gl[h];
            s /= G;
            const bool isv = (i == L);
            const double m = isv ? __longlong_as_double(0x7ff0000000000000ll) : a.util[ubase + i];
            double mn;
            if (isinf(m)) mn = s;
            else if (a.rule == KVC_RULE_SINGLE) mn = s;
            else if (a.rule == KVC_RULE_CUMULATIVE) mn = m + s;
            else mn = al * m + (1.0 - al) * s;
            msm[li] = mn;
            possm[li] = isv ? a.new_pos : a.pos[ubase + i];
            chosen[li] = 0;
            if (!isv) a.util[ubase + i] = mn;
            else S.vm = mn;
            if (a.probs) a.probs[ubase + i] = s;
        }
        __syncthreads();
        // -------------------------------------------- local T lowest
        const int want = min(a.T, nloc);
        for (int rnd = 0; rnd < want; rnd++) {
            Cand best{~0ull, 0x7fffffff, -1};
            for (int li = tid; li < nloc; li += blockDim.x) {
                if (chosen[li]) continue;
                Cand cd{double_key(msm[li]), possm[li], s0 + li};
                if (cand_less(cd, best)) best = cd;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                Cand o = shfl_cand(best, m);
                if (cand_less(o, best)) best = o;
            }
            if (lane == 0) S.bc[w] = best;
            __syncthreads();
            if (tid == 0) {
                Cand b = S.bc[0];
                for (int j = 1; j < 8; j++)
                    if (cand_less(S.bc[j], b)) b = S.bc[j];
                S.cand[rnd] = b;
                chosen[b.slot - s0] = 1;
            }
            __syncthreads();
        }
        if (tid == 0) S.ncand = want;
        cluster.sync();                                                // candidates visible
        // every CTA merges the candidate lists the same way
        if (tid == 0) {
            int ptr[kFusedMaxCS];
            for (int q = 0; q < CS; q++) ptr[q] = 0;
            Cand sel[kMaxQueue];
            int nsel = 0;
            while (nsel < a.T) {
                int bq = -1;
                Cand b{~0ull, 0x7fffffff, -1};
                for (int q = 0; q < CS; q++) {
                    FusedSmem<G> *R = cluster.map_shared_rank(&S, q);
                    if (ptr[q] < R->ncand && cand_less(R->cand[ptr[q]], b)) {
                        b = R->cand[ptr[q]];
                        bq = q;
                    }
                }
                if (bq < 0) break;
                ptr[bq]++;
                sel[nsel++] = b;
            }
            S.victim = sel[0].slot;
            if (r == 0) {
                int32_t *pq = a.pend + (size_t)u * kPendStride;
                pq[0] = a.t;
                pq[1] = nsel - 1;
                for (int j = 1; j < nsel; j++)
                    pq[2 + j - 1] = sel[j].slot == L ? sel[0].slot : sel[j].slot;
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
                S.pvp = (isv || !a.votes) ? 1.f : (float)a.votes[ubase + victim];
                S.pvpos = isv ? a.new_pos : possm[li];
            }
        }
        cluster.sync();                                                // victim visible
        FusedSmem<G> *O = cluster.map_shared_rank(&S, vic_owner);
        if (tid < G) {
            const float ae = O->ae_pub[tid];
            S.ae[tid] = ae;
            S.mass[tid] = ae / S.gl[tid];
            if (S.mass[tid] > 0.5f) atomicExch(&S.direct, 1);
        }
        for (int e = tid; e < kD; e += blockDim.x) {
            S.vk[e] = O->pk[e];
            S.vv[e] = O->pv[e];
        }
        if (tid == 0) { S.vp = O->pvp; S.vpos = O->pvpos; }
        __syncthreads();
        if (!S.direct) {
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
        cluster.sync();                                                // victim visible
        FusedSmem<G> *O = cluster.map_shared_rank(&S, vic_owner);
        for (int e = tid; e < kD; e += blockDim.x) {
            S.vk[e] = O->pk[e];
            S.vv[e] = O->pv[e];
        }
        if (tid == 0) { S.vp = O->pvp; S.vpos = O->pvpos; }
        __syncthreads();
    }

    // ------------------------------------------------ moment fold (West)
    const float n0 = S.n0;
    const float pe = S.vp;
    const float n1 = n0 + pe;
    const float fw = pe / n1;
    for (int e = tid; e < kD; e += blockDim.x) {
        const float mk = S.mk0[e], mv = S.mv0[e];
        S.muk[e] = mk + (S.vk[e] - mk) * fw;
        S.muv[e] = mv + (S.vv[e] - mv) * fw;
        S.vk[e] -= mk;                  // delta k (old mean)
        S.vv[e] -= mv;                  // delta v
    }
    __syncthreads();
    const int rows = (kD + CS - 1) / CS;
    const int r0 = min(kD, r * rows), r1 = min(kD, r0 + rows);
    const float sc_old = n0 / n1, sc_rank = pe * n0 / (n1 * n1);
    float *Cu = a.C + (size_t)u * kD * kD;
    // thread -> (row, quarter of columns); 4 threads per row.  The loop bound
    // is uniform so that every lane reaches the shuffles.
    for (int rb = r0; rb < r1; rb += (int)blockDim.x >> 2) {
        const int rr = rb + (tid >> 2);
        const bool valid = rr < r1;
        const int q4 = tid & 3;
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; h++) acc[h] = 0.f;
        if (valid) {
            float *crow = Cu + (size_t)rr * kD + q4 * 32;
            const float dv = S.vv[rr] * sc_rank;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 cv = *reinterpret_cast<float4 *>(crow + j);
                cv.x = fmaf(cv.x, sc_old, dv * S.vk[q4 * 32 + j]);
                cv.y = fmaf(cv.y, sc_old, dv * S.vk[q4 * 32 + j + 1]);
                cv.z = fmaf(cv.z, sc_old, dv * S.vk[q4 * 32 + j + 2]);
                cv.w = fmaf(cv.w, sc_old, dv * S.vk[q4 * 32 + j + 3]);
                *reinterpret_cast<float4 *>(crow + j) = cv;
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float *qq = &S.qs[h][q4 * 32 + j];
                    acc[h] = fmaf(cv.x, qq[0], acc[h]);
                    acc[h] = fmaf(cv.y, qq[1], acc[h]);
                    acc[h] = fmaf(cv.z, qq[2], acc[h]);
                    acc[h] = fmaf(cv.w, qq[3], acc[h]);
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
    // correction weights (every CTA, full dot with the new key mean)
    if (w < G) {
        float s = 0.f;
        for (int j = lane; j < kD; j += 32) s = fmaf(S.qs[w][j], S.muk[j], s);
        s = warp_sum(s);
        if (lane == 0) {
            const float logZE = logf(n1) + s;
            S.wR[w] = 1.f / (1.f + expf(logZE - S.lzR[w]));
        }
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
    for (int e = r0 + tid; e < r1; e += blockDim.x) a.mu_v[(size_t)u * kD + e] = S.muv[e];
    if (r == 0) {
        for (int e = tid; e < kD; e += blockDim.x) a.mu_k[(size_t)u * kD + e] = S.muk[e];
        if (tid == 0) {
            a.mn[u] = n1;
            a.n_evict[u] = 1;
            if (a.evict_idx) a.evict_idx[(size_t)u * a.kmax] = victim;
            if (a.evict_pos) a.evict_pos[(size_t)u * a.kmax] = S.vpos;
        }
    }
    // ------------------------------------------------ the new token's slot
    if (victim != L && r == vic_owner) {
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
    cluster.sync();             // no CTA leaves while another may read its shared memory
}

template <int G>
static cudaError_t launch_fused_g(const FusedArgs &a0, int U, int CS, cudaStream_t st)
{
    FusedArgs a = a0;
    const size_t dyn = align_up((size_t)G * (a.chunk + 1) * 4) + align_up((size_t)(a.chunk + 1) * 8) +
                       align_up((size_t)(a.chunk + 1) * 4) + align_up((size_t)(a.chunk + 1));
    cudaError_t e = cudaFuncSetAttribute(fused_step_kernel<G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fused_step_kernel<G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    (void)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(U * CS);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_step_kernel<G>, a);
}

int fused_cluster_size(int U, int L)
{
    int cs = (L + kFusedMaxChunk - 1) / kFusedMaxChunk;
    const int want = (4 * 152 + U - 1) / U;            // fill the SMs for small U
    cs = max(cs, min(want, (L + 31) / 32));
    cs = max(1, min(kFusedMaxCS, cs));
    return cs;
}

cudaError_t launch_fused_step(const kvc_params &p, int t, int new_pos, const uint16_t *q,
                              const uint16_t *k_new, const uint16_t *v_new, const kvc_cache &c,
                              const kvc_moments &m, float *o, double *probs, int kmax,
                              int32_t *evict_idx, int32_t *evict_pos, int32_t *n_evict,
                              const DecodeWs &ws, cudaStream_t st)
{
    if (p.refresh_period > kMaxQueue) return cudaErrorNotSupported;
    const int CS = fused_cluster_size(p.U, p.L);
    const int chunk = (p.L + CS - 1) / CS;
    if (chunk > kFusedMaxChunk || p.L + 1 > p.cap) return cudaErrorNotSupported;
    FusedArgs a{q, k_new, v_new, c.K, c.V, c.votes, c.pos, c.util, c.len,
                m.n, m.mu_k, m.mu_v, m.C, o, probs, evict_idx, evict_pos, n_evict,
                ws.pend, ws.status, p.cap, p.L, p.refresh_period, p.rule, p.correction,
                t, new_pos, kmax, chunk, p.alpha};
    switch (p.G) {
    case 1: return launch_fused_g<1>(a, p.U, CS, st);
    case 2: return launch_fused_g<2>(a, p.U, CS, st);
    case 4: return launch_fused_g<4>(a, p.U, CS, st);
    case 8: return launch_fused_g<8>(a, p.U, CS, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace kvc
