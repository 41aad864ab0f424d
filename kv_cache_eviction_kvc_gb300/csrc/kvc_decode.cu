// kvc_decode.cu -- the decode step as five separate kernels (any number of
// victims per step; step 1 over the whole prefill cache runs here).
//
//   attend_chunk  : append + vote-biased logits + per-chunk softmax partials
//   attend_final  : split merge -> lse, f_all; head-mean probabilities
//   aggregate     : utility update (refresh steps) + lowest-(m, pos) select
//   moment_fold   : weighted Chan/West merge of the victims into (n, mu, C)
//   correct       : retained-only output (identity or direct) + correction
//   compact       : fill holes below the new length from slots above it
//
// Method: MomentKV Algorithm 1 (phase order), sec 4.1-4.2, App. A.1, C.2;
// InertiaKV sec 3.1 eqs 1-4; KeepKV eqs 3, 6, 23.
#include <math.h>

#include "kvc_common.cuh"
#include "kvc_general.h"
#include "kvc_internal.h"

namespace kvc {

// ===================================================================== attend
//
// One CTA = one unit x one chunk of kAttendChunk slots, 8 warps.  A warp
// works on 4 slots at a time: 8 lanes per slot, lane c holding dims
// [8c, 8c+8) and [64+8c, 64+8c+8) (two coalesced 16-byte loads per row).
// Pass 1 computes the logits of the chunk into shared memory (and the
// workspace when probabilities are wanted) and the chunk max per head;
// pass 2 streams V with p = exp(x - max): no online rescaling is needed.

struct AttendArgs {
    const uint16_t *q, *k_new, *v_new;
    uint16_t *K, *V;
    int32_t *votes, *pos;
    double *util;
    const int32_t *len;
    float *xbuf, *part;
    int32_t *nlen, *status;
    int U, cap, max_len, new_pos, S;
    int want_x;
    int append;        // 0: attend over the live slots as they are (no new token)
};

template <int G>
__global__ void __launch_bounds__(256) attend_chunk_kernel(AttendArgs a)
{
    constexpr int CH = kAttendChunk;
    constexpr int kBuf = (G * CH > 8 * G * kD) ? G * CH : 8 * G * kD;
    __shared__ __align__(16) float sbuf[kBuf];
    __shared__ float red[8][G];
    float (*xs)[CH] = reinterpret_cast<float (*)[CH]>(sbuf);          // pass 1-2
    float (*accs)[G][kD] = reinterpret_cast<float (*)[G][kD]>(sbuf);  // after

    const int u = blockIdx.x, s = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int grp = lane >> 3, c = lane & 7;

    const int n_old = a.len[u];
    const int n = a.append ? n_old + 1 : n_old;
    if (n_old < 0 || n > a.max_len || n > a.cap) {
        if (s == 0 && tid == 0) {
            record_status(a.status, KVC_ERR_SHAPE);
            a.nlen[u] = -1;
        }
        return;
    }
    const int s0 = s * CH;
    if (s0 >= n) return;
    const int s1 = min(n, s0 + CH);
    if (s == 0 && tid == 0) a.nlen[u] = n;

    const size_t ubase = (size_t)u * a.cap;
    const uint16_t *knew = a.append ? a.k_new + (size_t)u * kD : nullptr;
    const uint16_t *vnew = a.append ? a.v_new + (size_t)u * kD : nullptr;

    // the chunk holding the new slot appends it
    if (a.append && n_old >= s0 && n_old < s1) {
        if (tid < 32) {
            uint16_t *kd = a.K + (ubase + n_old) * kD;
            uint16_t *vd = a.V + (ubase + n_old) * kD;
            reinterpret_cast<uint2 *>(kd)[tid] = reinterpret_cast<const uint2 *>(knew)[tid];
            reinterpret_cast<uint2 *>(vd)[tid] = reinterpret_cast<const uint2 *>(vnew)[tid];
        } else if (tid == 32) {
            if (a.votes) a.votes[ubase + n_old] = 1;
            a.pos[ubase + n_old] = a.new_pos;
            a.util[ubase + n_old] = __longlong_as_double(0x7ff0000000000000ll);
        }
    }

    // q of the group, scaled by 1/sqrt(d), dims of this lane
    const float rs = rsqrtf((float)kD);
    float qf[G][16];
#pragma unroll
    for (int h = 0; h < G; h++) {
        const uint16_t *qh = a.q + ((size_t)u * G + h) * kD;
        uint4 r0 = *reinterpret_cast<const uint4 *>(qh + 8 * c);
        uint4 r1 = *reinterpret_cast<const uint4 *>(qh + 64 + 8 * c);
        unpack8(r0, qf[h]);
        unpack8(r1, qf[h] + 8);
#pragma unroll
        for (int j = 0; j < 16; j++) qf[h][j] *= rs;
    }

    // ---- pass 1: logits (two groups of 4 slots per warp and iteration:
    // both groups' rows are requested before either is used)
    float mx[G];
#pragma unroll
    for (int h = 0; h < G; h++) mx[h] = -INFINITY;
    for (int base = s0 + w * 8; base < s1; base += 64) {
        uint4 kr[2][2];
#pragma unroll
        for (int q2 = 0; q2 < 2; q2++) {
            const int i = base + 4 * q2 + grp;
            if (i < s1) {
                const uint16_t *kp = (i == n_old) ? knew : a.K + (ubase + i) * kD;
                kr[q2][0] = (i == n_old) ? *reinterpret_cast<const uint4 *>(kp + 8 * c)
                                         : ldg_nc_v4(kp + 8 * c);
                kr[q2][1] = (i == n_old) ? *reinterpret_cast<const uint4 *>(kp + 64 + 8 * c)
                                         : ldg_nc_v4(kp + 64 + 8 * c);
            } else {
                kr[q2][0] = kr[q2][1] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int q2 = 0; q2 < 2; q2++) {
            const int i = base + 4 * q2 + grp;
            const bool ok = i < s1;
            float kf[16];
            unpack8(kr[q2][0], kf);
            unpack8(kr[q2][1], kf + 8);
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
                float lnp = 0.f;
                if (a.votes && i != n_old) lnp = logf((float)a.votes[ubase + i]);
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float x = part[h] + lnp;
                    mx[h] = fmaxf(mx[h], x);
                    if (c == h) {
                        xs[h][i - s0] = x;
                        if (a.want_x) a.xbuf[((size_t)u * G + h) * a.cap + i] = x;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < G; h++) {
        float v = warp_max(mx[h]);
        if (lane == 0) red[w][h] = v;
    }
    __syncthreads();
    float M[G];
#pragma unroll
    for (int h = 0; h < G; h++) {
        float v = red[0][h];
#pragma unroll
        for (int j = 1; j < 8; j++) v = fmaxf(v, red[j][h]);
        M[h] = v;
    }
    __syncthreads();

    // ---- pass 2: p = exp(x - M), accumulate p v and sum p
    float acc[G][16];
    float lsum[G];
#pragma unroll
    for (int h = 0; h < G; h++) {
        lsum[h] = 0.f;
#pragma unroll
        for (int j = 0; j < 16; j++) acc[h][j] = 0.f;
    }
    for (int base = s0 + w * 8; base < s1; base += 64) {
        uint4 vr[2][2];
#pragma unroll
        for (int q2 = 0; q2 < 2; q2++) {
            const int i = base + 4 * q2 + grp;
            if (i < s1) {
                const uint16_t *vp = (i == n_old) ? vnew : a.V + (ubase + i) * kD;
                vr[q2][0] = (i == n_old) ? *reinterpret_cast<const uint4 *>(vp + 8 * c)
                                         : ldg_nc_v4(vp + 8 * c);
                vr[q2][1] = (i == n_old) ? *reinterpret_cast<const uint4 *>(vp + 64 + 8 * c)
                                         : ldg_nc_v4(vp + 64 + 8 * c);
            }
        }
#pragma unroll
        for (int q2 = 0; q2 < 2; q2++) {
            const int i = base + 4 * q2 + grp;
            if (i < s1) {
                float vf[16];
                unpack8(vr[q2][0], vf);
                unpack8(vr[q2][1], vf + 8);
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float p = expf(xs[h][i - s0] - M[h]);
                    if (c == 0) lsum[h] += p;
#pragma unroll
                    for (int j = 0; j < 16; j++) acc[h][j] = fmaf(p, vf[j], acc[h][j]);
                }
            }
        }
    }
    // reduce over the 4 slot groups of the warp
#pragma unroll
    for (int h = 0; h < G; h++) {
#pragma unroll
        for (int j = 0; j < 16; j++) {
            acc[h][j] += __shfl_xor_sync(kFull, acc[h][j], 8);
            acc[h][j] += __shfl_xor_sync(kFull, acc[h][j], 16);
        }
        lsum[h] = warp_sum(lsum[h]);
    }
    __syncthreads();   // every warp is done with xs before accs overwrites it
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; h++)
#pragma unroll
            for (int j = 0; j < 8; j++) {
                accs[w][h][8 * c + j] = acc[h][j];
                accs[w][h][64 + 8 * c + j] = acc[h][8 + j];
            }
    }
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < G; h++) red[w][h] = lsum[h];
    __syncthreads();
    float *pp = a.part + ((size_t)u * a.S + s) * G * (kD + 2);
    for (int e = tid; e < G * kD; e += blockDim.x) {
        const int h = e / kD, dd = e % kD;
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) v += accs[j][h][dd];
        pp[h * (kD + 2) + 2 + dd] = v;
    }
    if (tid < G) {
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) l += red[j][tid];
        pp[tid * (kD + 2) + 0] = M[tid];
        pp[tid * (kD + 2) + 1] = l;
    }
}

// Merge the split partials of a unit: global max and sum per head; CTA
// (u, 0) writes lse, f_all and the new length; every CTA writes the
// probabilities of its slot chunk.
struct FinalArgs {
    const float *part, *xbuf;
    const int32_t *nlen;
    int32_t *len;
    float *lse, *f_all;
    double *probs;
    int U, cap, S;
};

template <int G>
__global__ void __launch_bounds__(256) attend_final_kernel(FinalArgs a)
{
    __shared__ float Ms[G], Ls[G];
    __shared__ double Rl[G];
    const int u = blockIdx.x, s2 = blockIdx.y, tid = threadIdx.x;
    const int n = a.nlen[u];
    if (n <= 0) return;
    const int Su = (n + kAttendChunk - 1) / kAttendChunk;
    const float *pu = a.part + (size_t)u * a.S * G * (kD + 2);
    const int lane = tid & 31, w = tid >> 5;
    if (w < G) {
        const int h = w;
        float m = -INFINITY;
        for (int s = lane; s < Su; s += 32) m = fmaxf(m, pu[(size_t)s * G * (kD + 2) + h * (kD + 2)]);
        m = warp_max(m);
        float l = 0.f;
        for (int s = lane; s < Su; s += 32) {
            const float *ph = pu + (size_t)s * G * (kD + 2) + h * (kD + 2);
            l += ph[1] * expf(ph[0] - m);
        }
        l = warp_sum(l);
        if (lane == 0) { Ms[h] = m; Ls[h] = l; Rl[h] = 1.0 / (double)l; }
    }
    __syncthreads();
    if (s2 == 0) {
        if (tid == 0) a.len[u] = n;
        if (tid < G) a.lse[(size_t)u * G + tid] = Ms[tid] + logf(Ls[tid]);
        for (int e = tid; e < G * kD; e += blockDim.x) {
            const int h = e / kD, dd = e % kD;
            float v = 0.f;
            for (int s = 0; s < Su; s++) {
                const float *ph = pu + (size_t)s * G * (kD + 2) + h * (kD + 2);
                v += ph[2 + dd] * expf(ph[0] - Ms[h]);
            }
            a.f_all[((size_t)u * G + h) * kD + dd] = v / Ls[h];
        }
    }
    if (a.probs) {
        // s_i = (1/G) sum_h exp(x_hi - M_h) / l_h.  While the largest head
        // term is above e^-60 the sum is far inside fp32's range and fp32
        // carries it to a few units in the last place (the fused step forms
        // it the same way); below that the fp64 form keeps the range.  G is a
        // power of two, so the 1/G factor is exact.
        const int i0 = s2 * kProbsChunk, i1 = min(n, i0 + kProbsChunk);
        float rl32[G];
#pragma unroll
        for (int h = 0; h < G; h++) rl32[h] = (float)(Rl[h] * (1.0 / G));
        for (int i = i0 + tid; i < i1; i += blockDim.x) {
            float y[G], ymax = -INFINITY;
#pragma unroll
            for (int h = 0; h < G; h++) {
                y[h] = a.xbuf[((size_t)u * G + h) * a.cap + i] - Ms[h];
                ymax = fmaxf(ymax, y[h]);
            }
            double sv;
            if (ymax > -60.f) {
                float s32 = 0.f;
#pragma unroll
                for (int h = 0; h < G; h++) s32 = fmaf(expf(y[h]), rl32[h], s32);
                sv = (double)s32;
            } else {
                double sacc = 0.0;
#pragma unroll
                for (int h = 0; h < G; h++) sacc = fma(exp_wide(y[h]), Rl[h], sacc);
                sv = sacc * (1.0 / G);
            }
            a.probs[(size_t)u * a.cap + i] = sv;
        }
    }
}

template <int G>
static cudaError_t launch_attend_g(const kvc_params &p, int new_pos, int max_len,
                                   const uint16_t *q, const uint16_t *k_new,
                                   const uint16_t *v_new, const kvc_cache &c,
                                   float *lse, float *f_all, double *probs,
                                   const DecodeWs &ws, cudaStream_t st, bool append = true)
{
    const int S = (p.cap + kAttendChunk - 1) / kAttendChunk;
    const int Sl = (max_len + kAttendChunk - 1) / kAttendChunk;
    AttendArgs a{q, k_new, v_new, c.K, c.V, c.votes, c.pos, c.util, c.len,
                 ws.xbuf, ws.part, ws.nlen, ws.status, p.U, p.cap, max_len,
                 new_pos, S, probs != nullptr, append ? 1 : 0};
    dim3 g1(p.U, Sl);
    attend_chunk_kernel<G><<<g1, 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    FinalArgs f{ws.part, ws.xbuf, ws.nlen, c.len, lse, f_all, probs, p.U, p.cap, S};
    const int S2 = probs ? (max_len + kProbsChunk - 1) / kProbsChunk : 1;
    attend_final_kernel<G><<<dim3(p.U, S2), 256, 0, st>>>(f);
    return cudaGetLastError();
}

cudaError_t launch_attend(const kvc_params &p, int t, int new_pos, int max_len,
                          const uint16_t *q, const uint16_t *k_new,
                          const uint16_t *v_new, const kvc_cache &c,
                          float *lse, float *f_all, double *probs,
                          const DecodeWs &ws, cudaStream_t st)
{
    (void)t;
    switch (p.G) {
    case 1: return launch_attend_g<1>(p, new_pos, max_len, q, k_new, v_new, c, lse, f_all, probs, ws, st);
    case 2: return launch_attend_g<2>(p, new_pos, max_len, q, k_new, v_new, c, lse, f_all, probs, ws, st);
    case 4: return launch_attend_g<4>(p, new_pos, max_len, q, k_new, v_new, c, lse, f_all, probs, ws, st);
    case 8: return launch_attend_g<8>(p, new_pos, max_len, q, k_new, v_new, c, lse, f_all, probs, ws, st);
    default: return cudaErrorInvalidValue;
    }
}

template <int G>
static cudaError_t launch_final_g(const kvc_params &p, int max_len, const kvc_cache &c, float *lse,
                                  float *f, double *probs, const DecodeWs &ws, cudaStream_t st)
{
    const int S = (p.cap + kAttendChunk - 1) / kAttendChunk;
    FinalArgs fa{ws.part, ws.xbuf, ws.nlen, c.len, lse, f, probs, p.U, p.cap, S};
    const int S2 = probs ? (max_len + kProbsChunk - 1) / kProbsChunk : 1;
    attend_final_kernel<G><<<dim3(p.U, S2), 256, 0, st>>>(fa);
    return cudaGetLastError();
}

cudaError_t launch_attend_final(const kvc_params &p, int max_len, const kvc_cache &c, float *lse,
                                float *f, double *probs, const DecodeWs &ws, cudaStream_t st)
{
    switch (p.G) {
    case 1: return launch_final_g<1>(p, max_len, c, lse, f, probs, ws, st);
    case 2: return launch_final_g<2>(p, max_len, c, lse, f, probs, ws, st);
    case 4: return launch_final_g<4>(p, max_len, c, lse, f, probs, ws, st);
    case 8: return launch_final_g<8>(p, max_len, c, lse, f, probs, ws, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attend_retained(const kvc_params &p, int max_len, const uint16_t *q,
                                   const kvc_cache &c, float *lse, float *f, const DecodeWs &ws,
                                   cudaStream_t st)
{
    switch (p.G) {
    case 1: return launch_attend_g<1>(p, 0, max_len, q, nullptr, nullptr, c, lse, f, nullptr, ws, st, false);
    case 2: return launch_attend_g<2>(p, 0, max_len, q, nullptr, nullptr, c, lse, f, nullptr, ws, st, false);
    case 4: return launch_attend_g<4>(p, 0, max_len, q, nullptr, nullptr, c, lse, f, nullptr, ws, st, false);
    case 8: return launch_attend_g<8>(p, 0, max_len, q, nullptr, nullptr, c, lse, f, nullptr, ws, st, false);
    default: return cudaErrorInvalidValue;
    }
}

// ================================================================== aggregate
//
// One CTA per unit.  Refresh steps update the utilities in place; then the
// k = len - L victims are the k smallest (utility, position) keys among the
// scored slots: a 4-pass 8-bit radix select on the utility's order key finds
// the k-th smallest utility, a second select on positions settles the group
// of equal utilities at the threshold.

struct AggArgs {
    const double *probs;
    double *util;
    const int32_t *pos, *len, *budget;
    int32_t *evict_idx, *evict_pos, *n_evict, *status, *pend;
    int cap, L, rule, refresh, kmax;
    float alpha;
};

// Utilities of slots not yet scored are +inf.  The tests below look at the
// bit pattern (integer operations): fp64 compares run on the fp64 pipe, which
// is narrow on this part, and these loops touch every slot several times.
__device__ __forceinline__ bool unscored_bits(uint64_t b)
{
    return (b & 0x7fffffffffffffffull) == 0x7ff0000000000000ull;
}

__device__ __forceinline__ uint64_t util_bits(const double *util, int i)
{
    return (uint64_t)__double_as_longlong(util[i]);
}

// k-th smallest (0-based rank) key among the slots where valid(i); returns
// the key and, through *below, how many valid keys are strictly smaller.
// blockDim.x is a multiple of 32 and at least 64.  Histogram updates are
// aggregated per warp over the lanes with the same digit (the digits of a
// pass are often concentrated in a few bins); warp 0 scans the 256 bins.
template <typename Key, typename KeyF, typename ValidF>
__device__ Key block_select(int n, int rank, KeyF key, ValidF valid,
                            int *hist, int *bcast, int *below, int *equal = nullptr)
{
    Key prefix = 0, mask = 0;
    const int rank0 = rank;
    const int lane = threadIdx.x & 31;
    for (int shift = (int)sizeof(Key) * 8 - 8; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
        __syncthreads();
        // four slots per thread per iteration: every key is read before any
        // is binned (the reads overlap)
        for (int b0 = 0; b0 < n; b0 += 4 * (int)blockDim.x) {
            int bin[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int i = b0 + j * (int)blockDim.x + (int)threadIdx.x;
                bin[j] = -1;
                if (i < n && valid(i)) {
                    const Key k = key(i);
                    if ((k & mask) == prefix) bin[j] = (int)((k >> shift) & 255);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const unsigned peers = __match_any_sync(kFull, bin[j]);
                if (bin[j] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[bin[j]], __popc(peers));
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l holds bins 8l .. 8l + 7
            int h[8], loc = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                h[j] = hist[8 * lane + j];
                loc += h[j];
            }
            int incl = loc;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int t = __shfl_up_sync(kFull, incl, m);
                if (lane >= m) incl += t;
            }
            const int excl = incl - loc;
            // the first lane whose bins take the cumulative count past rank
            const unsigned over = __ballot_sync(kFull, incl > rank);
            const int src = over ? __ffs(over) - 1 : 31;
            if (lane == src) {
                int cum = excl, b = 0;
                for (; b < 7; b++) {
                    if (cum + h[b] > rank) break;
                    cum += h[b];
                }
                bcast[0] = 8 * lane + b;
                bcast[1] = rank - cum;
                bcast[2] = h[b];                  // keys in the chosen bin
            }
        }
        __syncthreads();
        prefix |= ((Key)bcast[0]) << shift;
        mask |= ((Key)255) << shift;
        rank = bcast[1];
        if (shift == 0 && equal) *equal = bcast[2];   // keys equal to the result
        __syncthreads();
    }
    *below = rank0 - rank;
    return prefix;
}

// Victim selection of unit u (len n): the k = n - budget smallest (utility,
// position) pairs among its scored slots, in ascending slot order.  The
// whole block calls it.
__device__ void aggregate_select(const AggArgs &a, int u, int n, int *hist, int *bcast, int *scan)
{
    const int tid = threadIdx.x;
    double *util = a.util + (size_t)u * a.cap;
    const int32_t *pos = a.pos + (size_t)u * a.cap;
    const int Lb = a.budget ? a.budget[u] : a.L;      // this unit's budget
    if (Lb < 1 || Lb > a.L) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    const int k = n - Lb;
    if (k <= 0) {
        if (tid == 0) a.n_evict[u] = 0;
        return;
    }
    if (a.rule == KVC_RULE_MI && k > 1) {
        // MomentKV's loop re-scores after every fold: taking the k lowest
        // scores of one pass is not the method (kvc_mi_evict runs the loop)
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_UNSUPPORTED); }
        return;
    }
    if (k > a.kmax) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    int cnt = 0;
    for (int i0 = tid; i0 < n; i0 += 4 * blockDim.x) {
        bool sc[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = i0 + j * blockDim.x;
            sc[j] = i < n && !unscored_bits(util_bits(util, i));
        }
#pragma unroll
        for (int j = 0; j < 4; j++) cnt += sc[j];
    }
    int total;
    block_exscan(cnt, scan, &total);
    if (total < k) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_INVALID_ARG); }
        return;
    }
    auto scored = [&](int i) { return !unscored_bits(util_bits(util, i)); };
    auto ukey = [&](int i) { return double_key(util[i]); };
    int below, equal;
    const uint64_t kth = block_select<uint64_t>(n, k - 1, ukey, scored, hist, bcast, &below, &equal);
    const int need = k - below;       // slots to take from the tie group
    auto tie = [&](int i) {
        const uint64_t b = util_bits(util, i);
        return !unscored_bits(b) && double_key(__longlong_as_double((long long)b)) == kth;
    };
    auto pkey = [&](int i) { return (uint32_t)pos[i] ^ 0x80000000u; };
    // the positions settle the tie group only when part of it goes (with
    // distinct utilities the group is the one slot at the threshold)
    int below2;
    const uint32_t pth = equal == need
                             ? 0xffffffffu
                             : block_select<uint32_t>(n, need - 1, pkey, tie, hist, bcast, &below2);
    // write the victims in ascending slot order: warp w takes a contiguous
    // segment of the slots, counts its victims (one block scan of the
    // counts), then writes them from its offset
    auto selected = [&](int i) {
        const uint64_t b = util_bits(util, i);
        if (unscored_bits(b)) return false;
        const uint64_t kk = double_key(__longlong_as_double((long long)b));
        return kk < kth || (kk == kth && pkey(i) <= pth);
    };
    const int lane = tid & 31, nwarps = blockDim.x >> 5;
    const int seg = (((n + nwarps - 1) / nwarps) + 31) & ~31;
    const int sb = (tid >> 5) * seg, se = min(n, sb + seg);
    int wc = 0;
    for (int i0 = sb; i0 < se; i0 += 128) {
        bool sl[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = i0 + 32 * j + lane;
            sl[j] = i < se && selected(i);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) wc += __popc(__ballot_sync(kFull, sl[j]));
    }
    int written;
    int off = block_exscan(lane == 0 ? wc : 0, scan, &written);
    off = __shfl_sync(kFull, off, 0);
    for (int i0 = sb; i0 < se; i0 += 32) {
        const int i = i0 + lane;
        const bool sl = i < se && selected(i);
        const unsigned b = __ballot_sync(kFull, sl);
        const int r = off + __popc(b & ((1u << lane) - 1u));
        if (sl && r < a.kmax) {
            a.evict_idx[(size_t)u * a.kmax + r] = i;
            if (a.evict_pos) a.evict_pos[(size_t)u * a.kmax + r] = pos[i];
        }
        off += __popc(b);
    }
    if (tid == 0) {
        a.n_evict[u] = written == k ? k : 0;     // duplicate positions: refuse
        if (written != k) record_status(a.status, KVC_ERR_INVALID_ARG);
    }
}


__global__ void __launch_bounds__(512) aggregate_kernel(AggArgs a)
{
    __shared__ int hist[256];
    __shared__ int bcast[4];
    __shared__ int scan[40];
    const int u = blockIdx.x, tid = threadIdx.x;
    const int n = a.len[u];
    double *util = a.util + (size_t)u * a.cap;
    if (n < 0 || n > a.cap) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    if (a.refresh) {
        if (tid == 0) a.pend[(size_t)u * kPendStride] = 0;   // fused-step queue now stale
        const double *pr = a.probs + (size_t)u * a.cap;
        const double al = (double)a.alpha;
        for (int i0 = tid; i0 < n; i0 += 4 * blockDim.x) {
            double sv[4], mv[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int i = i0 + j * blockDim.x;
                sv[j] = i < n ? pr[i] : 0.0;
                mv[j] = i < n ? util[i] : 0.0;
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int i = i0 + j * blockDim.x;
                const double s = sv[j], m = mv[j];
                double r;
                if (unscored_bits((uint64_t)__double_as_longlong(m))) r = s;   // first observation
                else if (a.rule == KVC_RULE_SINGLE || a.rule == KVC_RULE_MI) r = s;   // MI: s is the score
                else if (a.rule == KVC_RULE_CUMULATIVE) r = m + s;
                else r = al * m + (1.0 - al) * s;
                if (i < n) util[i] = r;
            }
        }
        __syncthreads();
    }
    aggregate_select(a, u, n, hist, bcast, scan);
}

// InertiaKV's layer-chained EMA (rule KVC_RULE_EMA_CHAINED): one CTA per
// sequence (its NL x Hkv units hold the same positions in the same slots).
// On a refresh step every slot's utility passes the layers in order,
// m = s_l at the first observation, else alpha m + (1 - alpha) s_l, with s_l
// the layer's mean over its KV units' head-mean probabilities (all H heads),
// and is stored in every unit of the sequence; the victims are selected once
// (on the sequence's first unit) and written to every unit.
__global__ void __launch_bounds__(512) aggregate_chained_kernel(AggArgs a, int NL, int Hkv)
{
    __shared__ int hist[256];
    __shared__ int bcast[4];
    __shared__ int scan[40];
    __shared__ int okf;
    const int per = NL * Hkv, u0 = blockIdx.x * per, tid = threadIdx.x;
    const int n = a.len[u0];
    if (tid == 0) okf = 1;
    __syncthreads();
    for (int q = tid; q < per; q += blockDim.x)
        if (a.len[u0 + q] != n) okf = 0;
    __syncthreads();
    if (!okf || n < 0 || n > a.cap) {
        for (int q = tid; q < per; q += blockDim.x) a.n_evict[u0 + q] = 0;
        if (tid == 0) record_status(a.status, okf ? KVC_ERR_SHAPE : KVC_ERR_INVALID_ARG);
        return;
    }
    if (a.refresh) {
        for (int q = tid; q < per; q += blockDim.x) a.pend[(size_t)(u0 + q) * kPendStride] = 0;
        const double al = (double)a.alpha, rh = 1.0 / Hkv;
        for (int i = tid; i < n; i += blockDim.x) {
            double m = a.util[(size_t)u0 * a.cap + i];
            bool seen = !isinf(m);
            for (int l = 0; l < NL; l++) {
                double sl = 0.0;
                for (int g = 0; g < Hkv; g++) sl += a.probs[(size_t)(u0 + l * Hkv + g) * a.cap + i];
                sl *= rh;
                m = seen ? al * m + (1.0 - al) * sl : sl;
                seen = true;
            }
            for (int q = 0; q < per; q++) a.util[(size_t)(u0 + q) * a.cap + i] = m;
        }
        __syncthreads();
    }
    aggregate_select(a, u0, n, hist, bcast, scan);
    __syncthreads();
    // the sequence's other units take the same victims (global writes of this
    // block are visible to it after the barrier)
    const int k = a.n_evict[u0];
    for (int q = 1; q < per; q++) {
        if (tid == 0) a.n_evict[u0 + q] = k;
        for (int e = tid; e < k; e += blockDim.x) {
            a.evict_idx[(size_t)(u0 + q) * a.kmax + e] = a.evict_idx[(size_t)u0 * a.kmax + e];
            if (a.evict_pos)
                a.evict_pos[(size_t)(u0 + q) * a.kmax + e] = a.evict_pos[(size_t)u0 * a.kmax + e];
        }
    }
}

// Steps with many victims per unit: the same selection with the keys in
// shared memory.  One pass updates the utilities (refresh steps) and keeps
// the top 32 bits of every order key; the radix passes run on those; the
// group of slots whose top bits equal the threshold's is settled by the
// full key and the position.  One CTA of 1024 threads per unit, the keys
// of up to kAggKeysMax slots.
constexpr int kAggKeysMax = 49152;
constexpr int kAggGroupMax = 1024;
constexpr uint32_t kUnscored32 = 0xFFF00000u;     // top bits of +inf's order key

__global__ void __launch_bounds__(1024, 1) aggregate_keys_kernel(AggArgs a)
{
    extern __shared__ uint32_t k32[];              // [len]
    __shared__ int hist[256];
    __shared__ int bcast[4];
    __shared__ int scan[40];
    __shared__ int gidx[kAggGroupMax];
    __shared__ unsigned long long gkey[kAggGroupMax];
    __shared__ int gcount;
    __shared__ unsigned long long th_key;
    __shared__ int th_pos;
    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int n = a.len[u];
    double *util = a.util + (size_t)u * a.cap;
    const int32_t *pos = a.pos + (size_t)u * a.cap;
    if (n < 0 || n > a.cap || n > kAggKeysMax) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    const double al = (double)a.alpha;
    const double *pr = a.probs + (size_t)u * a.cap;
    if (a.refresh && tid == 0) a.pend[(size_t)u * kPendStride] = 0;   // fused-step queue now stale
    for (int i0 = tid; i0 < n; i0 += 4 * blockDim.x) {
        double sv[4], mv[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = i0 + j * blockDim.x;
            sv[j] = (a.refresh && i < n) ? pr[i] : 0.0;
            mv[j] = i < n ? util[i] : 0.0;
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = i0 + j * blockDim.x;
            if (i >= n) continue;
            double r = mv[j];
            if (a.refresh) {
                const double s = sv[j], m = mv[j];
                if (unscored_bits((uint64_t)__double_as_longlong(m))) r = s;   // first observation
                else if (a.rule == KVC_RULE_SINGLE || a.rule == KVC_RULE_MI) r = s;
                else if (a.rule == KVC_RULE_CUMULATIVE) r = m + s;
                else r = al * m + (1.0 - al) * s;
                util[i] = r;
            }
            k32[i] = (uint32_t)(double_key(r) >> 32);
        }
    }
    __syncthreads();
    const int Lb = a.budget ? a.budget[u] : a.L;
    if (Lb < 1 || Lb > a.L) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_SHAPE); }
        return;
    }
    const int k = n - Lb;
    if (k <= 0) {
        if (tid == 0) a.n_evict[u] = 0;
        return;
    }
    if ((a.rule == KVC_RULE_MI && k > 1) || k > a.kmax) {
        if (tid == 0) {
            a.n_evict[u] = 0;
            record_status(a.status, a.rule == KVC_RULE_MI && k > 1 ? KVC_ERR_UNSUPPORTED : KVC_ERR_SHAPE);
        }
        return;
    }
    int cnt = 0;
    for (int i = tid; i < n; i += blockDim.x) cnt += k32[i] < kUnscored32;
    int total;
    block_exscan(cnt, scan, &total);
    if (total < k) {
        if (tid == 0) { a.n_evict[u] = 0; record_status(a.status, KVC_ERR_INVALID_ARG); }
        return;
    }
    auto valid = [&](int i) { return k32[i] < kUnscored32; };
    auto key = [&](int i) { return k32[i]; };
    int below, equal;
    const uint32_t T32 = block_select<uint32_t>(n, k - 1, key, valid, hist, bcast, &below, &equal);
    const int need = k - below;            // from the group whose top bits equal T32
    const bool whole = need == equal;
    if (!whole) {
        if (equal > kAggGroupMax) {        // a large tie group: the selection on the full keys
            aggregate_select(a, u, n, hist, bcast, scan);
            return;
        }
        if (tid == 0) gcount = 0;
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x)
            if (k32[i] == T32) {
                const int j = atomicAdd(&gcount, 1);
                gidx[j] = i;
                gkey[j] = double_key(util[i]);
            }
        __syncthreads();
        const int m = gcount;
        for (int j = tid; j < m; j += blockDim.x) {
            const unsigned long long kj = gkey[j];
            const int pj = pos[gidx[j]];
            int rank = 0;
            for (int l = 0; l < m; l++) {
                const unsigned long long kl = gkey[l];
                rank += kl < kj || (kl == kj && pos[gidx[l]] < pj);
            }
            if (rank == need - 1) {
                th_key = kj;
                th_pos = pj;
            }
        }
        __syncthreads();
    }
    const unsigned long long tk = whole ? 0ull : th_key;
    const int tp = whole ? 0 : th_pos;
    auto selected = [&](int i) {
        const uint32_t k_ = k32[i];
        if (k_ < T32) return true;
        if (k_ != T32) return false;
        if (whole) return true;
        const unsigned long long kk = double_key(util[i]);
        return kk < tk || (kk == tk && pos[i] <= tp);
    };
    // victims in ascending slot order: contiguous warp segments, one scan
    const int nwarps = blockDim.x >> 5;
    const int seg = (((n + nwarps - 1) / nwarps) + 31) & ~31;
    const int sb = (tid >> 5) * seg, se = min(n, sb + seg);
    int wc = 0;
    for (int i0 = sb; i0 < se; i0 += 32) {
        const int i = i0 + lane;
        wc += __popc(__ballot_sync(kFull, i < se && selected(i)));
    }
    int written;
    int off = block_exscan(lane == 0 ? wc : 0, scan, &written);
    off = __shfl_sync(kFull, off, 0);
    for (int i0 = sb; i0 < se; i0 += 32) {
        const int i = i0 + lane;
        const bool sl = i < se && selected(i);
        const unsigned b = __ballot_sync(kFull, sl);
        const int r = off + __popc(b & ((1u << lane) - 1u));
        if (sl && r < a.kmax) {
            a.evict_idx[(size_t)u * a.kmax + r] = i;
            if (a.evict_pos) a.evict_pos[(size_t)u * a.kmax + r] = pos[i];
        }
        off += __popc(b);
    }
    if (tid == 0) {
        a.n_evict[u] = written == k ? k : 0;     // duplicate positions: refuse
        if (written != k) record_status(a.status, KVC_ERR_INVALID_ARG);
    }
}

cudaError_t launch_aggregate(const kvc_params &p, int t, const double *probs,
                             const kvc_cache &c, int kmax, int32_t *evict_idx,
                             int32_t *evict_pos, int32_t *n_evict,
                             const DecodeWs &ws, cudaStream_t st)
{
    AggArgs a{probs, c.util, c.pos, c.len, p.budget, evict_idx, evict_pos, n_evict,
              ws.status, ws.pend, p.cap, p.L, p.rule,
              p.rule == KVC_RULE_MI || is_refresh(t, p.refresh_period),
              kmax, p.alpha};
    if (p.rule == KVC_RULE_EMA_CHAINED) {
        const int per = p.chain_layers * p.chain_heads;
        aggregate_chained_kernel<<<p.U / per, 512, 0, st>>>(a, p.chain_layers, p.chain_heads);
    } else if (kmax > 16 && p.cap <= kAggKeysMax) {
        const size_t smem = (size_t)p.cap * 4;
        cudaError_t e = cudaFuncSetAttribute(aggregate_keys_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        aggregate_keys_kernel<<<p.U, 1024, smem, st>>>(a);
    } else {
        aggregate_kernel<<<p.U, 512, 0, st>>>(a);
    }
    return cudaGetLastError();
}

// Victim lists come from the caller: every kernel that reads one checks that
// the count fits kmax and every slot lies in [0, len) before touching memory.
__device__ bool victims_ok(const int32_t *ev, int k, int n, int cap, int *flag)
{
    if (threadIdx.x == 0) *flag = (n >= 0 && n <= cap) ? 1 : 0;
    __syncthreads();
    for (int e = threadIdx.x; e < k; e += blockDim.x) {
        const int s = ev[e];
        if (s < 0 || s >= n) *flag = 0;
    }
    __syncthreads();
    const bool ok = *flag != 0;
    __syncthreads();
    return ok;
}

// ================================================================ moment fold
//
// One CTA per unit, 256 threads; thread t owns the 8 x 8 block of the
// co-moment M = n C at rows 8*(t/16), columns 8*(t%16).  The victims are
// taken in tiles of 32: a tile's weighted mean and centred co-moment are
// merged into the running (n, mu_k, mu_v, M) by the pairwise update of Chan,
// Golub and LeVeque (1979); a one-token tile is West's (1979) weighted
// incremental update.

struct MomArgs {
    const uint16_t *K, *V;
    const int32_t *votes, *len;
    const int32_t *evict_idx, *n_evict;
    float *n, *mu_k, *mu_v, *C;
    int32_t *status;
    int cap, kmax;
};

constexpr int kFoldTile = 32;

__global__ void __launch_bounds__(256) moment_fold_kernel(MomArgs a)
{
    __shared__ __align__(16) float kt[kFoldTile][kD];
    __shared__ __align__(16) float vt[kFoldTile][kD];
    __shared__ float wt[kFoldTile];
    __shared__ float muk[kD], muv[kD], tk[kD], tv[kD];
    __shared__ float nb[2];
    __shared__ int okf;
    const int u = blockIdx.x, tid = threadIdx.x;
    const int k = a.n_evict[u];
    if (k <= 0) return;
    if (k > a.kmax || !victims_ok(a.evict_idx + (size_t)u * a.kmax, k, a.len[u], a.cap, &okf)) {
        if (tid == 0) record_status(a.status, KVC_ERR_INVALID_ARG);
        return;
    }
    const int r0 = 8 * (tid >> 4), c0 = 8 * (tid & 15);
    float *Cu = a.C + (size_t)u * kD * kD;
    float nacc = a.n[u];
    if (tid < kD) {
        muk[tid] = a.mu_k[(size_t)u * kD + tid];
        muv[tid] = a.mu_v[(size_t)u * kD + tid];
    }
    float M[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const float4 x0 = *reinterpret_cast<const float4 *>(Cu + (r0 + i) * kD + c0);
        const float4 x1 = *reinterpret_cast<const float4 *>(Cu + (r0 + i) * kD + c0 + 4);
        M[i][0] = x0.x * nacc; M[i][1] = x0.y * nacc; M[i][2] = x0.z * nacc; M[i][3] = x0.w * nacc;
        M[i][4] = x1.x * nacc; M[i][5] = x1.y * nacc; M[i][6] = x1.z * nacc; M[i][7] = x1.w * nacc;
    }
    const int32_t *ev = a.evict_idx + (size_t)u * a.kmax;
    const size_t ubase = (size_t)u * a.cap;
    for (int j0 = 0; j0 < k; j0 += kFoldTile) {
        const int nt = min(kFoldTile, k - j0);
        __syncthreads();
        {   // load the tile: thread -> (token, 16-dim chunk)
            const int tok = tid >> 3, ch = tid & 7;
            if (tok < nt) {
                const int slot = ev[j0 + tok];
                const uint16_t *kr = a.K + (ubase + slot) * kD + 16 * ch;
                const uint16_t *vr = a.V + (ubase + slot) * kD + 16 * ch;
                float f[16];
                unpack8(*reinterpret_cast<const uint4 *>(kr), f);
                unpack8(*reinterpret_cast<const uint4 *>(kr + 8), f + 8);
#pragma unroll
                for (int j = 0; j < 16; j++) kt[tok][16 * ch + j] = f[j];
                unpack8(*reinterpret_cast<const uint4 *>(vr), f);
                unpack8(*reinterpret_cast<const uint4 *>(vr + 8), f + 8);
#pragma unroll
                for (int j = 0; j < 16; j++) vt[tok][16 * ch + j] = f[j];
                if (ch == 0) wt[tok] = a.votes ? (float)a.votes[ubase + slot] : 1.f;
            } else if (tok < kFoldTile && ch == 0) {
                wt[tok] = 0.f;
            }
        }
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int j = 0; j < nt; j++) s += wt[j];
            nb[0] = s;
        }
        __syncthreads();
        const float nt_w = nb[0];
        // tile means
        if (tid < kD) {
            float s = 0.f;
            for (int j = 0; j < nt; j++) s = fmaf(wt[j], kt[j][tid], s);
            tk[tid] = s / nt_w;
        } else {
            const int dd = tid - kD;
            float s = 0.f;
            for (int j = 0; j < nt; j++) s = fmaf(wt[j], vt[j][dd], s);
            tv[dd] = s / nt_w;
        }
        __syncthreads();
        // centre the tile (values also carry the weight)
        for (int e = tid; e < nt * kD; e += blockDim.x) {
            const int j = e / kD, dd = e % kD;
            kt[j][dd] -= tk[dd];
            vt[j][dd] = wt[j] * (vt[j][dd] - tv[dd]);
        }
        __syncthreads();
        const float nn = nacc + nt_w;
        const float cross = nacc * nt_w / nn;
        float dv[8], dk[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            dv[i] = tv[r0 + i] - muv[r0 + i];
            dk[i] = tk[c0 + i] - muk[c0 + i];
        }
        for (int j = 0; j < nt; j++) {
            const float4 va = *reinterpret_cast<const float4 *>(&vt[j][r0]);
            const float4 vb = *reinterpret_cast<const float4 *>(&vt[j][r0 + 4]);
            const float4 ka = *reinterpret_cast<const float4 *>(&kt[j][c0]);
            const float4 kb = *reinterpret_cast<const float4 *>(&kt[j][c0 + 4]);
            const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            const float kk[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int jj = 0; jj < 8; jj++) M[i][jj] = fmaf(vv[i], kk[jj], M[i][jj]);
        }
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int jj = 0; jj < 8; jj++) M[i][jj] = fmaf(cross * dv[i], dk[jj], M[i][jj]);
        __syncthreads();
        if (tid < kD) muk[tid] += (tk[tid] - muk[tid]) * (nt_w / nn);
        else muv[tid - kD] += (tv[tid - kD] - muv[tid - kD]) * (nt_w / nn);
        nacc = nn;
    }
    __syncthreads();
    const float rn = 1.f / nacc;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float4 x0 = make_float4(M[i][0] * rn, M[i][1] * rn, M[i][2] * rn, M[i][3] * rn);
        float4 x1 = make_float4(M[i][4] * rn, M[i][5] * rn, M[i][6] * rn, M[i][7] * rn);
        *reinterpret_cast<float4 *>(Cu + (r0 + i) * kD + c0) = x0;
        *reinterpret_cast<float4 *>(Cu + (r0 + i) * kD + c0 + 4) = x1;
    }
    if (tid < kD) {
        a.mu_k[(size_t)u * kD + tid] = muk[tid];
        a.mu_v[(size_t)u * kD + tid] = muv[tid];
    }
    if (tid == 0) a.n[u] = nacc;
}

cudaError_t launch_moment(const kvc_params &p, const kvc_cache &c, int kmax,
                          const int32_t *evict_idx, const int32_t *n_evict,
                          const kvc_moments &m, const DecodeWs &ws,
                          cudaStream_t st)
{
    // many victims per unit (the first step over the prompt, a hand-off):
    // the tensor-core fold, one 128-victim tile at a time
    if (kmax >= kFoldTcMin)
        return launch_fold_tc(c, p.cap, p.U, kmax, evict_idx, n_evict, m, ws.status, st);
    MomArgs a{c.K, c.V, c.votes, c.len, evict_idx, n_evict, m.n, m.mu_k, m.mu_v, m.C,
              ws.status, p.cap, kmax};
    moment_fold_kernel<<<p.U, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// ==================================================================== correct
//
// One CTA per unit, 8 warps.  f_R / log Z_R by the eviction-error identity
// (KeepKV eq 3) when at most 16 slots went and their mass is <= 1/2 in every
// head; otherwise by a direct online-softmax pass over the live slots that
// are not evicted.  Then the inference phase of MomentKV Algorithm 1.

struct CorrArgs {
    const uint16_t *q, *K, *V;
    const int32_t *votes, *len;
    const int32_t *evict_idx, *n_evict;
    const float *lse, *f_all;
    const float *mn, *mu_k, *mu_v, *C;
    float *o, *f_R, *logZ_R;
    int32_t *status;
    int cap, kmax, correction;
    int retained;      // lse / f_all are already log Z_R / f_R (no victims to remove)
    // retained form: units left with n_evict = 0 (nothing went, or a merge
    // that keeps the full-cache output) take these (the pass over all slots)
    const float *lse_all, *f_all_all;
    const int32_t *n_evict_sel;
};

constexpr int kIdentityMax = 16;

template <int G>
__global__ void __launch_bounds__(256) correct_kernel(CorrArgs a)
{
    extern __shared__ uint32_t evbits[];   // ceil(cap/32) words
    __shared__ __align__(16) float qs[G][kD];
    __shared__ float fR[G][kD];
    __shared__ float lz[G];
    __shared__ float Ae[kIdentityMax][G];
    __shared__ float mass[G];
    __shared__ int direct_s;
    __shared__ int okf;
    __shared__ float wst[8][4][G][2];      // per warp/group (m, l)

    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int k = a.retained ? 0 : max(0, a.n_evict[u]);
    const int n = a.len[u];
    if (k > a.kmax || !victims_ok(a.evict_idx + (size_t)u * a.kmax, k, n, a.cap, &okf)) {
        if (tid == 0) record_status(a.status, KVC_ERR_INVALID_ARG);
        return;
    }
    const size_t ubase = (size_t)u * a.cap;
    const float rs = rsqrtf((float)kD);
    for (int e = tid; e < G * kD; e += blockDim.x)
        qs[e / kD][e % kD] = bf2f(a.q[(size_t)u * G * kD + e]);
    if (tid == 0) direct_s = 0;
    __syncthreads();

    const int32_t *ev = a.evict_idx + (size_t)u * a.kmax;
    if (k <= 0) {
        const bool whole = a.retained && a.n_evict_sel && a.n_evict_sel[u] == 0;
        const float *fa = whole ? a.f_all_all : a.f_all;
        const float *la = whole ? a.lse_all : a.lse;
        for (int e = tid; e < G * kD; e += blockDim.x)
            fR[e / kD][e % kD] = fa[(size_t)u * G * kD + e];
        if (tid < G) lz[tid] = la[(size_t)u * G + tid];
    } else if (k <= kIdentityMax) {
        // A_e^h = exp(q_h . k_e / sqrt(d) + ln p_e - lse_h)
        for (int e = w; e < k; e += 8) {
            const int slot = ev[e];
            const uint16_t *kr = a.K + (ubase + slot) * kD;
            float kv[4];
            for (int j = 0; j < 4; j++) kv[j] = bf2f(kr[lane * 4 + j]);
            const float lnp = a.votes ? logf((float)a.votes[ubase + slot]) : 0.f;
#pragma unroll
            for (int h = 0; h < G; h++) {
                float s = 0.f;
                for (int j = 0; j < 4; j++) s = fmaf(qs[h][lane * 4 + j] * rs, kv[j], s);
                s = warp_sum(s);
                if (lane == 0) Ae[e][h] = expf(s + lnp - a.lse[(size_t)u * G + h]);
            }
        }
        __syncthreads();
        if (tid < G) {
            float m = 0.f;
            for (int e = 0; e < k; e++) m += Ae[e][tid];
            mass[tid] = m;
            if (m > 0.5f) atomicExch(&direct_s, 1);
        }
        __syncthreads();
        if (!direct_s) {
            for (int e = tid; e < G * kD; e += blockDim.x) {
                const int h = e / kD, dd = e % kD;
                float num = a.f_all[(size_t)u * G * kD + e];
                for (int j = 0; j < k; j++)
                    num = fmaf(-Ae[j][h], bf2f(a.V[(ubase + ev[j]) * kD + dd]), num);
                fR[h][dd] = num / (1.f - mass[h]);
            }
            if (tid < G) lz[tid] = a.lse[(size_t)u * G + tid] + log1pf(-mass[tid]);
        }
    } else {
        if (tid == 0) direct_s = 1;
    }
    __syncthreads();

    if (direct_s) {
        const int words = (a.cap + 31) >> 5;
        for (int i = tid; i < words; i += blockDim.x) evbits[i] = 0;
        for (int e = tid; e < G * kD; e += blockDim.x) fR[e / kD][e % kD] = 0.f;
        __syncthreads();
        for (int e = tid; e < k; e += blockDim.x) {
            const int slot = ev[e];
            atomicOr(&evbits[slot >> 5], 1u << (slot & 31));
        }
        __syncthreads();
        const int grp = lane >> 3, c = lane & 7;
        float qf[G][16];
#pragma unroll
        for (int h = 0; h < G; h++)
#pragma unroll
            for (int j = 0; j < 8; j++) {
                qf[h][j] = qs[h][8 * c + j] * rs;
                qf[h][8 + j] = qs[h][64 + 8 * c + j] * rs;
            }
        float m[G], l[G], acc[G][16];
#pragma unroll
        for (int h = 0; h < G; h++) {
            m[h] = -INFINITY; l[h] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j++) acc[h][j] = 0.f;
        }
        // warp w walks the bitmap words w, w + 8, ...; the slots of a word
        // that were not evicted go four at a time (slot group grp takes the
        // grp-th lowest of the next four), so evicted slots cost nothing
        const int nwords = (n + 31) >> 5;
        int wi = w;
        uint32_t pend = 0;
        if (wi < nwords) {
            pend = ~evbits[wi];
            if (wi == nwords - 1 && (n & 31)) pend &= (1u << (n & 31)) - 1u;
        }
        for (;;) {
            while (pend == 0 && wi < nwords) {
                wi += 8;
                if (wi < nwords) {
                    pend = ~evbits[wi];
                    if (wi == nwords - 1 && (n & 31)) pend &= (1u << (n & 31)) - 1u;
                }
            }
            if (wi >= nwords) break;
            int i = -1;
#pragma unroll
            for (int g = 0; g < 4; g++) {
                if (pend) {
                    if (g == grp) i = 32 * wi + __ffs(pend) - 1;
                    pend &= pend - 1u;
                }
            }
            const bool live = i >= 0;
            float kf[16], vf[16];
            if (live) {
                const uint16_t *kr = a.K + (ubase + i) * kD;
                const uint16_t *vr = a.V + (ubase + i) * kD;
                unpack8(ldg_nc_v4(kr + 8 * c), kf);
                unpack8(ldg_nc_v4(kr + 64 + 8 * c), kf + 8);
                unpack8(ldg_nc_v4(vr + 8 * c), vf);
                unpack8(ldg_nc_v4(vr + 64 + 8 * c), vf + 8);
            } else {
#pragma unroll
                for (int j = 0; j < 16; j++) { kf[j] = 0.f; vf[j] = 0.f; }
            }
            float part[G];
#pragma unroll
            for (int h = 0; h < G; h++) {
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < 16; j++) s = fmaf(qf[h][j], kf[j], s);
                part[h] = s;
            }
#pragma unroll
            for (int mm = 1; mm < 8; mm <<= 1)
#pragma unroll
                for (int h = 0; h < G; h++) part[h] += __shfl_xor_sync(kFull, part[h], mm);
            if (live) {
                const float lnp = a.votes ? logf((float)a.votes[ubase + i]) : 0.f;
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const float x = part[h] + lnp;
                    if (x > m[h]) {
                        const float corr = expf(m[h] - x);
                        l[h] *= corr;
#pragma unroll
                        for (int j = 0; j < 16; j++) acc[h][j] *= corr;
                        m[h] = x;
                    }
                    const float pp = expf(x - m[h]);
                    l[h] += pp;
#pragma unroll
                    for (int j = 0; j < 16; j++) acc[h][j] = fmaf(pp, vf[j], acc[h][j]);
                }
            }
        }
        // merge the 4 slot groups of each warp, then the 8 warps
        if (c == 0)
#pragma unroll
            for (int h = 0; h < G; h++) { wst[w][grp][h][0] = m[h]; wst[w][grp][h][1] = l[h]; }
        __syncthreads();
        if (tid < G) {
            const int h = tid;
            float mm = -INFINITY;
            for (int j = 0; j < 32; j++) mm = fmaxf(mm, wst[j >> 2][j & 3][h][0]);
            float ll = 0.f;
            for (int j = 0; j < 32; j++) {
                const float mj = wst[j >> 2][j & 3][h][0];
                if (mj != -INFINITY) ll += wst[j >> 2][j & 3][h][1] * expf(mj - mm);
            }
            mass[h] = mm;                       // reuse: global max
            lz[h] = ll > 0.f ? mm + logf(ll) : -INFINITY;
            Ae[0][h] = ll;                      // reuse: global sum
        }
        __syncthreads();
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; h++) sc[h] = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mass[h]);
        for (int h = 0; h < G; h++)
            for (int j = 0; j < 16; j++) {
                float v = acc[h][j] * sc[h];
                v += __shfl_xor_sync(kFull, v, 8);
                v += __shfl_xor_sync(kFull, v, 16);
                acc[h][j] = v;
            }
        if (grp == 0)
            for (int h = 0; h < G; h++)
                for (int j = 0; j < 8; j++) {
                    atomicAdd(&fR[h][8 * c + j], acc[h][j]);
                    atomicAdd(&fR[h][64 + 8 * c + j], acc[h][8 + j]);
                }
        __syncthreads();
        for (int e = tid; e < G * kD; e += blockDim.x) {
            const int h = e / kD, dd = e % kD;
            const float ll = Ae[0][h];
            fR[h][dd] = ll > 0.f ? fR[h][dd] / ll : 0.f;
        }
        __syncthreads();
    }

    // ---- MomentKV Algorithm 1, normalization-corrected inference phase
    const float ne = a.mn[u];
    float *ou = a.o + (size_t)u * G * kD;
    if (a.f_R)
        for (int e = tid; e < G * kD; e += blockDim.x) a.f_R[(size_t)u * G * kD + e] = fR[e / kD][e % kD];
    if (a.logZ_R && tid < G) a.logZ_R[(size_t)u * G + tid] = lz[tid];
    if (ne <= 0.f || a.correction == KVC_CORR_OFF) {
        for (int e = tid; e < G * kD; e += blockDim.x) ou[e] = fR[e / kD][e % kD];
        return;
    }
    __shared__ float wR[G];
    __shared__ float cq[G][kD];
    const float *mk = a.mu_k + (size_t)u * kD, *mv = a.mu_v + (size_t)u * kD;
    if (w < G) {
        float s = 0.f;
        for (int j = lane; j < kD; j += 32) s = fmaf(qs[w][j], mk[j], s);
        s = warp_sum(s);
        if (lane == 0) {
            const float logZE = logf(ne) + s * rs;
            wR[w] = 1.f / (1.f + expf(logZE - lz[w]));
        }
    }
    if (a.correction == KVC_CORR_FIRST_ORDER) {
        const float *Cu = a.C + (size_t)u * kD * kD;
        const int row = tid >> 1, half = tid & 1;
        float acc[G];
#pragma unroll
        for (int h = 0; h < G; h++) acc[h] = 0.f;
        const float *cr = Cu + (size_t)row * kD + half * 64;
        for (int j = 0; j < 64; j += 4) {
            const float4 cv = *reinterpret_cast<const float4 *>(cr + j);
#pragma unroll
            for (int h = 0; h < G; h++) {
                const float *qq = &qs[h][half * 64 + j];
                acc[h] = fmaf(cv.x, qq[0], acc[h]);
                acc[h] = fmaf(cv.y, qq[1], acc[h]);
                acc[h] = fmaf(cv.z, qq[2], acc[h]);
                acc[h] = fmaf(cv.w, qq[3], acc[h]);
            }
        }
#pragma unroll
        for (int h = 0; h < G; h++) {
            acc[h] += __shfl_xor_sync(kFull, acc[h], 1);
            if (half == 0) cq[h][row] = acc[h] * rs;
        }
    } else {
        for (int e = tid; e < G * kD; e += blockDim.x) cq[e / kD][e % kD] = 0.f;
    }
    __syncthreads();
    for (int e = tid; e < G * kD; e += blockDim.x) {
        const int h = e / kD, dd = e % kD;
        const float fe = mv[dd] + cq[h][dd];
        ou[e] = wR[h] * fR[h][dd] + (1.f - wR[h]) * fe;
    }
}

template <int G>
static cudaError_t launch_correct_g(const CorrArgs &a, int U, int cap, cudaStream_t st)
{
    const size_t smem = (size_t)((cap + 31) / 32) * 4;
    if (smem > 16384) {
        cudaError_t e = cudaFuncSetAttribute(correct_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    correct_kernel<G><<<U, 256, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_correct(const kvc_params &p, const uint16_t *q,
                           const kvc_cache &c, int kmax,
                           const int32_t *evict_idx, const int32_t *n_evict,
                           const float *lse, const float *f_all,
                           const kvc_moments &m, float *o, float *f_R,
                           float *logZ_R, const DecodeWs &ws, cudaStream_t st)
{
    CorrArgs a{q, c.K, c.V, c.votes, c.len, evict_idx, n_evict, lse, f_all,
               m.n, m.mu_k, m.mu_v, m.C, o, f_R, logZ_R, ws.status, p.cap, kmax, p.correction, 0,
               nullptr, nullptr, nullptr};
    switch (p.G) {
    case 1: return launch_correct_g<1>(a, p.U, p.cap, st);
    case 2: return launch_correct_g<2>(a, p.U, p.cap, st);
    case 4: return launch_correct_g<4>(a, p.U, p.cap, st);
    case 8: return launch_correct_g<8>(a, p.U, p.cap, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_correct_retained(const kvc_params &p, const uint16_t *q, const kvc_cache &c,
                                    const float *lse_R, const float *f_R, const kvc_moments &m,
                                    float *o, const DecodeWs &ws, cudaStream_t st,
                                    const float *lse_all, const float *f_all, const int32_t *n_evict)
{
    CorrArgs a{q, c.K, c.V, c.votes, c.len, nullptr, nullptr, lse_R, f_R,
               m.n, m.mu_k, m.mu_v, m.C, o, nullptr, nullptr, ws.status, p.cap, 1, p.correction, 1,
               lse_all, f_all, n_evict};
    switch (p.G) {
    case 1: return launch_correct_g<1>(a, p.U, p.cap, st);
    case 2: return launch_correct_g<2>(a, p.U, p.cap, st);
    case 4: return launch_correct_g<4>(a, p.U, p.cap, st);
    case 8: return launch_correct_g<8>(a, p.U, p.cap, st);
    default: return cudaErrorInvalidValue;
    }
}

// ==================================================================== compact
//
// One CTA per unit.  With n2 = len - k, the r-th evicted slot below n2 (in
// ascending order) receives the r-th live slot at or above n2.  Ranks come
// from per-word prefix counts of an eviction bitmap; pairs are formed in
// windows of kCompactWin ranks.

struct CompactArgs {
    uint16_t *K, *V;
    int32_t *votes, *pos;
    double *util;
    int32_t *len;
    const int32_t *evict_idx, *n_evict;
    int32_t *status;
    int cap, kmax;
};

constexpr int kCompactWin = 2048;

__global__ void __launch_bounds__(512) compact_kernel(CompactArgs a)
{
    extern __shared__ uint32_t sm[];
    __shared__ int src[kCompactWin], dst[kCompactWin];
    __shared__ int scan[40];
    __shared__ int okf;
    const int u = blockIdx.x, tid = threadIdx.x;
    const int k = a.n_evict[u];
    if (k <= 0) return;
    const int n = a.len[u];
    if (k > a.kmax || k > n || !victims_ok(a.evict_idx + (size_t)u * a.kmax, k, n, a.cap, &okf)) {
        if (tid == 0) record_status(a.status, KVC_ERR_INVALID_ARG);
        return;
    }
    const int n2 = n - k;
    const int words = (n + 31) >> 5;
    uint32_t *bits = sm;
    int *wpre = reinterpret_cast<int *>(sm + ((a.cap + 31) >> 5));
    for (int i = tid; i < words; i += blockDim.x) bits[i] = 0;
    __syncthreads();
    const int32_t *ev = a.evict_idx + (size_t)u * a.kmax;
    for (int e = tid; e < k; e += blockDim.x) {
        const int s = ev[e];
        atomicOr(&bits[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    // exclusive prefix of popcounts over words
    int carry = 0;
    for (int b0 = 0; b0 < words; b0 += blockDim.x) {
        const int i = b0 + tid;
        const int v = i < words ? __popc(bits[i]) : 0;
        int tot;
        const int ex = block_exscan(v, scan, &tot);
        if (i < words) wpre[i] = carry + ex;
        carry += tot;
    }
    __syncthreads();
    auto ev_below = [&](int i) {   // evicted slots in [0, i)
        return wpre[i >> 5] + __popc(bits[i >> 5] & ((1u << (i & 31)) - 1u));
    };
    const int holes = (n2 > 0) ? ev_below(n2) : 0;
    const int ev_n2 = holes;
    const size_t ubase = (size_t)u * a.cap;
    for (int r0 = 0; r0 < holes; r0 += kCompactWin) {
        const int r1 = min(holes, r0 + kCompactWin);
        for (int i = tid; i < n2; i += blockDim.x) {
            if ((bits[i >> 5] >> (i & 31)) & 1u) {
                const int r = ev_below(i);
                if (r >= r0 && r < r1) dst[r - r0] = i;
            }
        }
        for (int i = n2 + tid; i < n; i += blockDim.x) {
            if (!((bits[i >> 5] >> (i & 31)) & 1u)) {
                const int r = (i - n2) - (ev_below(i) - ev_n2);
                if (r >= r0 && r < r1) src[r - r0] = i;
            }
        }
        __syncthreads();
        const int np = r1 - r0;
        // four 16-byte chunks per thread in flight (the source rows are at
        // or above n2, the destinations below: no chunk is both read and
        // written; eight cost a resident CTA per SM and were slower)
        constexpr int kU = 4;
        for (int e0 = tid; e0 < np * 32; e0 += kU * blockDim.x) {
            uint4 x[kU];
#pragma unroll
            for (int j = 0; j < kU; j++) {
                const int e = e0 + j * blockDim.x;
                if (e < np * 32) {
                    const int pr = e >> 5, ch = e & 31;
                    const size_t from = ubase + src[pr];
                    x[j] = ch < 16 ? reinterpret_cast<const uint4 *>(a.K + from * kD)[ch]
                                   : reinterpret_cast<const uint4 *>(a.V + from * kD)[ch - 16];
                }
            }
#pragma unroll
            for (int j = 0; j < kU; j++) {
                const int e = e0 + j * blockDim.x;
                if (e < np * 32) {
                    const int pr = e >> 5, ch = e & 31;
                    const size_t from = ubase + src[pr], to = ubase + dst[pr];
                    if (ch < 16)
                        reinterpret_cast<uint4 *>(a.K + to * kD)[ch] = x[j];
                    else
                        reinterpret_cast<uint4 *>(a.V + to * kD)[ch - 16] = x[j];
                    if (ch == 0) {
                        a.pos[to] = a.pos[from];
                        a.util[to] = a.util[from];
                        if (a.votes) a.votes[to] = a.votes[from];
                    }
                }
            }
        }
        __syncthreads();
    }
    if (tid == 0) a.len[u] = n2;
}

cudaError_t launch_compact(const kvc_params &p, const kvc_cache &c, int kmax,
                           const int32_t *evict_idx, const int32_t *n_evict,
                           const DecodeWs &ws, cudaStream_t st)
{
    const size_t smem = (size_t)((p.cap + 31) / 32) * 8;
    if (smem > 16384) {
        cudaError_t e = cudaFuncSetAttribute(compact_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    CompactArgs a{c.K, c.V, c.votes, c.pos, c.util, c.len, evict_idx, n_evict,
                  ws.status, p.cap, kmax};
    compact_kernel<<<p.U, 512, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
