// kvc_merge.cu -- KeepKV ZIP-merging of a step's single victim into its most
// similar retained slot (KeepKV reading notes, "ZIP-Merging" eqs 7-12, the
// cosine candidate choice of "why cosine similarity" with the most recent R
// tokens excluded, and the epsilon guard of "numerical stability" item 2).
//
// One CTA per unit.  Pass: every live key row is streamed once (16 lanes x
// 16 bytes per 256-byte row, four rows in flight per half-warp) and scored
// by k_e . k_i / |k_i| (the cosine up to the positive factor 1/|k_e|); the
// argmax over the key (score, older position first) is the partner.  Merge:
// the logits of the group's mean query for the victim and the partner give
// the weights w = p exp(xbar); the partner slot takes k_r, v_r (bf16, round
// to nearest), p_e + p_c and the sum of the two utilities; the victim's slot
// is refilled from the last live slot and the unit's length drops by one.
// The unit's n_evict becomes 0, so the moment fold, the correction and the
// compaction that follow leave it alone (its output is the full-cache one).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace kvc {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeUnroll = 4;          // rows in flight per half-warp
constexpr int kHalfWarps = kMergeThreads / 16;

struct ZipArgs {
    const uint16_t *q;        // [U][G][d]
    uint16_t *K, *V;          // [U][cap][d]
    int32_t *votes, *pos, *len;
    double *util;
    const int32_t *evict_idx; // [U][kmax]
    int32_t *n_evict;         // [U]
    int32_t *partner_pos;     // [U] or NULL
    int32_t *status;
    int cap, kmax, G, new_pos, R;
    float eps;
};

__global__ void __launch_bounds__(kMergeThreads) zip_merge_kernel(ZipArgs a)
{
    __shared__ unsigned long long bk_s[kMergeThreads / 32];
    __shared__ int bs_s[kMergeThreads / 32];
    __shared__ float red[4][2];
    __shared__ float coef[4];     // lambda_e, lambda_c, ell / xt (0 under the guard), guard
    __shared__ int c_s;

    const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (a.n_evict[u] != 1) {
        if (tid == 0 && a.partner_pos) a.partner_pos[u] = -1;
        return;
    }
    const int n = a.len[u];
    const int e = a.evict_idx[(size_t)u * a.kmax];
    const size_t ubase = (size_t)u * a.cap;
    if (n < 1 || n > a.cap || e < 0 || e >= n) {
        if (tid == 0) {
            record_status(a.status, KVC_ERR_INVALID_ARG);
            if (a.partner_pos) a.partner_pos[u] = -1;
        }
        return;
    }

    // ------------------------------------------------ partner search
    const int hl = lane & 15;                        // 16-byte segment of a row
    const int hw = w * 2 + (lane >> 4);              // half-warp index
    float ke[8];
    unpack8(ldg_nc_v4(a.K + (ubase + e) * kD + 8 * hl), ke);
    const long long lim = (long long)a.new_pos - a.R; // candidates: pos <= new_pos - R
    unsigned long long bkey = 0ull;                  // 0 = no candidate yet
    int bslot = -1;
    for (int i0 = 0; i0 < n; i0 += kHalfWarps * kMergeUnroll) {
        uint4 r[kMergeUnroll];
        int pj[kMergeUnroll];
#pragma unroll
        for (int j = 0; j < kMergeUnroll; j++) {
            const int sl = i0 + hw + kHalfWarps * j;
            r[j] = sl < n ? ldg_nc_v4(a.K + (ubase + sl) * kD + 8 * hl) : make_uint4(0, 0, 0, 0);
            pj[j] = sl < n ? a.pos[ubase + sl] : 0;
        }
#pragma unroll
        for (int j = 0; j < kMergeUnroll; j++) {
            const int sl = i0 + hw + kHalfWarps * j;
            float f[8];
            unpack8(r[j], f);
            float dot = 0.f, ss = 0.f;
#pragma unroll
            for (int t = 0; t < 8; t++) {
                dot = fmaf(ke[t], f[t], dot);
                ss = fmaf(f[t], f[t], ss);
            }
#pragma unroll
            for (int m = 8; m > 0; m >>= 1) {
                dot += __shfl_xor_sync(kFull, dot, m);
                ss += __shfl_xor_sync(kFull, ss, m);
            }
            if (sl < n && sl != e && (long long)pj[j] <= lim) {
                const float sc = ss > 0.f ? dot * rsqrtf(ss) : 0.f;
                const unsigned long long key =
                    ((unsigned long long)float_key(sc) << 32) | (uint32_t)(0x7fffffff - pj[j]);
                if (key > bkey) {
                    bkey = key;
                    bslot = sl;
                }
            }
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(kFull, bkey, m);
        const int os = __shfl_xor_sync(kFull, bslot, m);
        if (ok > bkey) {
            bkey = ok;
            bslot = os;
        }
    }
    if (lane == 0) {
        bk_s[w] = bkey;
        bs_s[w] = bslot;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long b = 0ull;
        int s = -1;
        for (int j = 0; j < kMergeThreads / 32; j++)
            if (bk_s[j] > b) {
                b = bk_s[j];
                s = bs_s[j];
            }
        c_s = s;
    }
    __syncthreads();
    const int c = c_s;
    if (c < 0) {                                     // no candidate: plain eviction follows
        if (tid == 0 && a.partner_pos) a.partner_pos[u] = -1;
        return;
    }

    // ------------------------------------------------ merged pair (eqs 7-12)
    const int G = a.G;
    float kef = 0.f, kcf = 0.f, vef = 0.f, vcf = 0.f;
    if (tid < kD) {
        kef = bf2f(a.K[(ubase + e) * kD + tid]);
        kcf = bf2f(a.K[(ubase + c) * kD + tid]);
        vef = bf2f(a.V[(ubase + e) * kD + tid]);
        vcf = bf2f(a.V[(ubase + c) * kD + tid]);
        float qb = 0.f;                               // sum of the group's queries
        for (int h = 0; h < G; h++) qb += bf2f(a.q[((size_t)u * G + h) * kD + tid]);
        float se = warp_sum(qb * kef), sc = warp_sum(qb * kcf);
        if (lane == 0) {
            red[w][0] = se;
            red[w][1] = sc;
        }
    }
    __syncthreads();
    if (tid == 0) {
        const float scale = rsqrtf((float)kD) / (float)G;
        const float xe = (red[0][0] + red[1][0] + red[2][0] + red[3][0]) * scale;
        const float xc = (red[0][1] + red[1][1] + red[2][1] + red[3][1]) * scale;
        const float pe = a.votes ? (float)a.votes[ubase + e] : 1.f;
        const float pc = a.votes ? (float)a.votes[ubase + c] : 1.f;
        const float m = fmaxf(xe, xc);
        const float we = pe * expf(xe - m), wc = pc * expf(xc - m), W = we + wc;
        const float le = we / W, lc = wc / W;
        const float xt = le * xe + lc * xc;
        const float ell = m + logf(W / (pe + pc));
        const bool guard = fabsf(xt) < a.eps;
        coef[0] = le;
        coef[1] = lc;
        coef[2] = guard ? 0.f : ell / xt;
        coef[3] = guard ? 1.f : 0.f;
    }
    __syncthreads();
    if (tid < kD) {
        const float le = coef[0], lc = coef[1];
        const float kr = coef[3] != 0.f ? 0.5f * (kef + kcf) : (le * kef + lc * kcf) * coef[2];
        const float vr = le * vef + lc * vcf;
        a.K[(ubase + c) * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(kr));
        a.V[(ubase + c) * kD + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(vr));
    }
    if (tid == kD) {
        if (a.votes) a.votes[ubase + c] += a.votes[ubase + e];
        a.util[ubase + c] += a.util[ubase + e];      // +inf (unscored) stays +inf
        if (a.partner_pos) a.partner_pos[u] = a.pos[ubase + c];
    }
    __syncthreads();

    // ------------------------------------------------ remove the victim
    const int last = n - 1;
    if (e != last) {
        if (tid < 16) {
            reinterpret_cast<uint4 *>(a.K + (ubase + e) * kD)[tid] =
                reinterpret_cast<const uint4 *>(a.K + (ubase + last) * kD)[tid];
        } else if (tid < 32) {
            reinterpret_cast<uint4 *>(a.V + (ubase + e) * kD)[tid - 16] =
                reinterpret_cast<const uint4 *>(a.V + (ubase + last) * kD)[tid - 16];
        } else if (tid == 32) {
            if (a.votes) a.votes[ubase + e] = a.votes[ubase + last];
            a.pos[ubase + e] = a.pos[ubase + last];
            a.util[ubase + e] = a.util[ubase + last];
        }
    }
    if (tid == 0) {
        a.len[u] = last;
        a.n_evict[u] = 0;
    }
}

}  // namespace

cudaError_t launch_zip_merge(const kvc_params &p, int new_pos, const uint16_t *q,
                             const kvc_cache &c, int kmax, const int32_t *evict_idx,
                             int32_t *n_evict, int32_t *partner_pos, const DecodeWs &ws,
                             cudaStream_t st)
{
    ZipArgs a;
    a.q = q;
    a.K = c.K;
    a.V = c.V;
    a.votes = c.votes;
    a.pos = c.pos;
    a.len = c.len;
    a.util = c.util;
    a.evict_idx = evict_idx;
    a.n_evict = n_evict;
    a.partner_pos = partner_pos;
    a.status = ws.status;
    a.cap = p.cap;
    a.kmax = kmax;
    a.G = p.G;
    a.new_pos = new_pos;
    a.R = p.merge_recent;
    a.eps = (float)KVC_ZIP_EPS;
    zip_merge_kernel<<<p.U, kMergeThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
