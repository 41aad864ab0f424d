// kvc_common.cuh -- device helpers shared by the libkvc kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kD = 128;                 // supported head dimension
constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- workspace
// The first 256 bytes of every workspace hold the device status word.
struct WsHeader {
    int32_t status;        // first error recorded by a kernel (KVC_OK = 0)
    int32_t pad[63];
};

__device__ __forceinline__ void record_status(int32_t *status, int32_t code)
{
    atomicCAS(status, KVC_OK, code);
}

// ---------------------------------------------------------------- bf16
// bf16 -> fp32 is exact: the bf16 pattern is the upper half of the float.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &r, float *f)
{
    f[0] = bf_lo(r.x); f[1] = bf_hi(r.x);
    f[2] = bf_lo(r.y); f[3] = bf_hi(r.y);
    f[4] = bf_lo(r.z); f[5] = bf_hi(r.z);
    f[6] = bf_lo(r.w); f[7] = bf_hi(r.w);
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------- ordering
// Total order of floats as unsigned keys (-0 folded onto +0).
__device__ __forceinline__ uint32_t float_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Total order of doubles as unsigned 64-bit keys (-0 folded onto +0).
__device__ __forceinline__ uint64_t double_key(double f)
{
    uint64_t u = (uint64_t)__double_as_longlong(f);
    if (u == 0x8000000000000000ull) u = 0;
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// exp(y) for y <= 0, returned in fp64 so that results below fp32's range
// survive.  Above -80 this is expf; below, exp(y) = 2^-k exp(y + k ln 2)
// with the shift done in fp64 and expf on the reduced argument.
__device__ __forceinline__ double exp_wide(float y)
{
    if (y > -80.f) return (double)expf(y);
    const int k = (int)ceilf(-y * 1.4426950408889634f);
    const double r = (double)y + (double)k * 0.6931471805599453;
    return ldexp((double)expf((float)r), -k);
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

__device__ __forceinline__ int warp_isum(int v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.  scratch: >= 33 ints.
__device__ __forceinline__ int block_exscan(int v, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nw = (blockDim.x + 31) >> 5;
    int incl = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        int t = __shfl_up_sync(kFull, incl, m);
        if (lane >= m) incl += t;
    }
    __syncthreads();
    if (lane == 31) scratch[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? scratch[lane] : 0;
        int si = s;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            int t = __shfl_up_sync(kFull, si, m);
            if (lane >= m) si += t;
        }
        if (lane < nw) scratch[lane] = si - s;
        if (lane == nw - 1) scratch[32] = si;
    }
    __syncthreads();
    int ex = scratch[wid] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return ex;
}

// Is step t a utility-refresh step?  t = 1 and every T-th step after it
// (InertiaKV-Lazy); T = 0 is the Score-Free operating point: the utilities
// are scored at the first decode step only and the ranking stays frozen.
__host__ __device__ __forceinline__ bool is_refresh(int t, int T)
{
    if (T == 0) return t == 1;
    return T == 1 || ((t - 1) % T) == 0;
}

}  // namespace kvc
