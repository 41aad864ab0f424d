// kvc_umma.cuh -- fifth-generation tensor core (tcgen05) helpers (sm_103a):
// shared-memory operand descriptors, the instruction descriptor for bf16
// inputs with fp32 accumulation, tensor-memory allocation, MMA issue and
// completion, and accumulator loads.
//
// Operand layout used throughout: a K-major 128 x 128 bf16 tile stored as two
// 16 KB boxes (k = 0..63, k = 64..127) of 128 rows x 128 bytes with the TMA
// 128-byte swizzle, i.e. exactly what a 2D TMA load of {64, 128} boxes with
// CU_TENSOR_MAP_SWIZZLE_128B writes.  Step ks (16 k-elements, 32 bytes) of the
// contraction starts (ks >> 2) boxes and (ks & 3) * 32 bytes into the tile.
#pragma once

#include "kvc_tma.cuh"

namespace kvc {

constexpr int kUmmaBox = 128 * 128;          // bytes of one 128-row x 64-column box

// Byte offset of k-step ks (0..7) inside a 128 x 128 operand tile.
__host__ __device__ constexpr uint32_t umma_kstep(int ks)
{
    return (uint32_t)((ks >> 2) * kUmmaBox + (ks & 3) * 32);
}

// Shared-memory matrix descriptor: start address >> 4 in bits 0-13, leading
// byte offset (unused by the swizzled K-major form; 16 bytes) in bits 16-29,
// stride byte offset between 8-row groups (1024 bytes) in bits 32-45, the
// descriptor version (1) at bit 46 and the 128-byte swizzle mode (2) in bits
// 61-63.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Descriptor of k-step ks of an operand whose k-step 0 has descriptor d0: the
// steps differ only in the start-address field (address >> 4, no carry for a
// shared-memory address), so this is one 64-bit add of a constant.
__device__ __forceinline__ uint64_t umma_sdesc_step(uint64_t d0, int ks)
{
    return d0 + (uint64_t)(umma_kstep(ks) >> 4);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Whole-warp tensor-memory allocation of ncols columns (a power of two >= 32);
// the base address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-wide load of 32 consecutive fp32 columns of this warp's 32 lanes
// (lane quarter = warp index mod 4); returns after the load has landed.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

#define KVC_R32(r)                                                                              \
    "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),          \
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),  \
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),            \
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),            \
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

// Asynchronous form: issue the load now, wait with tmem_wait_ld(), then pass
// every destination through tmem_bind() so that no use of the registers can
// be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32_async(uint32_t addr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_bind(uint32_t (&r)[32])
{
    asm volatile("" : KVC_R32(r)::"memory");
}

// 128 consecutive fp32 columns of this warp's 32 lanes: four loads in flight,
// one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t addr, float (&v)[128])
{
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32_async(addr, r0);
    tmem_ld32_async(addr + 32, r1);
    tmem_ld32_async(addr + 64, r2);
    tmem_ld32_async(addr + 96, r3);
    tmem_wait_ld();
    tmem_bind(r0);
    tmem_bind(r1);
    tmem_bind(r2);
    tmem_bind(r3);
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v[i] = __uint_as_float(r0[i]);
        v[32 + i] = __uint_as_float(r1[i]);
        v[64 + i] = __uint_as_float(r2[i]);
        v[96 + i] = __uint_as_float(r3[i]);
    }
}

// 64 consecutive fp32 columns of this warp's 32 lanes: two loads in flight.
__device__ __forceinline__ void tmem_ld64(uint32_t addr, float (&v)[64])
{
    uint32_t r0[32], r1[32];
    tmem_ld32_async(addr, r0);
    tmem_ld32_async(addr + 32, r1);
    tmem_wait_ld();
    tmem_bind(r0);
    tmem_bind(r1);
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v[i] = __uint_as_float(r0[i]);
        v[32 + i] = __uint_as_float(r1[i]);
    }
}

// 2^x on the special-function unit (relative error a few units in the last
// place; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace kvc
