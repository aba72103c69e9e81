// pkv_umma.cuh -- inline-PTX building blocks for the fifth-generation tensor
// cores (tcgen05) on sm_103a: tensor-memory (TMEM) allocation, shared-memory
// matrix descriptors, the instruction descriptor of a bf16 x bf16 -> fp32 MMA,
// MMA issue and completion, TMEM loads and stores, the fences that order them
// against thread synchronisation, and the named barriers of a warp group.
#pragma once

#include <stdint.h>

namespace pkv {

// Swizzle modes of a shared-memory matrix descriptor (bits 61-63).
enum : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

// Shared-memory matrix descriptor: start address (bits 0-13), leading-dimension
// byte offset (16-29) and stride-dimension byte offset (32-45), all in 16-byte
// units; descriptor version 1 (bit 46); base offset 0 (tiles are aligned to
// their swizzle pattern); swizzle mode (61-63).
//  * K-major, 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row groups
//    `sbo` bytes apart; a 16-element K step inside the 128-byte row advances the
//    start address by 32 bytes. `lbo` is unused.
//  * MN-major: rows of one K index hold the MN elements contiguously (64 bf16 in
//    a 128-byte row for the 128-byte swizzle, 32 in a 64-byte row for the 64-byte
//    one); `lbo` is the byte distance between such MN chunks, `sbo` between
//    groups of 8 K rows.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swizzle)
{
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (uint64_t(swizzle) << 61);
}

// Instruction descriptor of kind::f16 for bf16 A and B with an fp32 accumulator:
// D format fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), A / B
// MN-major (bits 15 / 16), N >> 3 (bits 17-22), M >> 4 (bits 24-28); dense, no
// negation, no saturation.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major,
                                                        bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
           (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread; asynchronous.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred acc;\n\t"
        "setp.ne.b32 acc, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, acc;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// One arrival on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// Warp-wide: allocate `ncols` TMEM columns (a power of two >= 32) and write the
// base address to shared memory at `slot`; then give up the right to allocate more.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide: free the columns tmem_alloc returned.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory writes of this thread become visible to the tensor cores and TMA
// (the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Warp-wide TMEM load, 32 lanes x 32 bits, 32 consecutive columns: lane i of the
// warp gets row (its lane quarter's first lane + i), columns col .. col + 31, into
// v[OFF .. OFF + 31]. Completes at tmem_wait_ld.
template <int OFF, int NV>
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[NV])
{
    static_assert(OFF + 32 <= NV, "tmem_ld32 target");
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[OFF + i] = __uint_as_float(r[i]);
}

// Warp-wide TMEM store of v[OFF .. OFF + 31], the layout of tmem_ld32. Completes at
// tmem_wait_st.
template <int OFF, int NV>
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[NV])
{
    static_assert(OFF + 32 <= NV, "tmem_st32 source");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[OFF + 0])), "r"(__float_as_uint(v[OFF + 1])), "r"(__float_as_uint(v[OFF + 2])),
        "r"(__float_as_uint(v[OFF + 3])), "r"(__float_as_uint(v[OFF + 4])), "r"(__float_as_uint(v[OFF + 5])),
        "r"(__float_as_uint(v[OFF + 6])), "r"(__float_as_uint(v[OFF + 7])), "r"(__float_as_uint(v[OFF + 8])),
        "r"(__float_as_uint(v[OFF + 9])), "r"(__float_as_uint(v[OFF + 10])), "r"(__float_as_uint(v[OFF + 11])),
        "r"(__float_as_uint(v[OFF + 12])), "r"(__float_as_uint(v[OFF + 13])), "r"(__float_as_uint(v[OFF + 14])),
        "r"(__float_as_uint(v[OFF + 15])), "r"(__float_as_uint(v[OFF + 16])), "r"(__float_as_uint(v[OFF + 17])),
        "r"(__float_as_uint(v[OFF + 18])), "r"(__float_as_uint(v[OFF + 19])), "r"(__float_as_uint(v[OFF + 20])),
        "r"(__float_as_uint(v[OFF + 21])), "r"(__float_as_uint(v[OFF + 22])), "r"(__float_as_uint(v[OFF + 23])),
        "r"(__float_as_uint(v[OFF + 24])), "r"(__float_as_uint(v[OFF + 25])), "r"(__float_as_uint(v[OFF + 26])),
        "r"(__float_as_uint(v[OFF + 27])), "r"(__float_as_uint(v[OFF + 28])), "r"(__float_as_uint(v[OFF + 29])),
        "r"(__float_as_uint(v[OFF + 30])), "r"(__float_as_uint(v[OFF + 31]))
        : "memory");
}

// The 16-column forms of tmem_ld32 / tmem_st32 (v[0 .. 15] of a 32-element array).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[32])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

// Named barrier `id` over `n` threads (a multiple of 32); the _or form returns
// whether any participating thread passed true.
__device__ __forceinline__ void bar_sync_named(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ bool bar_red_or_named(int id, int n, bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %3, 0;\n\t"
        "bar.red.or.pred pout, %1, %2, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(out)
        : "r"(id), "r"(n), "r"(uint32_t(pred))
        : "memory");
    return out != 0;
}

}  // namespace pkv
