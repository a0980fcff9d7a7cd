// tc_ptx.cuh -- inline-PTX wrappers of the tensor-core dot kernels (sm_103a):
// 2-D TMA loads, tcgen05 tensor-memory stores and loads, MMA issue and
// commit, the shared-memory descriptor of a 128-byte-swizzled K-major
// operand, and the exact int8 -> f16 conversion.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "common.cuh"

namespace loom {
namespace tc {

// 2-D tiled TMA load into this CTA's shared memory, completing on `bar` as a
// transaction count; x (innermost, bytes for a u8 map) must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory stores before later
// async-proxy reads (the MMA's operand fetch).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's lane, waited for.
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D (tensor memory) [+]= A (tensor memory) x B (shared-memory descriptor),
// kind::f16 with instruction descriptor `idesc`; accumulate when `acc` != 0.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Instruction descriptor of kind::f16: D f32, A and B f16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Shared-memory descriptor of a K-major operand with 128-byte swizzle:
// start address, leading offset (unused here, 16 B), stride between 8-row
// groups 1024 B, descriptor version 1, layout "128-byte swizzle".
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t start)
{
    return (uint64_t)((start >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Four signed bytes -> two f16x2 words (elements 0,1 and 2,3; low half first).
// A byte b becomes the f16 bit pattern 0x6400 | (b + 128), the value
// 1024 + b + 128, by a byte permute; one packed subtraction of 1152 leaves b
// (exact: every integer below 2048 is an f16).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;   // b + 128 as an unsigned byte
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));   // - 1152
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__device__ __forceinline__ int4 lds128(uint32_t addr)
{
    int4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// ---- bounded waits shared by the roles of a CTA ------------------------------
// A CTA keeps one abort word in shared memory.  A role whose wait runs out
// sets it (and LOOM_DEVERR_TIMEOUT in the error word); every other role gives
// up its next wait once it sees the word set.

__device__ __forceinline__ bool aborted(uint32_t abort_word)
{
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(abort_word));
    return v != 0;
}

__device__ __forceinline__ void set_abort(uint32_t abort_word, int32_t *error)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(abort_word), "r"(1u) : "memory");
    dev::flag_error(error, LOOM_DEVERR_TIMEOUT);
}

// Wait for a phase of `bar`; false once the CTA has aborted or `limit_ns`
// has passed (which aborts the CTA).
__device__ __forceinline__ bool role_wait(uint32_t abort_word, int32_t *error, uint64_t limit_ns, uint32_t bar,
                                          uint32_t parity)
{
    if (dev::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = dev::global_ns();
    for (uint32_t i = 1;; ++i) {
        if (dev::mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0) {
            if (aborted(abort_word))
                return false;
            if (dev::global_ns() - t0 > limit_ns) {
                set_abort(abort_word, error);
                return false;
            }
        }
    }
}

// The same, agreed by every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint32_t abort_word, int32_t *error, uint64_t limit_ns, uint32_t bar,
                                          uint32_t parity)
{
    return __all_sync(dev::FULL_MASK, role_wait(abort_word, error, limit_ns, bar, parity));
}

}  // namespace tc
}  // namespace loom
