// common.cuh -- device helpers shared by the streaming kernels (sm_103a).
//
//  * 1-D bulk copies global -> shared (cp.async.bulk) completing on an
//    mbarrier with a transaction count; these stage the read-ahead queue.
//  * Bounded mbarrier waits: a wait gives up after a time limit read from
//    %globaltimer, so a copy that never lands ends the kernel with an error
//    flag instead of a hang.
//  * Error-free double-word accumulation (TwoSum) for f32 streams.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/loom.h"

namespace loom {
namespace dev {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may be scheduled while the previous kernel on its stream drains.
// At entry it lets the next kernel be scheduled the same way, then waits
// until the previous kernel has completed and its memory operations are
// visible: nothing before this touches global memory, so stream order holds
// for every input and output whatever the previous kernel was.
__device__ __forceinline__ void follow_previous_kernel()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The wait alone (for a kernel that lets its dependents start later).
__device__ __forceinline__ void wait_previous_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// L2 policy for data that is read exactly once: evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data many CTAs re-read: evict last.
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is signalled on the
// mbarrier at `bar` as a transaction count of `bytes`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier; false once `limit_ns` has passed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0 && global_ns() - t0 > limit_ns)
            return false;
    }
}

__device__ __forceinline__ void flag_error(int32_t *word, int32_t bits)
{
    if (word)
        atomicOr(word, bits);
}

// The double word (hi, lo) rounded to f32.  Once the running sum has left the
// finite range, hi alone carries the IEEE result (an infinity, or NaN for
// opposite infinities or a NaN input) while lo, whose error terms subtract
// infinities, is NaN: hi is returned then.
__device__ __forceinline__ float dw_round(float hi, float lo) { return isfinite(hi) ? __fadd_rn(hi, lo) : hi; }

// ---------------------------------------------------------------------------
// Double-word f32 accumulator.  `hi + lo` carries the running sum; every
// addition to `hi` is split exactly into a rounded sum and its rounding error
// (Knuth's TwoSum, six operations, valid for any operand order), and the
// errors are summed in `lo` (the Sum2 scheme of Ogita, Rump and Oishi, 2005).
// The explicit _rn intrinsics keep the compiler from contracting or
// reassociating any of the steps.
// ---------------------------------------------------------------------------
struct DW {
    float hi;
    float lo;

    __device__ __forceinline__ void add(float x)
    {
        const float s = __fadd_rn(hi, x);
        const float bp = __fsub_rn(s, hi);
        const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
        hi = s;
        lo = __fadd_rn(lo, e);
    }

    // Combine with the accumulator of lane (lane ^ m) for m = 16..1.  Both
    // partners compute identical results (the rounded sum is commutative and
    // TwoSum's error term is exact), so every lane ends with the same value.
    __device__ __forceinline__ void warp_allreduce()
    {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            const float oh = __shfl_xor_sync(FULL_MASK, hi, m);
            const float ol = __shfl_xor_sync(FULL_MASK, lo, m);
            const float s = __fadd_rn(hi, oh);
            const float bp = __fsub_rn(s, hi);
            const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(oh, bp));
            hi = s;
            lo = __fadd_rn(__fadd_rn(lo, ol), e);
        }
    }

    // Add another double word (h, l): TwoSum on the high parts, low parts summed.
    __device__ __forceinline__ void add_dw(float h, float l)
    {
        const float s = __fadd_rn(hi, h);
        const float bp = __fsub_rn(s, hi);
        const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(h, bp));
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, l), e);
    }

    __device__ __forceinline__ float value() const { return dw_round(hi, lo); }
};

// ---------------------------------------------------------------------------
// Two independent double-word accumulators advanced together with packed
// f32x2 instructions (sm_100 and later): the same TwoSum steps as DW, each
// instruction working on two lanes of a 64-bit register pair.  Every packed
// operation rounds each half exactly as the scalar instruction would, so a
// DW2 gives the same bits as two DW accumulators fed the same values.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pack2(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

struct DW2 {
    uint64_t hi;
    uint64_t lo;

    __device__ __forceinline__ void add(uint64_t x)
    {
        const uint64_t s = add2(hi, x);
        const uint64_t bp = sub2(s, hi);
        const uint64_t e = add2(sub2(hi, sub2(s, bp)), sub2(x, bp));
        hi = s;
        lo = add2(lo, e);
    }

    // Add another packed double word, half by half (TwoSum on the high parts,
    // low parts summed), as DW::add_dw does for one half.
    __device__ __forceinline__ void add_dw(uint64_t h, uint64_t l)
    {
        const uint64_t s = add2(hi, h);
        const uint64_t bp = sub2(s, hi);
        const uint64_t e = add2(sub2(hi, sub2(s, bp)), sub2(h, bp));
        hi = s;
        lo = add2(add2(lo, l), e);
    }

    // The packed double word of lane (lane ^ m).
    __device__ __forceinline__ DW2 shfl_xor(int m) const
    {
        float h0, h1, l0, l1;
        unpack2(hi, h0, h1);
        unpack2(lo, l0, l1);
        return DW2{pack2(__shfl_xor_sync(FULL_MASK, h0, m), __shfl_xor_sync(FULL_MASK, h1, m)),
                   pack2(__shfl_xor_sync(FULL_MASK, l0, m), __shfl_xor_sync(FULL_MASK, l1, m))};
    }

    __device__ __forceinline__ void add_dw(const DW2 &o) { add_dw(o.hi, o.lo); }

    // Butterfly over the warp (lane ^ 16 .. lane ^ 1) of both halves at once;
    // as for DW, every lane ends with identical bits.
    __device__ __forceinline__ void warp_allreduce()
    {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            add_dw(shfl_xor(m));
    }
};

__device__ __forceinline__ DW2 select(bool c, const DW2 &a, const DW2 &b)
{
    return DW2{c ? a.hi : b.hi, c ? a.lo : b.lo};
}

// The butterfly of DW2::warp_allreduce applied to four values a, b, c, d at
// once.  At the first level the lanes with bit 4 clear keep (a, b) and the
// others keep (c, d), each sending its partner the pair it drops; at the
// second level bit 3 picks one of the two; the last three levels are the
// plain butterfly.  Every partial is formed from the same operands as in
// warp_allreduce (TwoSum and the low-part sum are symmetric in their
// operands), so lane l ends with exactly the bits warp_allreduce would give
// for value (l >> 3) & 3 -- a for lanes 0-7, b for 8-15, c for 16-23, d for
// 24-31 -- at about a third of the shuffles and additions.
__device__ __forceinline__ DW2 warp_allreduce4(const DW2 &a, const DW2 &b, const DW2 &c, const DW2 &d,
                                               int lane)
{
    const bool upper = (lane & 16) != 0;
    DW2 k1 = select(upper, c, a);
    DW2 k2 = select(upper, d, b);
    const DW2 r1 = select(upper, a, c).shfl_xor(16);
    const DW2 r2 = select(upper, b, d).shfl_xor(16);
    k1.add_dw(r1);
    k2.add_dw(r2);
    const bool odd = (lane & 8) != 0;
    DW2 k = select(odd, k2, k1);
    k.add_dw(select(odd, k1, k2).shfl_xor(8));
#pragma unroll
    for (int m = 4; m >= 1; m >>= 1)
        k.add_dw(k.shfl_xor(m));
    return k;
}

// ceil(a / b) for 0 <= a <= INT32_MAX and b >= 1, with no overflow near INT32_MAX.
__host__ __device__ __forceinline__ int32_t ceil_div_i32(int32_t a, int32_t b)
{
    return a / b + (a % b != 0);
}

__device__ __forceinline__ int32_t warp_sum_i32(int32_t v)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        v += __shfl_xor_sync(FULL_MASK, v, m);
    return v;
}

}  // namespace dev
}  // namespace loom
