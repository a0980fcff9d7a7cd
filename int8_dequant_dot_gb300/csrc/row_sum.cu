// row_sum.cu -- ragged full-tile f32 row sums on sm_103a.
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section "Derive
// full tiles from a ragged loop"): a segment values[rows][lanes] with a
// dynamic row count c is split into F = T*floor(c/T) full-tile rows and
// t = c - F tail rows; the full-tile rows are reduced across the lanes and
// added to a carried sum that starts at `initial`, and the tail rows are
// summed separately.  Outputs: (final_row = F, tail_count = t, full_sum,
// tail_sum).
//
// GB300 design
//  * One warp per segment (a "unit"); each warp owns a small sequence of
//    consecutive segments and a private ring of `depth` shared-memory stages.
//  * A segment's active rows [0, c) are one contiguous byte range (128*c
//    bytes when lanes = 32).  Lane 0 streams it into the ring as 4 KiB bulk
//    copies (cp.async.bulk) that complete on per-stage mbarriers; up to
//    `depth` chunks are in flight while the warp sums the oldest one.  This
//    is the read-ahead queue of the pages' pipeline(depth): depth 1 is the
//    serial control, and the depth never changes a result.
//  * Summation is error-free: every lane keeps double-word (hi, lo)
//    accumulators fed by TwoSum -- one packed f32x2 pair per output, so one
//    instruction advances two accumulators -- and the lanes are combined by a
//    __shfl_xor_sync butterfly (the subgroup reduce).  The pages add row sums
//    to the carried f32 sum in source order so that the result does not
//    depend on the schedule; here each addition is exact, so the carried
//    value is the exact sum (up to the rounding of the tiny lo parts) in any
//    association, and the association used is fixed by the shape alone.
//    Each f32 output is rounded once from hi + lo.
//  * Element e of a segment (row-major offset) goes to lane (e mod 128)/4 and
//    accumulator half e mod 2; every accumulator adds its elements in increasing e
//    and the two are folded in a fixed order (LaneSums::fold).  The direct path (plain
//    loads, for inputs that are not 16-byte aligned) uses the same mapping
//    and order, so both paths return identical bits.
//  * Over-dispatch: units past num_units in the last CTA do no loads and no
//    stores ("Kernels and launch configuration", "Over-dispatch safely").
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

using dev::DW;
using dev::DW2;
using dev::FULL_MASK;
using dev::pack2;

// Per-lane partial sums of one segment: one packed double word per side (full
// tiles, tail), its two halves taking the even and the odd elements of each
// float4 (elements 4q, 4q+2 to the first half and 4q+1, 4q+3 to the second,
// in element order).  One accumulator per side instead of one per float4 pair
// leaves the fold a single double-word addition and measured 2% faster on the
// segments, where instruction issue bounds the kernel.
struct LaneSums {
    DW2 full, tail;

    __device__ __forceinline__ void reset(float initial)
    {
        full.hi = pack2(initial, 0.f);
        full.lo = 0;
        tail.hi = tail.lo = 0;
    }
    __device__ __forceinline__ void full4(const float4 &v)
    {
        full.add(pack2(v.x, v.y));
        full.add(pack2(v.z, v.w));
    }
    __device__ __forceinline__ void tail4(const float4 &v)
    {
        tail.add(pack2(v.x, v.y));
        tail.add(pack2(v.z, v.w));
    }
    // A float4 whose first `nf` (1..3) elements are full-tile elements: each
    // element goes to one side and the other side receives an exact zero.
    __device__ __forceinline__ void straddle4(const float4 &v, int nf)
    {
        const bool f1 = nf > 1, f2 = nf > 2;
        full.add(pack2(v.x, f1 ? v.y : 0.f));
        full.add(pack2(f2 ? v.z : 0.f, 0.f));
        tail.add(pack2(0.f, f1 ? 0.f : v.y));
        tail.add(pack2(f2 ? 0.f : v.z, v.w));
    }
    // One trailing element at unit offset g (at most three per segment).
    __device__ __forceinline__ void add1(float x, int32_t g, int32_t split)
    {
        if (g < split)
            full.add(pack2(x, 0.f));
        else
            tail.add(pack2(x, 0.f));
    }

    // The lane's (full, tail) as one packed double word: the odd half of each
    // side added to its even half.
    __device__ __forceinline__ DW2 fold() const
    {
        float fh0, fh1, fl0, fl1, th0, th1, tl0, tl1;
        dev::unpack2(full.hi, fh0, fh1);
        dev::unpack2(full.lo, fl0, fl1);
        dev::unpack2(tail.hi, th0, th1);
        dev::unpack2(tail.lo, tl0, tl1);
        DW2 ft{pack2(fh0, th0), pack2(fl0, tl0)};
        ft.add_dw(pack2(fh1, th1), pack2(fl1, tl1));
        return ft;   // (full, tail)
    }

    // Elements [0, m) of a chunk starting at unit offset `off`, read through
    // `load(e)` (e = element offset in the chunk, a multiple of 4); elements
    // below `split` (unit offset) are full-tile elements.  Lane l takes the
    // float4s at e = 4l + 128i in increasing i.
    template <typename Load>
    __device__ __forceinline__ void chunk(Load load, int lane, int32_t off, int32_t m, int32_t split)
    {
        const int32_t mf = min(max(split - off, 0), m);   // chunk elements below the split
        int32_t e = lane * 4;
#pragma unroll 4
        for (; e + 4 <= mf; e += RS_SLOT_ELEMS)
            full4(load(e));
        if (e < m) {   // this lane's first float4 not wholly below the split
            if (e < mf)
                straddle4(load(e), mf - e);
            else
                tail4(load(e));
            e += RS_SLOT_ELEMS;
        }
#pragma unroll 4
        for (; e < m; e += RS_SLOT_ELEMS)
            tail4(load(e));
    }
};

// Issues the warp's chunks in order (lane 0 issues, every lane tracks the cursor).
struct Producer {
    int pk, pj, ps;
    uint32_t issued;

    __device__ __forceinline__ void issue(const RowSumParams &p, int lane, int n, int64_t u0,
                                          int32_t nchunks, int32_t nbulk, int D, uint32_t ring0,
                                          uint32_t bar0, uint64_t policy)
    {
        while (pk < n) {
            if (pj < __shfl_sync(FULL_MASK, nchunks, pk))
                break;
            ++pk;
            pj = 0;
        }
        if (pk >= n)
            return;
        const int32_t nb = __shfl_sync(FULL_MASK, nbulk, pk);
        if (lane == 0 && !p.inject_stall) {
            const int32_t off = pj * p.chunk_elems;
            const uint32_t bytes = (uint32_t)min(p.chunk_elems, nb - off) * 4u;
            const float *src = p.values + (u0 + pk) * p.unit_stride + off;
            dev::mbar_arrive_expect_tx(bar0 + 8 * ps, bytes);
            dev::bulk_g2s(ring0 + ps * (p.chunk_elems * 4), src, bytes, bar0 + 8 * ps, policy);
        }
        ++pj;
        ++issued;
        ps = (ps + 1 == D) ? 0 : ps + 1;
    }
};

// Reduces the (full, tail) partials of up to four consecutive units across
// the warp and stores their sums; units past `g` are padding.
__device__ __forceinline__ void finish_group(const RowSumParams &p, int lane, int64_t ubase, int g,
                                             const DW2 &a, const DW2 &b, const DW2 &c, const DW2 &d)
{
    const DW2 k = dev::warp_allreduce4(a, b, c, d, lane);
    const int j = (lane >> 3) & 3;
    if ((lane & 7) == 0 && j < g) {
        float h0, h1, l0, l1;
        dev::unpack2(k.hi, h0, h1);
        dev::unpack2(k.lo, l0, l1);
        p.full_sum[ubase + j] = dev::dw_round(h0, l0);
        p.tail_sum[ubase + j] = dev::dw_round(h1, l1);
    }
}

// MINB: register budget hint (CTAs of 256 threads per SM).  3 caps registers
// for many short-lived warps (small segments); 2 suits long rows.
template <bool STAGED, int MINB>
__global__ void __launch_bounds__(256, MINB) row_sum_kernel(const RowSumParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int64_t u0 = ((int64_t)blockIdx.x * warps + warp) * p.units_per_warp;
    if (u0 >= p.num_units)
        return;  // over-dispatched warp: no loads, no stores
    const int n = (int)min((int64_t)p.units_per_warp, p.num_units - u0);
    const int32_t CH = p.chunk_elems;

    // Lane k describes unit u0 + k (units_per_warp <= 32).
    int32_t c = 0;
    float init = 0.f;
    if (lane < n) {
        const int32_t raw = p.counts ? __ldg(p.counts + u0 + lane) : p.count_scalar;
        c = min(max(raw, 0), p.rows);
        if (c != raw)
            dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
        init = p.initial ? __ldg(p.initial + u0 + lane) : p.initial_scalar;
    }
    const int32_t F = (c / p.tile) * p.tile;  // full-tile rows
    const int32_t n_active = c * p.lanes;     // active elements
    const int32_t split = F * p.lanes;        // first tail element
    const int32_t nbulk = n_active & ~3;      // elements moved as 16-byte blocks
    const int32_t nchunks = dev::ceil_div_i32(nbulk, CH);

    const int D = p.depth;
    float *ring = reinterpret_cast<float *>(smem) + (size_t)warp * D * CH;
    const uint32_t ring0 = dev::smem_u32(ring);
    const uint32_t bar0 = dev::smem_u32(smem + (size_t)warps * D * CH * sizeof(float)) + warp * D * 8;

    uint64_t policy = 0;
    if (STAGED) {
        if (lane == 0) {
            for (int s = 0; s < D; ++s)
                dev::mbar_init(bar0 + 8 * s, 1);
            dev::fence_barrier_init();
        }
        __syncwarp();
        policy = dev::l2_evict_first_policy();
    }

    Producer prod{0, 0, 0, 0u};
    if (STAGED)
        for (int s = 0; s < D; ++s)
            prod.issue(p, lane, n, u0, nchunks, nbulk, D, ring0, bar0, policy);

    int cs = 0;            // consumer stage
    uint32_t cphase = 0;   // parity of the phase the consumer waits for
    uint32_t consumed = 0;
    int failed_at = n;     // first unit whose data never arrived
    DW2 pend0{0, 0}, pend1{0, 0}, pend2{0, 0}, pend3{0, 0};   // folded partials of a group of 4

    for (int k = 0; k < n; ++k) {
        const int32_t kc = __shfl_sync(FULL_MASK, nchunks, k);
        const int32_t kb = __shfl_sync(FULL_MASK, nbulk, k);
        const int32_t ka = __shfl_sync(FULL_MASK, n_active, k);
        const int32_t ks = __shfl_sync(FULL_MASK, split, k);
        const float kinit = __shfl_sync(FULL_MASK, init, k);
        const float *ubase = p.values + (u0 + k) * p.unit_stride;

        LaneSums acc;
        acc.reset(lane == 0 ? kinit : 0.f);
        bool ok = true;
        for (int j = 0; j < kc; ++j) {
            const int32_t off = j * CH;
            const int32_t m = min(CH, kb - off);
            if (STAGED) {
                const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, p.wait_ns);
                if (!__all_sync(FULL_MASK, landed)) {
                    ok = false;
                    break;
                }
                const float4 *s4 = reinterpret_cast<const float4 *>(ring + (size_t)cs * CH);
                acc.chunk([&](int32_t e) { return s4[e >> 2]; }, lane, off, m, ks);
                __syncwarp();
                ++consumed;
                cs = (cs + 1 == D) ? 0 : cs + 1;
                cphase ^= (cs == 0) ? 1u : 0u;
                prod.issue(p, lane, n, u0, nchunks, nbulk, D, ring0, bar0, policy);  // refill
            } else {
                const float *src = ubase + off;
                acc.chunk(
                    [&](int32_t e) {
                        return make_float4(__ldg(src + e), __ldg(src + e + 1), __ldg(src + e + 2),
                                           __ldg(src + e + 3));
                    },
                    lane, off, m, ks);
            }
        }
        if (!ok) {
            failed_at = k;
            break;
        }
        // At most three trailing elements that do not fill a 16-byte block.
        if (lane < ka - kb) {
            const int32_t g = kb + lane;
            acc.add1(__ldg(ubase + g), g, ks);
        }
        const DW2 ft = acc.fold();
        const int q = k & 3;
        if (q == 0)
            pend0 = ft;
        else if (q == 1)
            pend1 = ft;
        else if (q == 2)
            pend2 = ft;
        else
            pend3 = ft;
        if (q == 3 || k == n - 1) {
            const DW2 z{0, 0};
            finish_group(p, lane, u0 + (k & ~3), q + 1, pend0, q >= 1 ? pend1 : z, q >= 2 ? pend2 : z,
                         q >= 3 ? pend3 : z);
        }
    }

    if (failed_at < n) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        // Units of the unfinished group before the failure still get their sums.
        const int q = failed_at & 3;
        if (q > 0) {
            const DW2 z{0, 0};
            finish_group(p, lane, u0 + (failed_at & ~3), q, pend0, q >= 2 ? pend1 : z,
                         q >= 3 ? pend2 : z, z);
        }
        // Let copies already in flight land before the warp leaves (bounded).
        if (STAGED && !p.inject_stall) {
            int s = cs;
            uint32_t ph = cphase;
            for (uint32_t i = consumed; i < prod.issued; ++i) {
                dev::mbar_wait_bounded(bar0 + 8 * s, ph, p.wait_ns);
                s = (s + 1 == D) ? 0 : s + 1;
                ph ^= (s == 0) ? 1u : 0u;
            }
        }
        if (lane >= failed_at && lane < n) {
            p.full_sum[u0 + lane] = __int_as_float(0x7fc00000);
            p.tail_sum[u0 + lane] = __int_as_float(0x7fc00000);
        }
    }

    if (lane < n) {
        const int64_t u = u0 + lane;
        p.final_row[u] = F;
        p.tail_count[u] = c - F;
    }
}

// ---------------------------------------------------------------------------
// Segments of 32-lane rows that fit the ring (128 * rows <= ring bytes): one
// bulk copy per segment.  A warp owns `units_per_warp` consecutive segments
// and a byte ring of p.chunk_elems floats in shared memory.  The active prefix
// of each segment (128 c bytes) goes whole into the ring behind the previous
// one, or at the ring's start when it would cross the end; up to `depth`
// segments are in flight (one mbarrier each, so depth 1 is the serial
// control), so short segments keep more copies in flight than fixed stages
// would, and the small ring leaves room for many warps per SM.  The warp
// waits once per segment and issues the next copies as soon as space frees.
// Lane l takes float4 l & 7 of rows (l >> 3) + 4i, i.e. the float4s at byte
// 16 l + 512 i of the segment -- the element-to-lane mapping and per-lane
// order of LaneSums::chunk -- with rows below F going to the full-tile sums
// and the others to the tail sums; the folding and the warp reduction are
// those of row_sum_kernel, so both kernels (and the direct path) return
// identical bits.  Error-free sums make the kernel bound by instruction
// issue, so the per-segment work is kept to one wait, two row loops and the
// ring bookkeeping.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) row_sum_seg_kernel(const RowSumParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int64_t u0 = ((int64_t)blockIdx.x * warps + warp) * p.units_per_warp;
    if (u0 >= p.num_units)
        return;  // over-dispatched warp: no loads, no stores
    const int n = (int)min((int64_t)p.units_per_warp, p.num_units - u0);

    // Lane k describes segment u0 + k (units_per_warp <= 32).
    int32_t c = 0, F = 0;
    float init = 0.f;
    if (lane < n) {
        const int32_t raw = p.counts ? __ldg(p.counts + u0 + lane) : p.count_scalar;
        c = min(max(raw, 0), p.rows);
        if (c != raw)
            dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
        init = p.initial ? __ldg(p.initial + u0 + lane) : p.initial_scalar;
        F = (c / p.tile) * p.tile;   // full-tile rows
    }

    const int Q = p.depth;                          // segments in flight
    const uint32_t R = (uint32_t)p.chunk_elems * 4u;   // ring bytes
    unsigned char *ring = smem + (size_t)warp * (R + ((8u * Q + 15u) & ~15u));   // 16-byte aligned rings
    const uint32_t ring0 = dev::smem_u32(ring);
    const uint32_t bar0 = ring0 + R;
    if (lane == 0) {
        for (int s = 0; s < Q; ++s)
            dev::mbar_init(bar0 + 8 * s, 1);
        dev::fence_barrier_init();
    }
    __syncwarp();
    const uint64_t policy = dev::l2_evict_first_policy();

    // Where a segment of `sz` bytes goes after the byte `cur`: behind it, or
    // at the start when it would cross the end.  Producer and consumer apply
    // the same rule, so the consumer finds every segment without a record.
    auto place = [R](uint32_t cur, uint32_t sz) { return cur + sz > R ? 0u : cur; };
    uint32_t wpos = 0;     // producer: end of the last segment issued
    int pj = 0, ps = 0;    // producer: next segment, its barrier
    uint32_t rpos = 0;     // start of the oldest segment not yet summed (segment k)
    int k = 0;
    // Issue every next segment that fits: at most Q in flight, and its bytes
    // clear of the segments not yet summed (those occupy [rpos, wpos) around
    // the ring).  An empty segment moves nothing; its barrier phase is
    // completed by an arrival that expects no bytes.
    auto produce = [&]() {
        while (pj < n && pj - k < Q) {
            const uint32_t sz = (uint32_t)__shfl_sync(FULL_MASK, c, pj) * 128u;
            const uint32_t pos = place(wpos, sz);
            const bool fits = pj == k || (rpos < wpos ? (pos == wpos || sz <= rpos)
                                                      : (pos == wpos && wpos + sz <= rpos));
            if (!fits)
                break;
            if (lane == 0) {
                if (sz == 0) {
                    dev::mbar_arrive_expect_tx(bar0 + 8 * ps, 0);
                } else if (!p.inject_stall) {
                    dev::mbar_arrive_expect_tx(bar0 + 8 * ps, sz);
                    dev::bulk_g2s(ring0 + pos, p.values + (u0 + pj) * p.unit_stride, sz, bar0 + 8 * ps, policy);
                }
            }
            wpos = pos + sz;
            ++pj;
            ps = (ps + 1 == Q) ? 0 : ps + 1;
        }
    };
    produce();

    int cs = 0;            // consumer's barrier
    uint32_t cphase = 0;   // parity of the phase the consumer waits for
    int failed_at = n;     // first segment whose data never arrived
    DW2 pend0{0, 0}, pend1{0, 0}, pend2{0, 0}, pend3{0, 0};   // folded partials of a group of 4
    const int g = lane >> 3;   // this lane's rows: g, g + 4, ...
    for (; k < n;) {
        const int32_t kc = __shfl_sync(FULL_MASK, c, k);
        const int32_t kF = __shfl_sync(FULL_MASK, F, k);
        const float kinit = __shfl_sync(FULL_MASK, init, k);
        LaneSums acc;
        acc.reset(lane == 0 ? kinit : 0.f);
        const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, p.wait_ns);
        if (!__all_sync(FULL_MASK, landed)) {
            failed_at = k;
            break;
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(ring + rpos) + lane;
        const int nf = kF > g ? (kF - g + 3) >> 2 : 0;   // this lane's full-tile rows
        const int na = kc > g ? (kc - g + 3) >> 2 : 0;   // ... and all its active rows
        int i = 0;
#pragma unroll 4
        for (; i < nf; ++i)
            acc.full4(s4[32 * i]);
#pragma unroll 4
        for (; i < na; ++i)
            acc.tail4(s4[32 * i]);
        __syncwarp();
        // segment k is summed: its bytes are free, the next one is the oldest
        const uint32_t end = rpos + (uint32_t)kc * 128u;
        ++k;
        rpos = k < n ? place(end, (uint32_t)__shfl_sync(FULL_MASK, c, k) * 128u) : end;
        cs = (cs + 1 == Q) ? 0 : cs + 1;
        cphase ^= (cs == 0) ? 1u : 0u;
        produce();
        const DW2 ft = acc.fold();
        const int q = (k - 1) & 3;
        if (q == 0)
            pend0 = ft;
        else if (q == 1)
            pend1 = ft;
        else if (q == 2)
            pend2 = ft;
        else
            pend3 = ft;
        if (q == 3 || k == n) {
            const DW2 z{0, 0};
            finish_group(p, lane, u0 + ((k - 1) & ~3), q + 1, pend0, q >= 1 ? pend1 : z, q >= 2 ? pend2 : z,
                         q >= 3 ? pend3 : z);
        }
    }

    if (failed_at < n) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        // Segments of the unfinished group before the failure still get their sums.
        const int q = failed_at & 3;
        if (q > 0) {
            const DW2 z{0, 0};
            finish_group(p, lane, u0 + (failed_at & ~3), q, pend0, q >= 2 ? pend1 : z, q >= 3 ? pend2 : z, z);
        }
        // Let copies already in flight land before the warp leaves (bounded).
        if (!p.inject_stall) {
            int s = cs;
            uint32_t ph = cphase;
            for (int j = failed_at; j < pj; ++j) {
                dev::mbar_wait_bounded(bar0 + 8 * s, ph, p.wait_ns);
                s = (s + 1 == Q) ? 0 : s + 1;
                ph ^= (s == 0) ? 1u : 0u;
            }
        }
        if (lane >= failed_at && lane < n) {
            p.full_sum[u0 + lane] = __int_as_float(0x7fc00000);
            p.tail_sum[u0 + lane] = __int_as_float(0x7fc00000);
        }
    }

    if (lane < n) {
        const int64_t u = u0 + lane;
        p.final_row[u] = F;
        p.tail_count[u] = c - F;
    }
}

}  // namespace

int row_sum_default_units_per_warp(int32_t rows, int32_t lanes)
{
    // About 32 KiB of (maximum) data per warp: long enough for the read-ahead
    // ring to reach steady state, short enough for many CTAs per SM (63 x 32
    // segments: 4 per warp; rows of 8 KiB or more: 1 per warp).
    const int64_t unit_bytes = (int64_t)rows * lanes * 4;
    if (unit_bytes <= 0)
        return 32;
    int64_t upw = (32 * 1024) / unit_bytes;
    if (upw < 1)
        upw = 1;
    if (upw > 32)
        upw = 32;
    return (int)upw;
}

uint32_t row_sum_smem_bytes(bool staged, int depth, int warps, int chunk_elems)
{
    if (!staged)
        return 0;
    return (uint32_t)(warps * depth * (chunk_elems * 4 + 8));
}

uint32_t row_sum_seg_smem_bytes(int depth, int warps, int ring_bytes)
{
    return (uint32_t)(warps * (ring_bytes + ((8 * depth + 15) & ~15)));
}

cudaError_t launch_row_sum(const RowSumParams &p, bool staged, const loom_launch &L,
                           cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    if (L.kernel == LOOM_KERNEL_ROWSUM_SEGMENTS)
        return launch_with(row_sum_seg_kernel, L, stream, p);
    const bool small_units = (int64_t)p.rows * p.lanes <= 4096;
    if (staged)
        return small_units ? launch_with(row_sum_kernel<true, 3>, L, stream, p)
                           : launch_with(row_sum_kernel<true, 2>, L, stream, p);
    return small_units ? launch_with(row_sum_kernel<false, 3>, L, stream, p)
                       : launch_with(row_sum_kernel<false, 2>, L, stream, p);
}

}  // namespace loom
