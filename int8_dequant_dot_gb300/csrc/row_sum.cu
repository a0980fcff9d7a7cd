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
//  * Summation is error-free: every lane keeps a double-word (hi, lo)
//    accumulator per output fed by TwoSum, and the lanes are combined by a
//    __shfl_xor_sync butterfly (the subgroup reduce).  The pages add row sums
//    to the carried f32 sum in source order so that the result does not
//    depend on the schedule; here each addition is exact, so the carried
//    value is the exact sum (up to the rounding of the tiny lo parts) in any
//    association, and the association used is fixed by the shape alone.
//    Each f32 output is rounded once from hi + lo.
//  * Element e of a segment (row-major offset) goes to lane (e mod 128)/4;
//    every lane adds its elements in increasing e.  The direct path (plain
//    loads, for inputs that are not 16-byte aligned) uses the same mapping
//    and order, so both paths return identical bits.
//  * Over-dispatch: units past num_units in the last CTA do no loads and no
//    stores ("Kernels and launch configuration", "Over-dispatch safely").
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

using dev::DW;
using dev::FULL_MASK;

__device__ __forceinline__ void add_split(DW &full, DW &tail, float x, int32_t g, int32_t split)
{
    if (g < split)
        full.add(x);
    else
        tail.add(x);
}

// Four consecutive elements starting at unit offset g.
__device__ __forceinline__ void accumulate4(DW &full, DW &tail, const float4 &v, int32_t g,
                                            int32_t split)
{
    if (g + 4 <= split) {
        full.add(v.x);
        full.add(v.y);
        full.add(v.z);
        full.add(v.w);
    } else if (g >= split) {
        tail.add(v.x);
        tail.add(v.y);
        tail.add(v.z);
        tail.add(v.w);
    } else {
        add_split(full, tail, v.x, g, split);
        add_split(full, tail, v.y, g + 1, split);
        add_split(full, tail, v.z, g + 2, split);
        add_split(full, tail, v.w, g + 3, split);
    }
}

template <bool STAGED>
__global__ void __launch_bounds__(RS_WARPS * 32) row_sum_kernel(const RowSumParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t u0 = ((int64_t)blockIdx.x * RS_WARPS + warp) * p.units_per_warp;
    if (u0 >= p.num_units)
        return;  // over-dispatched warp: no loads, no stores
    const int n = (int)min((int64_t)p.units_per_warp, p.num_units - u0);

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
    const int32_t nchunks = (nbulk + RS_CHUNK_ELEMS - 1) / RS_CHUNK_ELEMS;

    const int D = p.depth;
    float *ring = reinterpret_cast<float *>(smem) + (size_t)warp * D * RS_CHUNK_ELEMS;
    const uint32_t ring0 = dev::smem_u32(ring);
    const uint32_t bar0 =
        dev::smem_u32(smem + (size_t)RS_WARPS * D * RS_CHUNK_ELEMS * sizeof(float)) + warp * D * 8;

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

    // Producer cursor: next chunk to issue is chunk pj of unit pk, into stage ps.
    int pk = 0, pj = 0, ps = 0;
    uint32_t issued = 0;
    auto produce = [&]() {
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
            const int32_t off = pj * RS_CHUNK_ELEMS;
            const uint32_t bytes = (uint32_t)min(RS_CHUNK_ELEMS, nb - off) * 4u;
            const float *src = p.values + (u0 + pk) * p.unit_stride + off;
            dev::mbar_arrive_expect_tx(bar0 + 8 * ps, bytes);
            dev::bulk_g2s(ring0 + ps * (RS_CHUNK_ELEMS * 4), src, bytes, bar0 + 8 * ps, policy);
        }
        ++pj;
        ++issued;
        ps = (ps + 1 == D) ? 0 : ps + 1;
    };

    if (STAGED)
        for (int s = 0; s < D; ++s)
            produce();

    int cs = 0;            // consumer stage
    uint32_t cphase = 0;   // parity of the phase the consumer waits for
    uint32_t consumed = 0;
    int failed_at = n;     // first unit whose data never arrived
    float out_full = 0.f, out_tail = 0.f;

    for (int k = 0; k < n; ++k) {
        const int32_t kc = __shfl_sync(FULL_MASK, nchunks, k);
        const int32_t kb = __shfl_sync(FULL_MASK, nbulk, k);
        const int32_t ka = __shfl_sync(FULL_MASK, n_active, k);
        const int32_t ks = __shfl_sync(FULL_MASK, split, k);
        const float kinit = __shfl_sync(FULL_MASK, init, k);
        const float *ubase = p.values + (u0 + k) * p.unit_stride;

        DW full{lane == 0 ? kinit : 0.f, 0.f};
        DW tail{0.f, 0.f};
        bool ok = true;
        for (int j = 0; j < kc; ++j) {
            const int32_t off = j * RS_CHUNK_ELEMS;
            const int32_t m = min(RS_CHUNK_ELEMS, kb - off);
            if (STAGED) {
                const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, p.wait_ns);
                if (!__all_sync(FULL_MASK, landed)) {
                    ok = false;
                    break;
                }
                const float4 *s4 = reinterpret_cast<const float4 *>(ring + cs * RS_CHUNK_ELEMS);
#pragma unroll 4
                for (int e = lane * 4; e < m; e += RS_SLOT_ELEMS)
                    accumulate4(full, tail, s4[e >> 2], off + e, ks);
                __syncwarp();
                ++consumed;
                cs = (cs + 1 == D) ? 0 : cs + 1;
                cphase ^= (cs == 0) ? 1u : 0u;
                produce();  // refill the stage just released
            } else {
                const float *src = ubase + off;
#pragma unroll 4
                for (int e = lane * 4; e < m; e += RS_SLOT_ELEMS) {
                    float4 v;
                    v.x = __ldg(src + e);
                    v.y = __ldg(src + e + 1);
                    v.z = __ldg(src + e + 2);
                    v.w = __ldg(src + e + 3);
                    accumulate4(full, tail, v, off + e, ks);
                }
            }
        }
        if (!ok) {
            failed_at = k;
            break;
        }
        // At most three trailing elements that do not fill a 16-byte block.
        if (lane < ka - kb) {
            const int32_t g = kb + lane;
            add_split(full, tail, __ldg(ubase + g), g, ks);
        }
        full.warp_allreduce();
        tail.warp_allreduce();
        if (lane == k) {
            out_full = full.value();
            out_tail = tail.value();
        }
    }

    if (failed_at < n) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        // Let copies already in flight land before the warp leaves (bounded).
        if (STAGED && !p.inject_stall) {
            int s = cs;
            uint32_t ph = cphase;
            for (uint32_t i = consumed; i < issued; ++i) {
                dev::mbar_wait_bounded(bar0 + 8 * s, ph, p.wait_ns);
                s = (s + 1 == D) ? 0 : s + 1;
                ph ^= (s == 0) ? 1u : 0u;
            }
        }
        if (lane >= failed_at) {
            out_full = __int_as_float(0x7fc00000);
            out_tail = __int_as_float(0x7fc00000);
        }
    }

    if (lane < n) {
        const int64_t u = u0 + lane;
        p.final_row[u] = F;
        p.tail_count[u] = c - F;
        p.full_sum[u] = out_full;
        p.tail_sum[u] = out_tail;
    }
}

}  // namespace

int row_sum_default_units_per_warp(int32_t rows, int32_t lanes)
{
    // About 32 KiB of (maximum) data per warp: long enough for the read-ahead
    // ring to reach steady state, short enough for many CTAs per SM.
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

uint32_t row_sum_smem_bytes(bool staged, int depth)
{
    if (!staged)
        return 0;
    return (uint32_t)(RS_WARPS * depth * (RS_CHUNK_ELEMS * 4 + 8));
}

cudaError_t launch_row_sum(const RowSumParams &p, bool staged, const loom_launch &L,
                           cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    return staged ? launch_with(row_sum_kernel<true>, L, stream, p)
                  : launch_with(row_sum_kernel<false>, L, stream, p);
}

}  // namespace loom
