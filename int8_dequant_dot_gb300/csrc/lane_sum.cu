// lane_sum.cu -- per-lane f32 sums: the pages' sum_rows, sum_vector_rows and
// guarded ragged rows, each over many independent segments.
//
// Method (Loom pages, "Tune loop unrolling and pipelining"):
//  * "Keep one checked source for experiments" (sum_rows): work-item l sums
//    column l of rows [0, count), an f32 recurrence from zero in row order.
//  * "Give each motif its own schedule" (sum_vector_rows): each row gives
//    lane l a four-element vector that is reduced into the carried sum, the
//    elements one at a time in element order.
//  * "Keep guards and inner loops in the source" (sum_guarded_rows): the row
//    range is rounded up to a multiple of four; rows at or past the count add
//    the identity and are never read; a row's partial is the f32 sum of its
//    first `columns` components, each the identity on lanes at or past
//    `active_lanes`.
// Every result is a fixed sequence of f32 additions, so the kernels give the
// oracle's bits exactly, for any schedule.
//
// GB300 design: one warp per segment (lane = column), a warp owning a few
// consecutive segments.  A segment's active rows are one contiguous byte
// range; lane 0 streams it into the warp's ring of `depth` chunks with bulk
// copies (cp.async.bulk) completing on per-stage mbarriers -- the pages'
// read-ahead queue, depth 1 being the serial control -- and every lane reads
// its column of each row from shared memory (consecutive lanes, consecutive
// words: conflict-free).  Inputs a bulk copy cannot take (unaligned, or rows
// that are not a multiple of 16 bytes) use plain loads with the same order.
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

using dev::FULL_MASK;

// The f32 additions of one row of one lane (`v` holds its WIDTH components).
template <int WIDTH, bool GUARDED>
__device__ __forceinline__ float add_row(float sum, const float (&v)[4], int columns, bool active)
{
    if (!GUARDED) {
#pragma unroll
        for (int j = 0; j < WIDTH; ++j)
            sum = __fadd_rn(sum, v[j]);
        return sum;
    }
    float component_sum = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (j < columns)
            component_sum = __fadd_rn(component_sum, active ? v[j] : 0.f);
    return __fadd_rn(sum, component_sum);
}

// A row past the count of a guarded segment adds the identity.
template <bool GUARDED>
__device__ __forceinline__ float pad_rows(float sum, int32_t count)
{
    if (GUARDED) {
        const int32_t end = (count + 3) / 4 * 4;
        for (int32_t r = count; r < end; ++r)
            sum = __fadd_rn(sum, 0.f);
    }
    return sum;
}

template <int WIDTH, bool GUARDED>
__device__ __forceinline__ void load_row(float (&v)[4], const float *row_base, int lane)
{
    if (WIDTH == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(row_base + lane * 4);
        v[0] = x.x;
        v[1] = x.y;
        v[2] = x.z;
        v[3] = x.w;
    } else {
        v[0] = row_base[lane];
        v[1] = v[2] = v[3] = 0.f;
    }
}

template <int WIDTH, bool GUARDED>
__global__ void __launch_bounds__(256) lane_sum_staged_kernel(const LaneSumParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int64_t u0 = ((int64_t)blockIdx.x * warps + warp) * p.units_per_warp;
    if (u0 >= p.num_units)
        return;   // over-dispatched warp: no loads, no stores
    const int n = (int)min((int64_t)p.units_per_warp, p.num_units - u0);
    const int D = p.depth;
    const int32_t row_elems = p.lanes * WIDTH;
    const int32_t CH = p.chunk_rows * row_elems;   // elements per chunk (whole rows)
    float *ring = reinterpret_cast<float *>(smem) + (size_t)warp * D * CH;
    const uint32_t ring0 = dev::smem_u32(ring);
    const uint32_t bar0 = dev::smem_u32(smem + (size_t)warps * D * CH * sizeof(float)) + warp * D * 8;

    // lane k describes unit u0 + k
    int32_t c = 0;
    if (lane < n) {
        const int32_t raw = p.counts ? __ldg(p.counts + u0 + lane) : p.count_scalar;
        c = min(max(raw, 0), p.rows);
        if (c != raw)
            dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
    }
    const int32_t nchunks = dev::ceil_div_i32(c, p.chunk_rows);

    if (lane == 0) {
        for (int s = 0; s < D; ++s)
            dev::mbar_init(bar0 + 8 * s, 1);
        dev::fence_barrier_init();
    }
    __syncwarp();
    const uint64_t policy = dev::l2_evict_first_policy();

    // producer cursor: unit pk, chunk pj; every lane tracks it, lane 0 issues
    int pk = 0, pj = 0, ps = 0;
    uint32_t issued = 0;
    auto issue = [&]() {
        while (pk < n && pj >= __shfl_sync(FULL_MASK, nchunks, pk)) {
            ++pk;
            pj = 0;
        }
        if (pk >= n)
            return;
        const int32_t kc = __shfl_sync(FULL_MASK, c, pk);
        if (lane == 0 && !p.inject_stall) {
            const int32_t r0 = pj * p.chunk_rows;
            const uint32_t bytes = (uint32_t)(min(p.chunk_rows, kc - r0) * row_elems) * 4u;
            const float *src = p.values + (u0 + pk) * p.unit_stride + (int64_t)r0 * row_elems;
            dev::mbar_arrive_expect_tx(bar0 + 8 * ps, bytes);
            dev::bulk_g2s(ring0 + ps * (uint32_t)CH * 4u, src, bytes, bar0 + 8 * ps, policy);
        }
        ++pj;
        ++issued;
        ps = (ps + 1 == D) ? 0 : ps + 1;
    };
    for (int s = 0; s < D; ++s)
        issue();

    int cs = 0;
    uint32_t cphase = 0, consumed = 0;
    bool ok = true;
    const bool active = !GUARDED || lane < p.active_lanes;
    for (int k = 0; k < n && ok; ++k) {
        const int32_t kc = __shfl_sync(FULL_MASK, c, k);
        const int32_t kn = __shfl_sync(FULL_MASK, nchunks, k);
        float sum = 0.f;
        for (int j = 0; j < kn; ++j) {
            const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, p.wait_ns);
            if (!__all_sync(FULL_MASK, landed)) {
                ok = false;
                break;
            }
            const int32_t rows_here = min(p.chunk_rows, kc - j * p.chunk_rows);
            const float *chunk = ring + (size_t)cs * CH;
            if (lane < p.lanes) {
#pragma unroll 8
                for (int32_t r = 0; r < rows_here; ++r) {
                    float v[4];
                    load_row<WIDTH, GUARDED>(v, chunk + (size_t)r * row_elems, lane);
                    sum = add_row<WIDTH, GUARDED>(sum, v, p.columns, active);
                }
            }
            __syncwarp();
            ++consumed;
            cs = (cs + 1 == D) ? 0 : cs + 1;
            cphase ^= (cs == 0) ? 1u : 0u;
            issue();   // refill the stage just freed
        }
        if (!ok) {
            // this unit and the rest of the warp's are lost: NaN, and a timeout flag
            dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
            for (int kk = k; kk < n; ++kk)
                if (lane < p.lanes)
                    p.out[(u0 + kk) * p.lanes + lane] = __int_as_float(0x7fc00000);
            break;
        }
        sum = pad_rows<GUARDED>(sum, kc);
        if (lane < p.lanes)
            p.out[(u0 + k) * p.lanes + lane] = sum;
    }
    if (!ok && !p.inject_stall) {
        // let copies already in flight land before the warp leaves (bounded)
        int s = cs;
        uint32_t ph = cphase;
        for (uint32_t i = consumed; i < issued; ++i) {
            dev::mbar_wait_bounded(bar0 + 8 * s, ph, p.wait_ns);
            s = (s + 1 == D) ? 0 : s + 1;
            ph ^= (s == 0) ? 1u : 0u;
        }
    }
}

// Plain loads: lane l reads its own column, rows in order.
template <int WIDTH, bool GUARDED>
__global__ void __launch_bounds__(256) lane_sum_direct_kernel(const LaneSumParams p)
{
    dev::follow_previous_kernel();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t u0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + warp) * p.units_per_warp;
    if (u0 >= p.num_units)
        return;
    const int n = (int)min((int64_t)p.units_per_warp, p.num_units - u0);
    const bool active = !GUARDED || lane < p.active_lanes;
    for (int k = 0; k < n; ++k) {
        const int32_t raw = p.counts ? __ldg(p.counts + u0 + k) : p.count_scalar;
        const int32_t c = min(max(raw, 0), p.rows);
        if (c != raw && lane == 0)
            dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
        if (lane >= p.lanes)
            continue;
        const float *seg = p.values + (u0 + k) * p.unit_stride;
        float sum = 0.f;
        for (int32_t r = 0; r < c; ++r) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            const float *x = seg + ((int64_t)r * p.lanes + lane) * WIDTH;
#pragma unroll
            for (int j = 0; j < WIDTH; ++j)
                v[j] = __ldg(x + j);
            sum = add_row<WIDTH, GUARDED>(sum, v, p.columns, active);
        }
        p.out[(u0 + k) * p.lanes + lane] = pad_rows<GUARDED>(sum, c);
    }
}

template <typename K>
cudaError_t go(K kernel, const LaneSumParams &p, const loom_launch &L, cudaStream_t stream)
{
    return launch_with(kernel, L, stream, p);
}

}  // namespace

uint32_t lane_sum_smem_bytes(bool staged, int depth, int warps, int chunk_elems)
{
    return staged ? (uint32_t)(warps * depth * (chunk_elems * 4 + 8)) : 0u;
}

cudaError_t launch_lane_sum(const LaneSumParams &p, int width, bool guarded, bool staged, const loom_launch &L,
                            cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    if (guarded)
        return staged ? go(lane_sum_staged_kernel<4, true>, p, L, stream)
                      : go(lane_sum_direct_kernel<4, true>, p, L, stream);
    if (width == 4)
        return staged ? go(lane_sum_staged_kernel<4, false>, p, L, stream)
                      : go(lane_sum_direct_kernel<4, false>, p, L, stream);
    return staged ? go(lane_sum_staged_kernel<1, false>, p, L, stream)
                  : go(lane_sum_direct_kernel<1, false>, p, L, stream);
}

}  // namespace loom
