// routed.cu -- routed row combine (a mixture-of-experts combine) on sm_103a.
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section
// "Separate route and payload lookahead"): for each token the routes are
// visited in order; a route's row id selects a row of the payload matrix; a
// missing id (negative) suppresses the route's weight and payload reads and
// leaves the sum unchanged; otherwise the weighted payload -- the route's
// weight times each element of the selected row, one f32 product -- is
// added to the token's f32 sum.  Reading taken: product and sum are rounded
// separately (no fused multiply-add), so the result is defined to the bit.
//
// GB300 design
//  * One warp per token.  The pages read each route's id two routes ahead
//    and its payload one route ahead; here lane r loads route r's id (and,
//    when the id is present, its weight) once, before any payload is read,
//    so every id is known when the payload stream starts.
//  * The token's output row is produced in column blocks of 512 floats; for
//    each block, lane 0 streams the valid routes' 2 KiB row pieces, in route
//    order, into the warp's ring of `depth` stages with bulk copies
//    (cp.async.bulk) completing on per-stage mbarriers, and runs ahead into
//    the next block.  Every lane adds its four float4 slots of each piece
//    into sixteen f32 accumulators (consecutive lanes, consecutive 16-byte
//    words: conflict-free reads), then stores them.
//  * Two stages per warp keep the ring at 4 KiB, so 24 CTAs of two warps fit
//    an SM and a 4096-token workload runs in one wave (measured: depth 2
//    42 us, depth 4 64 us, depth 8 50 us).
//  * Rows whose width is not a multiple of 4 floats, unaligned inputs or
//    more than 32 routes take plain loads in the same order (same bits).
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT and
//    the token's outputs are NaN.  Ids at or past the row count are flagged
//    (LOOM_DEVERR_COUNT_RANGE) and treated as missing.
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

using dev::FULL_MASK;

constexpr int RC_BLOCK = 512;                   // floats of one column block
constexpr int RC_SLOTS = RC_BLOCK / 128;        // float4 slots per lane per block

__device__ __forceinline__ float weighted_add(float sum, float w, float x)
{
    return __fadd_rn(sum, __fmul_rn(w, x));
}

// Route r of token t: its id when present and in range, else -1 (flagging
// ids past the last row).
__device__ __forceinline__ int32_t route_id(const RoutedParams &p, int64_t t, int r)
{
    const int32_t id = __ldg(p.ids + t * p.routes + r);
    if (id >= p.rows) {
        dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
        return -1;
    }
    return id < 0 ? -1 : id;
}

__global__ void __launch_bounds__(256) routed_staged_kernel(const RoutedParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * warps + warp;
    if (t >= p.tokens)
        return;   // over-dispatched warp: no loads, no stores
    const int D = p.depth;
    const uint32_t stage_bytes = RC_BLOCK * 4;
    const uint32_t ring0 = dev::smem_u32(smem) + (uint32_t)warp * D * stage_bytes;
    const uint32_t bar0 = dev::smem_u32(smem) + (uint32_t)warps * D * stage_bytes + (uint32_t)warp * D * 8;

    // lane r: route r's id and weight (the weight only when the id is present)
    int32_t id = -1;
    float w = 0.f;
    if (lane < p.routes) {
        id = route_id(p, t, lane);
        if (id >= 0)
            w = __ldg(p.weights + t * p.routes + lane);
    }
    const uint32_t valid = __ballot_sync(FULL_MASK, id >= 0);
    const int nv = __popc(valid);
    const int nb = dev::ceil_div_i32(p.width, RC_BLOCK);
    const int total = nb * nv;   // pieces: block-major, valid routes in order

    if (lane == 0) {
        for (int s = 0; s < D; ++s)
            dev::mbar_init(bar0 + 8 * s, 1);
        dev::fence_barrier_init();
    }
    __syncwarp();
    const uint64_t policy = dev::l2_evict_first_policy();

    // lane k: the route of the k-th valid route (the k-th set bit of `valid`),
    // and that route's row id and weight, so that a piece needs one shuffle
    int kth = 0;
    {
        uint32_t m = valid;
        for (int i = 0; i < lane && m; ++i)
            m &= m - 1;
        kth = m ? __ffs(m) - 1 : 0;
    }
    const int32_t kid = __shfl_sync(FULL_MASK, id, kth);
    const float kw = __shfl_sync(FULL_MASK, w, kth);
    // piece i: block i / nv, the (i % nv)-th valid route; the cursor advances by increments
    int issued = 0, pb = 0, pk = 0, ps = 0;
    auto issue = [&]() {
        if (issued >= total)
            return;
        const int32_t rid = __shfl_sync(FULL_MASK, kid, pk);
        if (lane == 0 && !p.inject_stall) {
            const int32_t c0 = pb * RC_BLOCK;
            const uint32_t bytes = (uint32_t)min(RC_BLOCK, p.width - c0) * 4u;
            dev::mbar_arrive_expect_tx(bar0 + 8 * ps, bytes);
            dev::bulk_g2s(ring0 + (uint32_t)ps * stage_bytes, p.payload + (int64_t)rid * p.width + c0, bytes,
                          bar0 + 8 * ps, policy);
        }
        ++issued;
        if (++pk == nv) {
            pk = 0;
            ++pb;
        }
        ps = (ps + 1 == D) ? 0 : ps + 1;
    };
    for (int s = 0; s < D; ++s)
        issue();

    bool ok = true;
    int consumed = 0, cs = 0;
    uint32_t cphase = 0;
    float *out_row = p.out + t * p.width;
    for (int b = 0; b < nb; ++b) {
        const int32_t c0 = b * RC_BLOCK;
        const int32_t n4 = min(RC_BLOCK, p.width - c0) / 4;   // float4 slots in this block
        float acc[RC_SLOTS][4];
#pragma unroll
        for (int i = 0; i < RC_SLOTS; ++i)
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        for (int k = 0; k < nv && ok; ++k) {
            const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, p.wait_ns);
            if (!__all_sync(FULL_MASK, landed)) {
                ok = false;
                break;
            }
            const float wk = __shfl_sync(FULL_MASK, kw, k);
            const float4 *piece = reinterpret_cast<const float4 *>(smem + (size_t)warp * D * stage_bytes +
                                                                   (size_t)cs * stage_bytes);
#pragma unroll
            for (int i = 0; i < RC_SLOTS; ++i) {
                const int q = lane + 32 * i;
                if (q < n4) {
                    const float4 x = piece[q];
                    acc[i][0] = weighted_add(acc[i][0], wk, x.x);
                    acc[i][1] = weighted_add(acc[i][1], wk, x.y);
                    acc[i][2] = weighted_add(acc[i][2], wk, x.z);
                    acc[i][3] = weighted_add(acc[i][3], wk, x.w);
                }
            }
            __syncwarp();
            ++consumed;
            cs = (cs + 1 == D) ? 0 : cs + 1;
            cphase ^= (cs == 0) ? 1u : 0u;
            issue();   // refill the stage just freed
        }
        const float nan = __int_as_float(0x7fc00000);
#pragma unroll
        for (int i = 0; i < RC_SLOTS; ++i) {
            const int q = lane + 32 * i;
            if (q < n4)
                reinterpret_cast<float4 *>(out_row + c0)[q] =
                    ok ? make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]) : make_float4(nan, nan, nan, nan);
        }
    }
    if (!ok) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        // let copies already in flight land before the warp leaves (bounded)
        if (!p.inject_stall) {
            int s = cs;
            uint32_t ph = cphase;
            for (int i = consumed; i < issued; ++i) {
                dev::mbar_wait_bounded(bar0 + 8 * s, ph, p.wait_ns);
                s = (s + 1 == D) ? 0 : s + 1;
                ph ^= (s == 0) ? 1u : 0u;
            }
        }
    }
}

// Plain loads: one warp per token, lanes across the columns, routes in order.
__global__ void __launch_bounds__(256) routed_direct_kernel(const RoutedParams p)
{
    dev::follow_previous_kernel();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= p.tokens)
        return;
    float *out_row = p.out + t * p.width;
    for (int64_t c = lane; c < p.width; c += 32)
        out_row[c] = 0.f;
    for (int r = 0; r < p.routes; ++r) {
        const int32_t id = route_id(p, t, r);
        if (id < 0)
            continue;   // a missing route: no weight, no payload
        const float w = __ldg(p.weights + t * p.routes + r);
        const float *row = p.payload + (int64_t)id * p.width;
        for (int64_t c = lane; c < p.width; c += 32)
            out_row[c] = weighted_add(out_row[c], w, __ldg(row + c));
    }
}

}  // namespace

uint32_t routed_smem_bytes(bool staged, int depth, int warps)
{
    return staged ? (uint32_t)(warps * depth * (RC_BLOCK * 4 + 8)) : 0u;
}

cudaError_t launch_routed(const RoutedParams &p, bool staged, const loom_launch &L, cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    return staged ? launch_with(routed_staged_kernel, L, stream, p) : launch_with(routed_direct_kernel, L, stream, p);
}

}  // namespace loom
