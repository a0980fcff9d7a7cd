// stream_floor.cu -- a read-only streaming probe: one launch that reads a byte
// range of device memory once and does nothing else with it.
//
// It is not a step of the method.  It measures what one launch over a given
// number of bytes can reach on this device -- launch, ramp to full bandwidth
// and tail included -- so that each kernel's time can be set against the
// time of a launch that only moves the same bytes.  Three schedules, each a
// way the kernels of this library move their inputs:
//  * grid-stride 16-byte loads, `depth` of them in flight per thread;
//  * one contiguous range per warp, 16-byte loads, `depth` in flight per lane;
//  * a ring of `depth` 8 KiB stages per CTA filled by bulk copies
//    (cp.async.bulk, one issuing lane, mbarrier completion).
// The loaded words are folded into a checksum that is stored only when it
// equals a fixed constant, so no load can be dropped and nothing else is
// written.
#include "common.cuh"
#include "internal.h"
#include "../../include/loom_tuning.h"

namespace loom {
namespace {

constexpr uint32_t FLOOR_MAGIC = 0x9E3779B9u;
constexpr int FLOOR_THREADS = 256;
constexpr uint32_t FLOOR_STAGE_BYTES = 8192;

__device__ __forceinline__ int4 ld_stream(const int4 *p)
{
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t fold(const int4 &v) { return (uint32_t)(v.x ^ v.y ^ v.z ^ v.w); }

template <int D>
__global__ void __launch_bounds__(FLOOR_THREADS) floor_grid_stride(const int4 *src, int64_t n16, uint64_t *sink)
{
    dev::follow_previous_kernel();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (D - 1) * stride < n16; i += D * stride) {
        int4 v[D];
#pragma unroll
        for (int j = 0; j < D; ++j)
            v[j] = ld_stream(src + i + j * stride);
#pragma unroll
        for (int j = 0; j < D; ++j)
            acc ^= fold(v[j]);
    }
    for (; i < n16; i += stride)
        acc ^= fold(ld_stream(src + i));
    if (acc == FLOOR_MAGIC)
        *sink = acc;
}

// Warp w of W reads the 16-byte words [w * n16 / W, (w + 1) * n16 / W).
template <int D>
__global__ void __launch_bounds__(FLOOR_THREADS) floor_warp_range(const int4 *src, int64_t n16, uint64_t *sink)
{
    dev::follow_previous_kernel();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t b = n16 / warps * w + min(w, n16 % warps);
    const int64_t e = b + n16 / warps + (w < n16 % warps ? 1 : 0);
    uint32_t acc = 0;
    int64_t i = b + lane;
    for (; i + (D - 1) * 32 < e; i += D * 32) {
        int4 v[D];
#pragma unroll
        for (int j = 0; j < D; ++j)
            v[j] = ld_stream(src + i + j * 32);
#pragma unroll
        for (int j = 0; j < D; ++j)
            acc ^= fold(v[j]);
    }
    for (; i < e; i += 32)
        acc ^= fold(ld_stream(src + i));
    if (acc == FLOOR_MAGIC)
        *sink = acc;
}

// CTA c of G streams the 8 KiB stages [c * S / G, (c + 1) * S / G) of the
// range (the last stage may be short) through a ring of `depth` stages; one
// warp, lane 0 issues the copies, every lane checks one word of each stage.
__global__ void __launch_bounds__(32) floor_bulk_ring(const char *src, int64_t bytes, int32_t depth, uint64_t wait_ns,
                                                     uint64_t *sink, int32_t *error)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x;
    const int64_t stages = (bytes + FLOOR_STAGE_BYTES - 1) / FLOOR_STAGE_BYTES;
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t s0 = stages / G * c + min(c, stages % G);
    const int64_t s1 = s0 + stages / G + (c < stages % G ? 1 : 0);
    const uint32_t ring = dev::smem_u32(smem);
    const uint32_t bar0 = ring + (uint32_t)depth * FLOOR_STAGE_BYTES;
    if (lane == 0) {
        for (int s = 0; s < depth; ++s)
            dev::mbar_init(bar0 + 8 * s, 1);
        dev::fence_barrier_init();
    }
    __syncwarp();
    const uint64_t pol = dev::l2_evict_first_policy();
    auto issue = [&](int64_t st) {
        if (lane == 0) {
            const int slot = (int)((st - s0) % depth);
            const int64_t off = st * FLOOR_STAGE_BYTES;
            const uint32_t n = (uint32_t)min((int64_t)FLOOR_STAGE_BYTES, bytes - off);
            dev::mbar_arrive_expect_tx(bar0 + 8 * slot, n);
            dev::bulk_g2s(ring + (uint32_t)slot * FLOOR_STAGE_BYTES, src + off, n, bar0 + 8 * slot, pol);
        }
    };
    int64_t next = s0;
    for (; next < s1 && next < s0 + depth; ++next)
        issue(next);
    uint32_t acc = 0;
    for (int64_t st = s0; st < s1; ++st) {
        const int slot = (int)((st - s0) % depth);
        const uint32_t parity = (uint32_t)(((st - s0) / depth) & 1);
        if (!__all_sync(dev::FULL_MASK, dev::mbar_wait_bounded(bar0 + 8 * slot, parity, wait_ns))) {
            dev::flag_error(error, LOOM_DEVERR_TIMEOUT);
            // let the copies already issued land before the CTA leaves (bounded)
            for (int64_t j = st; j < next; ++j)
                dev::mbar_wait_bounded(bar0 + 8 * ((j - s0) % depth), (uint32_t)(((j - s0) / depth) & 1), wait_ns);
            return;
        }
        uint32_t v;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(ring + (uint32_t)slot * FLOOR_STAGE_BYTES + 4u * lane));
        acc ^= v;
        __syncwarp();
        if (next < s1)
            issue(next++);
    }
    if (acc == FLOOR_MAGIC)
        *sink = acc;
}

}  // namespace

cudaError_t launch_stream_floor(const void *src, int64_t bytes, int32_t kind, int32_t depth, int32_t ctas_per_sm,
                                int32_t sm_count, uint64_t *sink, int32_t *error, uint64_t wait_ns,
                                cudaStream_t stream)
{
    if (bytes == 0)
        return cudaSuccess;
    loom_launch L = {};
    L.grid[1] = L.grid[2] = L.block[1] = L.block[2] = 1;
    L.grid[0] = (uint32_t)sm_count * (uint32_t)ctas_per_sm;
    const int64_t n16 = bytes / 16;
    if (kind == LOOM_FLOOR_BULK_RING) {
        L.block[0] = 32;
        L.smem_bytes = (uint32_t)depth * (FLOOR_STAGE_BYTES + 8);
        return launch_with(floor_bulk_ring, L, stream, static_cast<const char *>(src), bytes, depth, wait_ns, sink,
                           error);
    }
    L.block[0] = FLOOR_THREADS;
    const int4 *p = static_cast<const int4 *>(src);
    if (kind == LOOM_FLOOR_GRID_STRIDE)
        return depth == 4 ? launch_with(floor_grid_stride<4>, L, stream, p, n16, sink)
                          : launch_with(floor_grid_stride<8>, L, stream, p, n16, sink);
    return depth == 4 ? launch_with(floor_warp_range<4>, L, stream, p, n16, sink)
                      : launch_with(floor_warp_range<8>, L, stream, p, n16, sink);
}

}  // namespace loom
