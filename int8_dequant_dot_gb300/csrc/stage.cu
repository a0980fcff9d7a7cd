// stage.cu -- upload of ragged row-sum inputs: only the rows a row sum reads.
//
// A ragged segment's count says how many of its rows the row sums read; the
// rest of its rows are not inputs of the computation.  On GB300 the GPU's
// SMs read pinned (or, with address translation services, any) host memory
// in place over the host link, so the upload reads exactly each segment's
// active prefix there and writes it to the same offsets of the device
// buffer: a ragged gather that moves only the bytes the kernels will use.
// The link bounds it (about 211 GB/s on the GB300s measured, the same as the
// copy engines reach for a dense copy); the saving is in the bytes.
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

constexpr int ST_THREADS = 256;
constexpr int ST_CHUNK = ST_THREADS * 8;   // floats one CTA copies (8 per thread)

__global__ void __launch_bounds__(ST_THREADS) stage_rows_kernel(const StageParams p)
{
    dev::follow_previous_kernel();
    const int64_t s = (int64_t)blockIdx.x / p.chunks_per_unit;
    const int64_t k = (int64_t)blockIdx.x % p.chunks_per_unit;
    if (s >= p.num_units)
        return;
    const int32_t raw = p.counts ? __ldg(p.counts + s) : p.count_scalar;
    const int64_t c = min(max(raw, 0), p.rows);
    const int64_t active = c * p.lanes;
    const int64_t begin = k * ST_CHUNK;
    const int64_t end = min(active, begin + ST_CHUNK);
    if (begin >= end)
        return;
    const float *src = p.src + s * p.unit_stride;
    float *dst = p.dst + s * p.unit_stride;
    if (p.vec4) {
        // begin is a multiple of 4; float4 body, then at most three scalars
        const int64_t end4 = begin + ((end - begin) & ~int64_t(3));
        for (int64_t i = begin + 4 * threadIdx.x; i < end4; i += 4 * ST_THREADS)
            *reinterpret_cast<float4 *>(dst + i) = *reinterpret_cast<const float4 *>(src + i);
        if (threadIdx.x < end - end4)
            dst[end4 + threadIdx.x] = src[end4 + threadIdx.x];
    } else {
        for (int64_t i = begin + threadIdx.x; i < end; i += ST_THREADS)
            dst[i] = src[i];
    }
}

}  // namespace

int64_t stage_chunks_per_unit(int64_t rows, int64_t lanes)
{
    const int64_t n = rows * lanes;
    return n > 0 ? (n + ST_CHUNK - 1) / ST_CHUNK : 1;
}

cudaError_t launch_stage_rows(const StageParams &p, cudaStream_t stream)
{
    if (p.num_units == 0)
        return cudaSuccess;
    loom_launch L = {};
    L.grid[0] = (uint32_t)(p.num_units * p.chunks_per_unit);
    L.grid[1] = L.grid[2] = 1;
    L.block[0] = ST_THREADS;
    L.block[1] = L.block[2] = 1;
    return launch_with(stage_rows_kernel, L, stream, p);
}

}  // namespace loom
