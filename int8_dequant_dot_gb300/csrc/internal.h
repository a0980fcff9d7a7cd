// internal.h -- parameters and launchers shared between the host API layer
// (loom_api.cu) and the kernel translation units.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/loom.h"

namespace loom {

// ---- row sum -------------------------------------------------------------
constexpr int RS_DEFAULT_WARPS = 1;    // warps per CTA (a CTA's slot frees when its warp ends)
constexpr int RS_DEFAULT_WARPS_WIDE = 1;  // lanes = 1 (wide rows): a CTA slot frees when its row ends
constexpr int RS_DEFAULT_CHUNK_ELEMS = 1024;       // one staged chunk: 4 KiB of f32 ...
constexpr int RS_DEFAULT_CHUNK_ELEMS_LONG = 2048;  // ... 8 KiB for units above 4096 elements
constexpr int RS_SLOT_ELEMS = 128;      // one warp-wide read: 32 lanes x float4
constexpr int RS_DEFAULT_DEPTH = 2;    // measured best on GB300 (more warps per SM)

struct RowSumParams {
    const float *values;
    int64_t num_units;    // segments
    int64_t unit_stride;  // elements between segment starts
    int32_t rows, lanes, tile;
    const int32_t *counts;  // device counts, or NULL to use count_scalar
    int32_t count_scalar;
    const float *initial;   // device initial sums, or NULL to use initial_scalar
    float initial_scalar;
    int32_t *final_row, *tail_count;
    float *full_sum, *tail_sum;
    int32_t *error;         // device error word or NULL
    int32_t depth;          // chunks in flight per warp (staged path)
    int32_t units_per_warp;
    int32_t chunk_elems;    // elements per staged chunk (multiple of 128)
    uint64_t wait_ns;       // limit of each barrier wait
    int32_t inject_stall;   // test hook: issue no copies (every wait runs out)
};

// One-copy-per-segment kernel (32-lane rows): a byte ring per warp holding whole
// segments, `depth` of them in flight.
constexpr int RS_SEG_RING_BYTES = 8192;         // default ring: one segment of up to 64 rows, or several shorter
constexpr int RS_SEG_DEFAULT_DEPTH = 4;
constexpr int RS_SEG_DEFAULT_UNITS_PER_WARP = 4;   // measured best of 1..32 (4.3 waves of resident warps)
int row_sum_default_units_per_warp(int32_t rows, int32_t lanes);
uint32_t row_sum_smem_bytes(bool staged, int depth, int warps, int chunk_elems);
uint32_t row_sum_seg_smem_bytes(int depth, int warps, int ring_bytes);
cudaError_t launch_row_sum(const RowSumParams &p, bool staged, const loom_launch &L,
                           cudaStream_t stream);

// ---- dequantised dot -----------------------------------------------------
constexpr int DOT_DEFAULT_WARPS = 2;     // warps per CTA of the lanes-across-batch kernel
constexpr int DOT_K_DEFAULT_WARPS = 8;    // lanes-across-k kernel: warps per CTA ...
constexpr int DOT_K_DEFAULT_CTAS_PER_SM = 2;   // ... and CTAs per SM, and ...
constexpr int DOT_K_DEFAULT_DEPTH = 1;    // ... stages per warp: 16 one-stage rings of 8 KiB per SM
constexpr uint32_t DOT_K_X_SMEM_MAX = 64 * 1024;   // activations staged in shared memory up to this
constexpr int DOT_K_PIECE_WORDS = 2048;   // lanes-across-k kernel: a piece is 8 KiB of one row
constexpr int DOT_K_MAX_ROWS_PER_CTA = 1024;
constexpr int DOT_B_ROWS = 8;             // lanes-across-batch path: rows per warp
constexpr int DOT_B_CHUNK_WORDS = 128;    // ... 512 B of each of those rows per chunk
constexpr int DOT_MAX_BATCH_PER_PASS = 16;
constexpr int DOT_DEFAULT_DEPTH = 2;

struct DotParams {
    const int32_t *w;      // [n_rows][k/4]
    const float *scale_w;
    const int32_t *x;      // [batch][k/4]
    const float *scale_x;
    int32_t n_rows, k_words, batch;  // batch of this pass (<= 16)
    int32_t y_stride;      // elements between output rows (the full batch)
    float *y;              // already offset to this pass's first vector
    int32_t *acc;          // same layout as y, or NULL
    int32_t *error;
    int32_t depth;
    int32_t rows_per_cta;   // lanes-across-k kernel
    int32_t x_in_smem;      // lanes-across-k kernel: activations copied into shared memory
    uint64_t wait_ns;
    int32_t inject_stall;
    void *workspace;        // tensor-core path: split-band workspace, or NULL
    int64_t workspace_bytes;
};

enum class DotKernel { StagedK, StagedB, Direct, Tensor };

DotKernel dot_select(bool aligned, int32_t k, int32_t batch_pass);
uint32_t dot_smem_bytes(DotKernel kind, int depth, int warps, int64_t rows_per_cta);
// Default ring depth of a dp4a kernel.
inline int dot_default_depth(DotKernel kind) { return kind == DotKernel::StagedK ? DOT_K_DEFAULT_DEPTH : DOT_DEFAULT_DEPTH; }
// Lanes-across-k kernel: whether batch x k activation bytes are staged in shared
// memory behind `smem` bytes of rings and totals.
inline bool dot_k_x_fits(uint32_t smem, int64_t batch, int64_t k)
{
    return batch * k <= (int64_t)DOT_K_X_SMEM_MAX && smem + batch * k <= 227 * 1024;
}
// Lanes-across-k kernel: offset of the activations in shared memory (rings,
// barriers, row totals in front), also the size of everything before them.
__host__ __device__ inline uint32_t dot_k_x_offset(int warps, int depth, int64_t rows_per_cta)
{
    return ((uint32_t)(warps * depth * (DOT_K_PIECE_WORDS * 4 + 8) + 8 + rows_per_cta * 2 * 4) + 15u) & ~15u;
}
// Rows per CTA of a dp4a kernel: the lanes-across-k kernel spreads the rows over
// ctas_per_sm (0 = default) CTAs on each of `sms` SMs; the others take a fixed
// number of rows per warp.
int64_t dot_rows_per_cta(DotKernel kind, int64_t n_rows, int warps, int ctas_per_sm, int64_t sms);
cudaError_t launch_dot(const DotParams &p, DotKernel kind, const loom_launch &L, cudaStream_t stream);

// tensor-core path (dot_tc.cu): a persistent grid of one CTA per SM splits
// the list of 128-row x 128-k weight units into equal contiguous ranges; each
// CTA runs one or two pipelines on the halves of its range
struct DotTcConfig {
    int32_t depth;            // shared-memory stages per pipeline; 0 = default
    int32_t units_per_stage;  // 1 .. converter groups per pipeline; 0 = default
    int32_t a_bufs;           // f16 A buffers per pipeline in tensor memory; 0 = default
    int32_t pipes;            // pipelines per CTA, 1 or 2; 0 = default
    int32_t schedule;         // 0 choose, 1 whole bands, 2 split (workspace), 3 cluster per band,
                              // 4 whole rows per CTA (dot_tc_rows.cu)
};
struct DotTcPlan {
    int64_t grid;
    int64_t total_units;
    int32_t units_per_band, quantum;
    int32_t depth, ups, na, ng, pipes, groups;
    int32_t mode, cluster;    // how bands map onto CTAs; CTAs per band (cluster schedule)
    uint32_t cta_area, pipe_cols, pipe_bytes, smem_bytes;
    bool split;               // bands may be split between CTAs (needs the workspace)
    int64_t sm_count;         // SMs the grid was sized for
    // row-block schedule (mode DOT_TC_ROWS, dot_tc_rows.cu)
    int32_t rows_per_cta, block_rows, stages_per_block;
    uint32_t wbox, stage_bytes;
};
// mode of a DotTcPlan whose CTAs each own whole rows (dot_tc_rows.cu); the
// band schedules of dot_tc.cu use the modes below it
constexpr int DOT_TC_ROWS = 3;
bool dot_tc_eligible(bool aligned, int32_t k, int32_t batch_pass);
int dot_tc_threads(int pipes);
int dot_tc_rows_per_band();
bool dot_tc_plan(int64_t n_rows, int32_t k, int64_t sm_count, const DotTcConfig &cfg, bool split,
                 DotTcPlan *out);
int64_t dot_tc_workspace_bytes(const DotTcPlan &plan);
bool dot_tc_cluster_fits(const DotTcPlan &plan);
cudaError_t launch_dot_tc(const DotParams &p, const DotTcPlan &plan, cudaStream_t stream);
bool dot_tc_rows_plan(int64_t n_rows, int32_t k, int64_t sm_count, const DotTcConfig &cfg, bool forced,
                      DotTcPlan *out);
int dot_tc_rows_threads();
cudaError_t launch_dot_tc_rows(const DotParams &p, const DotTcPlan &plan, cudaStream_t stream);
// 2-D tensor map of a row-major u8 array [outer][inner] (recently used maps are reused)
bool encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                             uint32_t box_outer, CUtensorMapSwizzle swizzle);

// ---- per-lane f32 sums (lane_sum.cu): sum_rows, sum_vector_rows, guarded rows ----
struct LaneSumParams {
    const float *values;
    int64_t num_units;        // segments
    int64_t unit_stride;      // elements between segment starts
    int32_t rows, lanes;      // rows of lanes x width f32
    const int32_t *counts;    // per segment, or NULL: count_scalar
    int32_t count_scalar;
    int32_t columns, active_lanes;   // guarded rows only
    float *out;               // [segments][lanes]
    int32_t *error;
    int32_t depth;            // chunks in flight per warp (staged)
    int32_t units_per_warp;
    int32_t chunk_rows;       // rows per staged chunk
    uint64_t wait_ns;
    int32_t inject_stall;
};
uint32_t lane_sum_smem_bytes(bool staged, int depth, int warps, int chunk_elems);
cudaError_t launch_lane_sum(const LaneSumParams &p, int width, bool guarded, bool staged, const loom_launch &L,
                            cudaStream_t stream);

// ---- upload of ragged rows (stage.cu) ------------------------------------------
struct StageParams {
    const float *src;          // readable by the device: pinned host memory or device memory
    float *dst;                // device memory, same layout
    int64_t num_units, unit_stride, chunks_per_unit;
    int32_t rows, lanes;
    const int32_t *counts;     // device counts, or NULL: count_scalar
    int32_t count_scalar;
    int32_t vec4;              // 16-byte copies (both bases and the stride allow them)
};
int64_t stage_chunks_per_unit(int64_t rows, int64_t lanes);
cudaError_t launch_stage_rows(const StageParams &p, cudaStream_t stream);

// ---- routed row combine (routed.cu) -------------------------------------------
struct RoutedParams {
    const int32_t *ids;       // [tokens][routes], negative = missing
    const float *weights;     // [tokens][routes]
    const float *payload;     // [rows][width]
    float *out;               // [tokens][width]
    int64_t tokens;
    int32_t routes, rows, width;
    int32_t *error;
    int32_t depth;            // pieces in flight per warp (staged)
    uint64_t wait_ns;
    int32_t inject_stall;
};
constexpr int RC_DEFAULT_DEPTH = 2;   // measured best: every CTA of the workload resident at once
constexpr int RC_MAX_STAGED_ROUTES = 32;
uint32_t routed_smem_bytes(bool staged, int depth, int warps);
cudaError_t launch_routed(const RoutedParams &p, bool staged, const loom_launch &L, cudaStream_t stream);

// ---- the pages' packed-dot example (packed_dot.cu) ---------------------------
constexpr int PD_DEFAULT_DEPTH = 3;        // stages of the read-ahead ring ...
constexpr int PD_DEFAULT_RPS = 4;          // ... of 4 records (10 KiB): seven CTAs per SM (measured best)
constexpr int PD_MAX_RPS = 32;
constexpr int PD_MAX_STAGED_STREAMS = 64;  // one TMA box row holds every stream of a record
constexpr int PD_LANES_PER_CTA = 256;      // direct path; staged path: lanes per tile

struct PackedParams {
    const int32_t *fields;     // [problems][records][lanes] packed signed bytes
    const uint16_t *scales;    // [problems][records][lanes] f16 bit patterns
    const float *rhs;          // [problems][records][streams][4]
    int32_t problems, records, lanes, streams;
    const int32_t *counts;     // [problems] or NULL (count for every instance)
    int32_t count;
    const float *initial;      // [problems][lanes] or NULL
    float *out;                // [problems][lanes]
    int32_t *error;
    int32_t depth, rps;
    uint64_t wait_ns;
    int32_t inject_stall;
};
bool packed_dot_stageable(const PackedParams &q);
uint32_t packed_dot_smem_bytes(bool staged, int depth, int rps, int streams);
uint32_t packed_dot_threads(bool staged);
int64_t packed_dot_tiles(int64_t problems, int64_t lanes);   // staged path: tiles of 256 lanes
cudaError_t launch_packed_dot(const PackedParams &q, bool staged, const loom_launch &L, cudaStream_t stream);

// ---- read-only streaming probe (stream_floor.cu) --------------------------------
cudaError_t launch_stream_floor(const void *src, int64_t bytes, int32_t kind, int32_t depth, int32_t ctas_per_sm,
                                int32_t sm_count, uint64_t *sink, int32_t *error, uint64_t wait_ns,
                                cudaStream_t stream);

// ---- unpack ----------------------------------------------------------------
constexpr int UNPACK_BLOCK = 256;
cudaError_t launch_unpack(const int32_t *packed, int64_t n_words, float *out, const loom_launch &L,
                          cudaStream_t stream);

// Launch a kernel with the geometry of L (grid, block, dynamic smem) as a
// programmatic dependent of the previous kernel on the stream (the kernels
// wait for it at entry: see follow_previous_kernel in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_with(void (*kernel)(KArgs...), const loom_launch &L, cudaStream_t stream,
                        Args &&...args)
{
    if (L.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)L.smem_bytes);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid[0], L.grid[1], L.grid[2]);
    cfg.blockDim = dim3(L.block[0], L.block[1], L.block[2]);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace loom
