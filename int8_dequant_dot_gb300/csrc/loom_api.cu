// loom_api.cu -- host side of libloom: argument validation, the launch
// configuration routine and the extern "C" entry points of loom.h and
// loom_tuning.h.
//
// The launch configuration follows the Loom pages ("Kernels and launch
// configuration", sections "A kernel owns two signatures" and "Workload is
// not workgroup count"): workload scalars alone decide the geometry, the
// grid is the ceiling division of the workload by the units one CTA owns,
// and every entry point launches with exactly the geometry this routine
// returns, so the division lives in one place.
#include <cuda.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "../../include/loom_tuning.h"

namespace loom {
namespace {

constexpr uint64_t DEFAULT_WAIT_NS = 1000000000ull;  // 1 s per barrier wait
constexpr int64_t MAX_K = 131068;                   // 128*128*k < 2^31 and k % 4 == 0

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

int64_t ceil_div(int64_t n, int64_t d) { return (n + d - 1) / d; }

void fill_launch(loom_launch *out, int64_t grid, uint32_t block, uint32_t smem, uint32_t units,
                 uint32_t kernel)
{
    std::memset(out, 0, sizeof(*out));
    out->grid[0] = (uint32_t)grid;
    out->grid[1] = out->grid[2] = 1;
    out->block[0] = block;
    out->block[1] = out->block[2] = 1;
    out->cluster[0] = out->cluster[1] = out->cluster[2] = 1;
    out->subgroup_size = 32;
    out->smem_bytes = smem;
    out->units_per_cta = units;
    out->kernel = kernel;
}

struct Tuning {
    int depth;
    int path;
    int upw;
    int warps;
    int chunk_bytes;
    int stall;
    uint64_t wait_ns;
    DotTcConfig tc;
};

#ifdef LOOM_TEST_HOOKS
// Test build only (libloom_test.so): while set, the staged kernels issue no
// copies, so every wait on them runs out after the tuning's wait limit.  The
// shipping library has no way to turn this on.
std::atomic<int32_t> g_test_stall{0};
int32_t test_stall() { return g_test_stall.load(std::memory_order_relaxed); }
#else
int32_t test_stall() { return 0; }
#endif

bool valid_warps(int64_t w) { return w == 1 || w == 2 || w == 4 || w == 8; }
bool valid_chunk(int64_t b) { return b >= 512 && b <= 32768 && b % 512 == 0; }

// Measured on GB300: 4 KiB chunks for small segments, 8 KiB for long rows.
int64_t default_chunk_bytes(int64_t rows, int64_t lanes)
{
    return 4 * (rows * lanes > 4096 ? RS_DEFAULT_CHUNK_ELEMS_LONG : RS_DEFAULT_CHUNK_ELEMS);
}

loom_status read_tuning(const loom_tuning *t, int default_depth, Tuning *out)
{
    out->depth = default_depth;
    out->path = LOOM_PATH_AUTO;
    out->upw = 0;
    out->warps = 0;
    out->chunk_bytes = 0;
    out->stall = test_stall();
    out->wait_ns = DEFAULT_WAIT_NS;
    out->tc = DotTcConfig{0, 0, 0, 0, 0};
    if (!t)
        return LOOM_OK;
    if (t->depth < 0 || t->depth > LOOM_MAX_DEPTH || t->path < 0 || t->path > 3 ||
        t->units_per_warp < 0 || t->units_per_warp > 32 || t->wait_ns < 0 ||
        (t->warps_per_cta != 0 && !valid_warps(t->warps_per_cta)) ||
        (t->chunk_bytes != 0 && !valid_chunk(t->chunk_bytes)) || t->tc_units_per_stage < 0 ||
        t->tc_units_per_stage > 4 || t->tc_a_buffers < 0 || t->tc_a_buffers > 8 ||
        t->tc_pipelines < 0 || t->tc_pipelines > 2 || t->tc_schedule < 0 || t->tc_schedule > 4)
        return LOOM_ERR_ARG;
    if (t->depth)
        out->depth = t->depth;
    out->path = t->path;
    out->upw = t->units_per_warp;
    out->warps = t->warps_per_cta;
    out->chunk_bytes = t->chunk_bytes;
    if (t->wait_ns)
        out->wait_ns = (uint64_t)t->wait_ns;
    out->tc = DotTcConfig{t->depth, t->tc_units_per_stage, t->tc_a_buffers, t->tc_pipelines, t->tc_schedule};
    return LOOM_OK;
}

// SMs of the current device (the persistent tensor-core grid is sized by it).
loom_status current_sm_count(int64_t *sms)
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    *sms = n;
    return LOOM_OK;
}

// ---- geometry of each op ----------------------------------------------------

// depth or chunk_bytes of 0 take the kernel's default; *depth_out and
// *chunk_out (may be NULL) receive the values used.
loom_status row_sum_geometry(int64_t num_segments, int64_t rows, int64_t lanes, bool staged,
                             int64_t depth, int64_t upw, int64_t warps, int64_t chunk_bytes,
                             loom_launch *out, int32_t *depth_out = nullptr, int32_t *chunk_out = nullptr)
{
    if (num_segments < 0 || rows < 0 || (lanes != 1 && lanes != 32) || rows * lanes >= (1ll << 31))
        return LOOM_ERR_SHAPE;
    if (warps == 0)
        warps = lanes == 1 ? RS_DEFAULT_WARPS_WIDE : RS_DEFAULT_WARPS;
    // 32-lane segments whose active rows fit the ring (chunk_bytes, default 8 KiB) take
    // one copy each; with a smaller chunk size they stream in chunks
    const bool segs = staged && lanes == 32 && rows * 128 <= (chunk_bytes ? chunk_bytes : RS_SEG_RING_BYTES);
    if (chunk_bytes == 0)
        chunk_bytes = segs ? RS_SEG_RING_BYTES : default_chunk_bytes(rows, lanes);
    if (depth == 0)
        depth = segs ? RS_SEG_DEFAULT_DEPTH : RS_DEFAULT_DEPTH;
    if (depth < 1 || depth > LOOM_MAX_DEPTH || upw < 0 || upw > 32 || !valid_warps(warps) ||
        !valid_chunk(chunk_bytes))
        return LOOM_ERR_ARG;
    if (upw == 0)
        upw = segs ? RS_SEG_DEFAULT_UNITS_PER_WARP : row_sum_default_units_per_warp((int32_t)rows, (int32_t)lanes);
    const int64_t per_cta = warps * upw;
    const int64_t grid = ceil_div(num_segments, per_cta);
    if (grid > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    const uint32_t smem = segs ? row_sum_seg_smem_bytes((int)depth, (int)warps, (int)chunk_bytes)
                               : row_sum_smem_bytes(staged, (int)depth, (int)warps, (int)(chunk_bytes / 4));
    if (smem > 227 * 1024)
        return LOOM_ERR_ARG;
    fill_launch(out, grid, (uint32_t)warps * 32, smem, (uint32_t)per_cta,
                segs ? LOOM_KERNEL_ROWSUM_SEGMENTS : staged ? LOOM_KERNEL_ROWSUM_STAGED : LOOM_KERNEL_ROWSUM_DIRECT);
    if (depth_out)
        *depth_out = (int32_t)depth;
    if (chunk_out)
        *chunk_out = (int32_t)chunk_bytes;
    return LOOM_OK;
}

// engine: 0 = automatic, 1 = dp4a kernels only, 2 = tensor cores.  For the
// tensor-core kernel `tc` holds its schedule (tc.depth = stages), `split`
// whether a workspace lets bands be split between CTAs.  `sms` is the SM
// count the grid is sized for (0 = the current device's, read when the
// kernel needs it); *plan receives the tensor-core schedule.  For the
// lanes-across-k kernel `rows_per_warp` is its CTAs per SM (0 = default).
loom_status dot_geometry(int64_t n_rows, int64_t k, int64_t batch, bool aligned, int64_t depth,
                         int64_t warps, int64_t rows_per_warp, int64_t engine, const DotTcConfig &tc,
                         bool split, int64_t sms, loom_launch *out, DotTcPlan *plan)
{
    if (n_rows < 0 || n_rows > 0x7fffffff || k < 0 || k > MAX_K || (k % 4) != 0 || batch < 0 ||
        batch > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    if (depth < 0 || depth > LOOM_MAX_DEPTH || (warps != 0 && !valid_warps(warps)) || rows_per_warp < 0 ||
        rows_per_warp > 32 || engine < 0 || engine > 2 || sms < 0)
        return LOOM_ERR_ARG;
    const int32_t pass = (int32_t)(batch < DOT_MAX_BATCH_PER_PASS ? batch : DOT_MAX_BATCH_PER_PASS);
    const bool tc_ok = dot_tc_eligible(aligned, (int32_t)k, pass);
    const bool use_tc = (engine == 2 || (engine == 0 && pass >= 3)) && tc_ok;
    if (engine == 2 && !tc_ok)
        return aligned ? LOOM_ERR_SHAPE : LOOM_ERR_ALIGN;
    const DotKernel kind = use_tc ? DotKernel::Tensor : dot_select(aligned, (int32_t)k, pass);
    if (sms == 0 && (kind == DotKernel::Tensor || kind == DotKernel::StagedK)) {
        const loom_status st = current_sm_count(&sms);   // both grids are sized by the device
        if (st != LOOM_OK)
            return st;
    }
    if (use_tc) {
        DotTcPlan pl;
        DotTcConfig c = tc;
        c.depth = (int32_t)depth;
        if (!dot_tc_plan(n_rows, (int32_t)k, sms, c, split, &pl))
            return LOOM_ERR_ARG;
        const int64_t grid = batch == 0 ? 0 : pl.grid;
        // per CTA (at most): rows of W for the row-block schedule; else 128 x 128 weight
        // units, a cluster's share of one band or a share of the list
        const int64_t per_cta = pl.grid == 0                ? 0
                                : pl.mode == DOT_TC_ROWS    ? pl.rows_per_cta
                                : pl.cluster > 1            ? ceil_div(pl.units_per_band, pl.cluster)
                                                            : pl.quantum * ceil_div(pl.total_units / pl.quantum, pl.grid);
        const uint32_t id = pl.mode == DOT_TC_ROWS ? LOOM_KERNEL_DOT_TENSOR_ROWS
                            : pl.split             ? LOOM_KERNEL_DOT_TENSOR_SPLIT
                                                   : LOOM_KERNEL_DOT_TENSOR;
        fill_launch(out, grid, (uint32_t)dot_tc_threads(pl.pipes), pl.smem_bytes, (uint32_t)per_cta, id);
        out->cluster[0] = (uint32_t)pl.cluster;
        if (plan)
            *plan = pl;
        return LOOM_OK;
    }
    if (depth == 0)
        depth = dot_default_depth(kind);
    if (warps == 0)   // lanes across k: at most 128 KiB of rings per CTA whatever the depth
        warps = kind != DotKernel::StagedK ? DOT_DEFAULT_WARPS
                : depth <= 2               ? DOT_K_DEFAULT_WARPS
                : depth <= 4               ? DOT_K_DEFAULT_WARPS / 2
                                           : DOT_K_DEFAULT_WARPS / 4;
    const int64_t rows_per_cta = dot_rows_per_cta(kind, n_rows, (int)warps, (int)rows_per_warp, sms);
    const int64_t grid = (batch == 0) ? 0 : ceil_div(n_rows, rows_per_cta);
    uint32_t smem = dot_smem_bytes(kind, (int)depth, (int)warps, rows_per_cta);
    if (kind == DotKernel::StagedK && dot_k_x_fits(smem, pass, k))
        smem += (uint32_t)(pass * k);   // the activations, staged in shared memory
    if (smem > 227 * 1024)
        return LOOM_ERR_ARG;
    const uint32_t id = kind == DotKernel::StagedK   ? LOOM_KERNEL_DOT_STAGED_K
                        : kind == DotKernel::StagedB ? LOOM_KERNEL_DOT_STAGED_B
                                                     : LOOM_KERNEL_DOT_DIRECT;
    fill_launch(out, grid, (uint32_t)warps * 32, smem, (uint32_t)rows_per_cta, id);
    return LOOM_OK;
}

// ---- row sums -------------------------------------------------------------

loom_status row_sum_common(const float *values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                           int32_t lanes, const int32_t *counts, int32_t count_scalar,
                           const float *initial, float initial_scalar, int32_t tile,
                           int32_t *final_row, int32_t *tail_count, float *full_sum, float *tail_sum,
                           int32_t *error, const loom_tuning *tuning, void *stream)
{
    if (num_segments < 0 || rows < 0 || (lanes != 1 && lanes != 32) ||
        (int64_t)rows * lanes >= (1ll << 31) || tile < 1 || tile > 64 || seg_stride < 0)
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride < (int64_t)rows * lanes)
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride > 0 && num_segments - 1 > (INT64_MAX - rows * (int64_t)lanes) / seg_stride)
        return LOOM_ERR_SHAPE;
    Tuning t;
    loom_status st = read_tuning(tuning, 0, &t);   // depth 0: the kernel's own default
    if (st != LOOM_OK)
        return st;
    if (num_segments == 0)
        return LOOM_OK;
    if (!values || !final_row || !tail_count || !full_sum || !tail_sum)
        return LOOM_ERR_NULL;
    if (misaligned(values, 4) || misaligned(counts, 4) || misaligned(initial, 4) ||
        misaligned(final_row, 4) || misaligned(tail_count, 4) || misaligned(full_sum, 4) ||
        misaligned(tail_sum, 4) || misaligned(error, 4))
        return LOOM_ERR_ALIGN;

    const bool can_stage = !misaligned(values, 16) && (seg_stride % 4 == 0 || num_segments == 1);
    bool staged;
    if (t.path == LOOM_PATH_STAGED) {
        if (!can_stage)
            return LOOM_ERR_ALIGN;
        staged = true;
    } else if (t.path == LOOM_PATH_DIRECT) {
        staged = false;
    } else {
        staged = can_stage;
    }
    loom_launch L;
    int32_t depth = 0, chunk_bytes = 0;
    st = row_sum_geometry(num_segments, rows, lanes, staged, t.depth, t.upw, t.warps, t.chunk_bytes, &L, &depth,
                          &chunk_bytes);
    if (st != LOOM_OK)
        return st;

    RowSumParams p;
    p.values = values;
    p.num_units = num_segments;
    p.unit_stride = seg_stride;
    p.rows = rows;
    p.lanes = lanes;
    p.tile = tile;
    p.counts = counts;
    p.count_scalar = count_scalar;
    p.initial = initial;
    p.initial_scalar = initial_scalar;
    p.final_row = final_row;
    p.tail_count = tail_count;
    p.full_sum = full_sum;
    p.tail_sum = tail_sum;
    p.error = error;
    p.depth = depth;
    p.units_per_warp = (int32_t)(L.units_per_cta / (L.block[0] / 32));
    p.chunk_elems = chunk_bytes / 4;
    p.wait_ns = t.wait_ns;
    p.inject_stall = t.stall;
    cudaError_t e = launch_row_sum(p, staged, L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LOOM_OK : LOOM_ERR_CUDA;
}

// ---- dequantised dot ------------------------------------------------------

// Workspace of the tensor-core path for n_rows x k on `sms` SMs: enough for
// the persistent grid (one CTA per SM) whatever the schedule.
int64_t dot_workspace_bytes(int64_t n_rows, int64_t k, int64_t sms)
{
    DotTcPlan pl;
    DotTcConfig c{0, 1, 0, 0, 2};   // the split schedule: the largest any schedule needs
    if (n_rows <= 0 || k < 16 || !dot_tc_plan(n_rows, (int32_t)k, sms, c, true, &pl))
        return 0;
    return dot_tc_workspace_bytes(pl);
}

// Argument checks of every dot entry point; *empty is set when there is no work.
loom_status dot_check(const int32_t *w, const float *scale_w, int32_t n_rows, int32_t k, const int32_t *x,
                      const float *scale_x, int32_t batch, const float *y, const int32_t *acc,
                      const int32_t *error, bool *empty)
{
    *empty = false;
    if (n_rows < 0 || batch < 0 || k < 0 || k > MAX_K || (k % 4) != 0)
        return LOOM_ERR_SHAPE;
    if (n_rows == 0 || batch == 0) {
        *empty = true;
        return LOOM_OK;
    }
    if ((k > 0 && (!w || !x)) || !scale_w || !scale_x || !y)  // k == 0 reads no weights
        return LOOM_ERR_NULL;
    if (misaligned(w, 4) || misaligned(scale_w, 4) || misaligned(x, 4) || misaligned(scale_x, 4) ||
        misaligned(y, 4) || misaligned(acc, 4) || misaligned(error, 4))
        return LOOM_ERR_ALIGN;
    return LOOM_OK;
}

loom_status dot_common(const int32_t *w, const float *scale_w, int32_t n_rows, int32_t k,
                       const int32_t *x, const float *scale_x, int32_t batch, float *y, int32_t *acc,
                       void *workspace, int64_t workspace_bytes, int32_t *error,
                       const loom_tuning *tuning, void *stream)
{
    if (n_rows < 0 || batch < 0 || k < 0 || k > MAX_K || (k % 4) != 0)
        return LOOM_ERR_SHAPE;
    Tuning t;
    loom_status st = read_tuning(tuning, 0, &t);   // depth 0: each kernel's own default
    if (st != LOOM_OK)
        return st;
    bool empty = false;
    st = dot_check(w, scale_w, n_rows, k, x, scale_x, batch, y, acc, error, &empty);
    if (st != LOOM_OK || empty)
        return st;
    if (misaligned(workspace, 256))
        return LOOM_ERR_ALIGN;
    if (workspace_bytes < 0 || (workspace && workspace_bytes == 0))
        return LOOM_ERR_ARG;
    const bool can_stage = !misaligned(w, 16) && !misaligned(x, 16) && (k % 16) == 0;
    bool staged;
    int engine = 0;
    if (t.path == LOOM_PATH_STAGED || t.path == LOOM_PATH_TENSOR) {
        if (!can_stage)
            return LOOM_ERR_ALIGN;
        staged = true;
        engine = t.path == LOOM_PATH_TENSOR ? 2 : 1;
    } else if (t.path == LOOM_PATH_DIRECT) {
        staged = false;
        engine = 1;
    } else {
        staged = can_stage;
    }
    const int32_t kw = k / 4;
    int64_t sms = 0;
    if (staged) {
        st = current_sm_count(&sms);   // the tensor-core and lanes-across-k grids are sized by the device
        if (st != LOOM_OK)
            return st;
    }
    const bool split = workspace != nullptr;
    for (int64_t b0 = 0; b0 < batch; b0 += DOT_MAX_BATCH_PER_PASS) {
        const int32_t nb = (int32_t)((batch - b0) < DOT_MAX_BATCH_PER_PASS ? (batch - b0) : DOT_MAX_BATCH_PER_PASS);
        loom_launch L;
        DotTcPlan plan;
        st = dot_geometry(n_rows, k, nb, staged, t.depth, t.warps, t.upw, engine, t.tc, split, sms, &L, &plan);
        if (st != LOOM_OK)
            return st;
        const bool tensor = L.kernel == LOOM_KERNEL_DOT_TENSOR || L.kernel == LOOM_KERNEL_DOT_TENSOR_SPLIT ||
                            L.kernel == LOOM_KERNEL_DOT_TENSOR_ROWS;
        if (tensor && t.tc.schedule == 0 && !dot_tc_cluster_fits(plan)) {
            // the clusters would not all be resident at once: share the units out instead
            DotTcConfig c = t.tc;
            c.schedule = split ? 2 : 1;
            st = dot_geometry(n_rows, k, nb, staged, t.depth, t.warps, t.upw, engine, c, split, sms, &L, &plan);
            if (st != LOOM_OK)
                return st;
        }
        // the first pass is the widest, so a short workspace stops the call before any launch
        if (L.kernel == LOOM_KERNEL_DOT_TENSOR_SPLIT && workspace_bytes < dot_tc_workspace_bytes(plan))
            return LOOM_ERR_ARG;
        const DotKernel kind = tensor ? DotKernel::Tensor : dot_select(staged, k, nb);
        const int depth_used = (int)(t.depth ? t.depth : dot_default_depth(kind));
        DotParams p;
        p.w = w;
        p.scale_w = scale_w;
        p.x = x + (int64_t)b0 * kw;
        p.scale_x = scale_x + b0;
        p.n_rows = n_rows;
        p.k_words = kw;
        p.batch = nb;
        p.y_stride = batch;
        p.y = y + b0;
        p.acc = acc ? acc + b0 : nullptr;
        p.error = error;
        p.depth = depth_used;
        p.rows_per_cta = kind == DotKernel::Tensor ? 0 : (int32_t)L.units_per_cta;
        p.x_in_smem = kind == DotKernel::StagedK &&
                      dot_k_x_fits(dot_smem_bytes(kind, depth_used, (int)(L.block[0] / 32), L.units_per_cta), nb, k);
        p.wait_ns = t.wait_ns;
        p.inject_stall = t.stall;
        p.workspace = workspace;
        p.workspace_bytes = workspace_bytes;
        cudaError_t e = kind == DotKernel::Tensor
                            ? launch_dot_tc(p, plan, static_cast<cudaStream_t>(stream))
                            : launch_dot(p, kind, L, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess)
            return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

// ---- upload of ragged rows ---------------------------------------------------------

loom_status stage_geometry(int64_t num_segments, int64_t rows, int64_t lanes, loom_launch *out)
{
    if (num_segments < 0 || rows < 0 || lanes < 1 || rows * lanes >= (1ll << 31))
        return LOOM_ERR_SHAPE;
    const int64_t per = stage_chunks_per_unit(rows, lanes);
    if (num_segments > 0x7fffffff / per)
        return LOOM_ERR_SHAPE;
    fill_launch(out, num_segments * per, 256, 0, 1, LOOM_KERNEL_STAGE_ROWS);
    return LOOM_OK;
}

// The device can read `p` (device, managed or registered host memory, or any
// host memory where the device has pageable-memory access).
bool device_readable(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type != cudaMemoryTypeUnregistered)
        return true;
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return pageable != 0;
}

// ---- routed row combine ----------------------------------------------------------

loom_status routed_geometry(int64_t tokens, int64_t routes, int64_t rows, int64_t width, bool aligned, int64_t depth,
                            int64_t warps, loom_launch *out)
{
    if (tokens < 0 || routes < 0 || rows < 0 || width < 0 || rows > 0x7fffffff || width > 0x7fffffff ||
        routes > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    if (depth == 0)
        depth = RC_DEFAULT_DEPTH;
    if (warps == 0)
        warps = 2;
    if (depth < 1 || depth > LOOM_MAX_DEPTH || !valid_warps(warps))
        return LOOM_ERR_ARG;
    const bool staged = aligned && width % 4 == 0 && routes <= RC_MAX_STAGED_ROUTES;
    if (ceil_div(tokens, warps) > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    fill_launch(out, ceil_div(tokens, warps), (uint32_t)(32 * warps), routed_smem_bytes(staged, (int)depth, (int)warps),
                (uint32_t)warps, staged ? LOOM_KERNEL_ROUTED_STAGED : LOOM_KERNEL_ROUTED_DIRECT);
    return LOOM_OK;
}

loom_status routed_common(const int32_t *ids, const float *weights, const float *payload, int64_t tokens,
                          int32_t routes, int32_t rows, int32_t width, float *out, int32_t *error,
                          const loom_tuning *tuning, void *stream)
{
    Tuning t;
    loom_status st = read_tuning(tuning, 0, &t);
    if (st != LOOM_OK)
        return st;
    if (t.path == LOOM_PATH_TENSOR)
        return LOOM_ERR_ARG;
    if (tokens < 0 || routes < 0 || rows < 0 || width < 0)
        return LOOM_ERR_SHAPE;
    if (tokens == 0 || width == 0)
        return LOOM_OK;
    if (!out || (routes > 0 && (!ids || !weights)) || (routes > 0 && rows > 0 && !payload))
        return LOOM_ERR_NULL;
    if (misaligned(ids, 4) || misaligned(weights, 4) || misaligned(payload, 4) || misaligned(out, 4) ||
        misaligned(error, 4))
        return LOOM_ERR_ALIGN;
    const bool can_stage = !misaligned(payload, 16) && !misaligned(out, 16) && width % 4 == 0 &&
                           routes <= RC_MAX_STAGED_ROUTES;
    if (t.path == LOOM_PATH_STAGED && !can_stage)
        return (width % 4 != 0 || routes > RC_MAX_STAGED_ROUTES) ? LOOM_ERR_SHAPE : LOOM_ERR_ALIGN;
    const bool staged = can_stage && t.path != LOOM_PATH_DIRECT;
    loom_launch L;
    st = routed_geometry(tokens, routes, rows, width, staged, t.depth, t.warps, &L);
    if (st != LOOM_OK)
        return st;
    RoutedParams p;
    p.ids = ids;
    p.weights = weights;
    p.payload = payload;
    p.out = out;
    p.tokens = tokens;
    p.routes = routes;
    p.rows = rows;
    p.width = width;
    p.error = error;
    p.depth = t.depth ? t.depth : RC_DEFAULT_DEPTH;
    p.wait_ns = t.wait_ns;
    p.inject_stall = t.stall;
    const cudaError_t e = launch_routed(p, L.kernel == LOOM_KERNEL_ROUTED_STAGED, L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

// ---- per-lane f32 sums ------------------------------------------------------------

constexpr int LS_DEFAULT_DEPTH = 2;
constexpr int64_t LS_DEFAULT_CHUNK_BYTES = 4096;

// `aligned`: values 16-byte aligned and segment starts 16-byte apart; the
// staged kernel also needs rows of a multiple of 16 bytes (lanes * width % 4).
loom_status lane_sum_geometry(int64_t num_segments, int64_t rows, int64_t lanes, int64_t width, bool aligned,
                              int64_t depth, int64_t warps, int64_t upw, int64_t chunk_bytes, loom_launch *out,
                              int32_t *chunk_rows)
{
    if (num_segments < 0 || rows < 0 || lanes < 1 || lanes > 32 || (width != 1 && width != 4) ||
        rows * lanes * width >= (1ll << 31))
        return LOOM_ERR_SHAPE;
    if (depth == 0)
        depth = LS_DEFAULT_DEPTH;
    if (warps == 0)
        warps = 1;
    if (chunk_bytes == 0)
        chunk_bytes = LS_DEFAULT_CHUNK_BYTES;
    if (depth < 1 || depth > LOOM_MAX_DEPTH || !valid_warps(warps) || upw < 0 || upw > 32 || !valid_chunk(chunk_bytes))
        return LOOM_ERR_ARG;
    if (upw == 0)
        upw = row_sum_default_units_per_warp((int32_t)rows, (int32_t)(lanes * width));
    const bool staged = aligned && (lanes * width) % 4 == 0;
    // whole rows per chunk (staged rows are a multiple of 16 bytes, so is every chunk)
    const int64_t row_bytes = lanes * width * 4;
    int64_t crow = chunk_bytes / row_bytes;
    if (crow < 1)
        crow = 1;
    const uint32_t smem = lane_sum_smem_bytes(staged, (int)depth, (int)warps, (int)(crow * lanes * width));
    if (smem > 227 * 1024)
        return LOOM_ERR_ARG;
    const int64_t per_cta = warps * upw;
    if (ceil_div(num_segments, per_cta) > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    fill_launch(out, ceil_div(num_segments, per_cta), (uint32_t)(32 * warps), smem, (uint32_t)per_cta,
                staged ? LOOM_KERNEL_LANESUM_STAGED : LOOM_KERNEL_LANESUM_DIRECT);
    if (chunk_rows)
        *chunk_rows = (int32_t)crow;
    return LOOM_OK;
}

loom_status lane_sum_common(const float *values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                            int32_t lanes, int32_t width, bool guarded, const int32_t *counts, int32_t count,
                            int32_t columns, int32_t active_lanes, float *out, int32_t *error,
                            const loom_tuning *tuning, void *stream)
{
    Tuning t;
    loom_status st = read_tuning(tuning, 0, &t);
    if (st != LOOM_OK)
        return st;
    if (t.path == LOOM_PATH_TENSOR)
        return LOOM_ERR_ARG;
    if (num_segments < 0 || rows < 0 || lanes < 1 || lanes > 32 || (width != 1 && width != 4) || seg_stride < 0 ||
        (int64_t)rows * lanes * width >= (1ll << 31))
        return LOOM_ERR_SHAPE;
    if (guarded && (columns < 0 || columns > 4 || active_lanes < 0 || active_lanes > lanes))
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride < (int64_t)rows * lanes * width)
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride > 0 &&
        num_segments - 1 > (INT64_MAX - (int64_t)rows * lanes * width) / seg_stride)
        return LOOM_ERR_SHAPE;
    if (!counts && (count < 0 || count > rows))
        return LOOM_ERR_RANGE;
    if (num_segments == 0)
        return LOOM_OK;
    if (!out || (rows > 0 && !values))
        return LOOM_ERR_NULL;
    if (misaligned(values, 4) || misaligned(counts, 4) || misaligned(out, 4) || misaligned(error, 4))
        return LOOM_ERR_ALIGN;
    const bool can_stage = !misaligned(values, 16) && (seg_stride % 4 == 0 || num_segments == 1) &&
                           (lanes * width) % 4 == 0;
    if (t.path == LOOM_PATH_STAGED && !can_stage)
        return LOOM_ERR_ALIGN;
    const bool staged = can_stage && t.path != LOOM_PATH_DIRECT;
    loom_launch L;
    int32_t crow = 0;
    st = lane_sum_geometry(num_segments, rows, lanes, width, staged, t.depth, t.warps, t.upw, t.chunk_bytes, &L,
                           &crow);
    if (st != LOOM_OK)
        return st;
    LaneSumParams p;
    p.values = values;
    p.num_units = num_segments;
    p.unit_stride = seg_stride;
    p.rows = rows;
    p.lanes = lanes;
    p.counts = counts;
    p.count_scalar = count;
    p.columns = guarded ? columns : width;
    p.active_lanes = guarded ? active_lanes : lanes;
    p.out = out;
    p.error = error;
    p.depth = t.depth ? t.depth : LS_DEFAULT_DEPTH;
    p.units_per_warp = (int32_t)(L.units_per_cta / (L.block[0] / 32));
    p.chunk_rows = crow;
    p.wait_ns = t.wait_ns;
    p.inject_stall = t.stall;
    const cudaError_t e = launch_lane_sum(p, width, guarded, L.kernel == LOOM_KERNEL_LANESUM_STAGED, L,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

// ---- the pages' packed-dot example ------------------------------------------------

// `aligned`: the inputs meet the TMA path's alignment; the staged kernel is
// taken when the shape allows it too (lanes a multiple of 8, <= 64 streams).
// It runs one or two CTAs per SM (as many as their rings allow) over tiles of
// 256 lanes (`sms`: the SM count, 0 = the current device's).
loom_status packed_geometry(int64_t problems, int64_t records, int64_t lanes, int64_t streams, bool aligned,
                            int64_t depth, int64_t rps, int64_t sms, loom_launch *out)
{
    if (problems < 0 || problems > 65535 || records < 0 || lanes < 0 || streams < 1 ||
        ceil_div(lanes, PD_LANES_PER_CTA) > 0x7fffffff)
        return LOOM_ERR_SHAPE;
    if (depth == 0)
        depth = PD_DEFAULT_DEPTH;
    if (rps == 0)
        rps = PD_DEFAULT_RPS;
    if (depth < 1 || depth > LOOM_MAX_DEPTH || rps < 1 || rps > PD_MAX_RPS)
        return LOOM_ERR_ARG;
    const bool staged = aligned && lanes % 8 == 0 && streams <= PD_MAX_STAGED_STREAMS;
    const uint32_t smem = packed_dot_smem_bytes(staged, (int)depth, (int)rps, (int)streams);
    if (smem > 227 * 1024)
        return LOOM_ERR_ARG;
    if (!staged) {
        fill_launch(out, ceil_div(lanes, PD_LANES_PER_CTA), packed_dot_threads(false), 0, PD_LANES_PER_CTA,
                    LOOM_KERNEL_PACKED_DIRECT);
        out->grid[1] = (uint32_t)problems;
        return LOOM_OK;
    }
    if (sms == 0) {
        const loom_status st = current_sm_count(&sms);
        if (st != LOOM_OK)
            return st;
    }
    // as many CTAs per SM as their rings fit, at most seven (the registers of
    // seven CTAs of four consumer warps and a producer)
    int64_t per_sm = (227 * 1024) / ((int64_t)smem + 1024);
    per_sm = per_sm > 7 ? 7 : (per_sm < 1 ? 1 : per_sm);
    const int64_t tiles = packed_dot_tiles(problems, lanes);
    const int64_t grid = tiles < per_sm * sms ? tiles : per_sm * sms;
    // units per CTA: tiles (of 256 lanes of one instance), at most
    fill_launch(out, grid, packed_dot_threads(true), smem, (uint32_t)(grid ? ceil_div(tiles, grid) : 0),
                LOOM_KERNEL_PACKED_STAGED);
    return LOOM_OK;
}

loom_status packed_common(const int32_t *fields, const uint16_t *scales, const float *rhs, int32_t problems,
                          int32_t records, int32_t lanes, int32_t streams, const int32_t *counts, int32_t count,
                          const float *initial, float *out, int32_t *error, const loom_tuning *tuning,
                          void *stream)
{
    Tuning t;
    loom_status st = read_tuning(tuning, 0, &t);
    if (st != LOOM_OK)
        return st;
    if (t.path == LOOM_PATH_TENSOR)
        return LOOM_ERR_ARG;
    if (problems < 0 || problems > 65535 || records < 0 || lanes < 0 || streams < 1)
        return LOOM_ERR_SHAPE;
    if (!counts && (count < 0 || count > records))
        return LOOM_ERR_RANGE;
    if (problems == 0 || lanes == 0)
        return LOOM_OK;   // no outputs: no launch
    if (!out || (records > 0 && (!fields || !scales || !rhs)))
        return LOOM_ERR_NULL;
    if (misaligned(fields, 4) || misaligned(scales, 2) || misaligned(rhs, 4) || misaligned(counts, 4) ||
        misaligned(initial, 4) || misaligned(out, 4) || misaligned(error, 4))
        return LOOM_ERR_ALIGN;
    PackedParams q;
    q.fields = fields;
    q.scales = scales;
    q.rhs = rhs;
    q.problems = problems;
    q.records = records;
    q.lanes = lanes;
    q.streams = streams;
    q.counts = counts;
    q.count = count;
    q.initial = initial;
    q.out = out;
    q.error = error;
    q.wait_ns = t.wait_ns;
    q.inject_stall = t.stall;
    const bool stageable = packed_dot_stageable(q);
    if (t.path == LOOM_PATH_STAGED && !stageable)
        return (lanes % 8 != 0 || streams > PD_MAX_STAGED_STREAMS) ? LOOM_ERR_SHAPE : LOOM_ERR_ALIGN;
    const bool staged = stageable && t.path != LOOM_PATH_DIRECT;
    loom_launch L;
    st = packed_geometry(problems, records, lanes, streams, staged, t.depth, t.upw, 0, &L);
    if (st != LOOM_OK)
        return st;
    q.depth = t.depth ? t.depth : PD_DEFAULT_DEPTH;
    q.rps = t.upw ? t.upw : PD_DEFAULT_RPS;
    const cudaError_t e = launch_packed_dot(q, L.kernel == LOOM_KERNEL_PACKED_STAGED, L,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

// ---- fixed device scratch of loom_i8_dequant_dot_noalloc ---------------------
// One array per device; the streaming kernel writes every record of it that
// the finishing kernel reads, so it needs no initialisation.  8 MiB covers the
// workspace of a grid of one CTA on each of up to 511 SMs.
constexpr int64_t NOALLOC_SCRATCH_BYTES = 8ll << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;

// The scratch address of each device, with the context it was looked up in: a
// context destroyed and created again (cudaDeviceReset) may load the module at
// another address, so the address is looked up again when the context differs.
struct ScratchAddr {
    CUcontext ctx;
    void *addr;
};
std::mutex g_noalloc_mu;
ScratchAddr g_noalloc_addr[NOALLOC_MAX_DEVICES];

using CtxGetCurrent = CUresult (*)(CUcontext *);

CUcontext current_context()
{
    static CtxGetCurrent fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrent>(p);
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS)
        return nullptr;
    return c;
}

// Device address of the scratch array on the current device, looked up with
// cudaGetSymbolAddress once per device and context (the first call on a device
// makes the lookup, which may load the module).
loom_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    ScratchAddr &a = g_noalloc_addr[dev];
    CUcontext ctx = current_context();
    if (ctx && a.ctx == ctx && a.addr) {
        *out = a.addr;
        return LOOM_OK;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    a.ctx = current_context();   // the lookup makes the device's primary context current
    a.addr = p;
    *out = p;
    return LOOM_OK;
}

}  // namespace
}  // namespace loom

using namespace loom;

extern "C" {

#ifdef LOOM_TEST_HOOKS
// Exported by the test build only (declared in csrc/test_hooks.h).
void loom_test_inject_stall(int32_t on) { g_test_stall.store(on != 0, std::memory_order_relaxed); }
#endif

int32_t loom_abi_version(void) { return LOOM_ABI_VERSION; }

const char *loom_status_string(int32_t status)
{
    switch (status) {
    case LOOM_OK:
        return "ok";
    case LOOM_ERR_NULL:
        return "a required pointer is NULL";
    case LOOM_ERR_ALIGN:
        return "a pointer is not aligned as required";
    case LOOM_ERR_SHAPE:
        return "a size, stride or tile is outside the supported range";
    case LOOM_ERR_RANGE:
        return "a count is outside [0, rows]";
    case LOOM_ERR_CUDA:
        return "the CUDA runtime refused the launch";
    case LOOM_ERR_TIMEOUT:
        return "a device wait ran out";
    case LOOM_ERR_ARG:
        return "invalid argument";
    default:
        return "unknown status";
    }
}

loom_status loom_launch_config(loom_op op, const int64_t *workload, int32_t n_workload,
                               loom_launch *out)
{
    if (!workload || !out)
        return LOOM_ERR_NULL;
    auto opt = [&](int i, int64_t dflt) { return n_workload > i ? workload[i] : dflt; };
    switch (op) {
    case LOOM_OP_I8_UNPACK: {
        if (n_workload < 1)
            return LOOM_ERR_ARG;
        if (workload[0] < 0 || ceil_div(workload[0], UNPACK_BLOCK) > 0x7fffffff)
            return LOOM_ERR_SHAPE;
        fill_launch(out, ceil_div(workload[0], UNPACK_BLOCK), UNPACK_BLOCK, 0, UNPACK_BLOCK,
                    LOOM_KERNEL_UNPACK);
        return LOOM_OK;
    }
    case LOOM_OP_FULL_TILE_SUM:
        if (n_workload < 2)
            return LOOM_ERR_ARG;
        return row_sum_geometry(1, workload[0], workload[1], opt(2, 1) != 0,
                                opt(3, 0), 1, opt(4, 0), opt(5, 0), out);
    case LOOM_OP_ROW_SUM_BATCHED:
        if (n_workload < 3)
            return LOOM_ERR_ARG;
        return row_sum_geometry(workload[0], workload[1], workload[2], opt(3, 1) != 0,
                                opt(4, 0), opt(6, 0), opt(5, 0), opt(7, 0), out);
    case LOOM_OP_I8_DEQUANT_DOT: {
        if (n_workload < 3)
            return LOOM_ERR_ARG;
        int64_t sms = opt(9, 0);
        if (sms < 0 || sms > 4096)
            return LOOM_ERR_ARG;
        const bool aligned = opt(3, 1) != 0;
        const DotTcConfig tc{0, (int32_t)opt(10, 0), (int32_t)opt(11, 0), (int32_t)opt(12, 0), (int32_t)opt(13, 0)};
        return dot_geometry(workload[0], workload[1], workload[2], aligned, opt(4, 0), opt(5, 0),
                            opt(6, 0), opt(7, 0), tc, opt(8, 1) != 0, sms, out, nullptr);
    }
    case LOOM_OP_STAGE_ROWS:
        if (n_workload < 3)
            return LOOM_ERR_ARG;
        return stage_geometry(workload[0], workload[1], workload[2], out);
    case LOOM_OP_ROUTED_COMBINE:
        if (n_workload < 4)
            return LOOM_ERR_ARG;
        return routed_geometry(workload[0], workload[1], workload[2], workload[3], opt(4, 1) != 0, opt(5, 0),
                               opt(6, 0), out);
    case LOOM_OP_LANE_SUMS:
        if (n_workload < 4)
            return LOOM_ERR_ARG;
        return lane_sum_geometry(workload[0], workload[1], workload[2], workload[3], opt(4, 1) != 0, opt(5, 0),
                                 opt(6, 0), opt(7, 0), opt(8, 0), out, nullptr);
    case LOOM_OP_PACKED_DOT:
        if (n_workload < 4)
            return LOOM_ERR_ARG;
        return packed_geometry(workload[0], workload[1], workload[2], workload[3], opt(4, 1) != 0, opt(5, 0),
                               opt(6, 0), opt(7, 0), out);
    default:
        return LOOM_ERR_ARG;
    }
}

loom_status loom_full_tile_sum(const float *d_values, int32_t rows, int32_t lanes, int32_t count,
                               float initial, int32_t tile_size, int32_t *d_final_row,
                               int32_t *d_tail_count, float *d_full_sum, float *d_tail_sum, void *stream)
{
    if (rows < 0 || (lanes != 1 && lanes != 32) || (int64_t)rows * lanes >= (1ll << 31) ||
        tile_size < 1 || tile_size > 64)
        return LOOM_ERR_SHAPE;
    if (count < 0 || count > rows)
        return LOOM_ERR_RANGE;
    loom_tuning t = {};
    t.units_per_warp = 1;
    return row_sum_common(d_values, 1, (int64_t)rows * lanes, rows, lanes, nullptr, count, nullptr,
                          initial, tile_size, d_final_row, d_tail_count, d_full_sum, d_tail_sum,
                          nullptr, &t, stream);
}

loom_status loom_row_sum_batched(const float *d_values, int64_t num_segments, int64_t seg_stride,
                                 int32_t rows, int32_t lanes, const int32_t *d_counts,
                                 const float *d_initial, int32_t tile_size, int32_t *d_final_row,
                                 int32_t *d_tail_count, float *d_full_sum, float *d_tail_sum,
                                 int32_t *d_error, void *stream)
{
    return loom_row_sum_batched_ex(d_values, num_segments, seg_stride, rows, lanes, d_counts,
                                   d_initial, tile_size, d_final_row, d_tail_count, d_full_sum,
                                   d_tail_sum, d_error, nullptr, stream);
}

loom_status loom_row_sum_batched_ex(const float *d_values, int64_t num_segments, int64_t seg_stride,
                                    int32_t rows, int32_t lanes, const int32_t *d_counts,
                                    const float *d_initial, int32_t tile_size, int32_t *d_final_row,
                                    int32_t *d_tail_count, float *d_full_sum, float *d_tail_sum,
                                    int32_t *d_error, const loom_tuning *tuning, void *stream)
{
    if (num_segments > 0 && !d_counts)
        return LOOM_ERR_NULL;
    return row_sum_common(d_values, num_segments, seg_stride, rows, lanes, d_counts, 0, d_initial, 0.f,
                          tile_size, d_final_row, d_tail_count, d_full_sum, d_tail_sum, d_error,
                          tuning, stream);
}

loom_status loom_i8_dequant_dot_workspace_bytes(int32_t n_rows, int32_t k, int32_t batch,
                                                int64_t *bytes)
{
    if (!bytes)
        return LOOM_ERR_NULL;
    if (n_rows < 0 || batch < 0 || k < 0 || k > MAX_K || (k % 4) != 0)
        return LOOM_ERR_SHAPE;
    *bytes = 0;
    if (n_rows == 0 || batch < 3 || k < 16 || (k % 16) != 0)
        return LOOM_OK;   // the tensor-core path is not taken
    int64_t sms = 0;
    const loom_status st = current_sm_count(&sms);
    if (st != LOOM_OK)
        return st;
    *bytes = dot_workspace_bytes(n_rows, k, sms);
    return LOOM_OK;
}

loom_status loom_i8_dequant_dot(const int32_t *d_w_packed, const float *d_scale_w, int32_t n_rows,
                                int32_t k, const int32_t *d_x_packed, const float *d_scale_x,
                                int32_t batch, float *d_y, int32_t *d_acc, void *d_workspace,
                                int64_t workspace_bytes, void *stream)
{
    return dot_common(d_w_packed, d_scale_w, n_rows, k, d_x_packed, d_scale_x, batch, d_y, d_acc,
                      d_workspace, workspace_bytes, nullptr, nullptr, stream);
}

loom_status loom_i8_dequant_dot_ex(const int32_t *d_w_packed, const float *d_scale_w, int32_t n_rows,
                                   int32_t k, const int32_t *d_x_packed, const float *d_scale_x,
                                   int32_t batch, float *d_y, int32_t *d_acc, void *d_workspace,
                                   int64_t workspace_bytes, int32_t *d_error,
                                   const loom_tuning *tuning, void *stream)
{
    return dot_common(d_w_packed, d_scale_w, n_rows, k, d_x_packed, d_scale_x, batch, d_y, d_acc,
                      d_workspace, workspace_bytes, d_error, tuning, stream);
}

loom_status loom_i8_dequant_dot_noalloc(const int32_t *d_w_packed, const float *d_scale_w,
                                        int32_t n_rows, int32_t k, const int32_t *d_x_packed,
                                        const float *d_scale_x, int32_t batch, float *d_y,
                                        int32_t *d_acc, void *stream)
{
    bool empty = false;
    loom_status st = dot_check(d_w_packed, d_scale_w, n_rows, k, d_x_packed, d_scale_x, batch, d_y,
                               d_acc, nullptr, &empty);
    if (st != LOOM_OK || empty)
        return st;
    int64_t need = 0;
    st = loom_i8_dequant_dot_workspace_bytes(n_rows, k, batch, &need);
    if (st != LOOM_OK)
        return st;
    if (need > NOALLOC_SCRATCH_BYTES)
        return LOOM_ERR_ARG;   // the grid would outgrow the fixed scratch
    void *scratch = nullptr;
    if (need > 0) {
        st = noalloc_scratch(&scratch);
        if (st != LOOM_OK)
            return st;
    }
    return dot_common(d_w_packed, d_scale_w, n_rows, k, d_x_packed, d_scale_x, batch, d_y, d_acc,
                      scratch, scratch ? NOALLOC_SCRATCH_BYTES : 0, nullptr, nullptr, stream);
}

loom_status loom_packed_dot(const int32_t *d_fields, const uint16_t *d_scales, const float *d_rhs,
                            int32_t problems, int32_t records, int32_t lanes, int32_t streams,
                            const int32_t *d_counts, int32_t count, const float *d_initial, float *d_out,
                            void *stream)
{
    return packed_common(d_fields, d_scales, d_rhs, problems, records, lanes, streams, d_counts, count,
                         d_initial, d_out, nullptr, nullptr, stream);
}

loom_status loom_packed_dot_ex(const int32_t *d_fields, const uint16_t *d_scales, const float *d_rhs,
                               int32_t problems, int32_t records, int32_t lanes, int32_t streams,
                               const int32_t *d_counts, int32_t count, const float *d_initial, float *d_out,
                               int32_t *d_error, const loom_tuning *tuning, void *stream)
{
    return packed_common(d_fields, d_scales, d_rhs, problems, records, lanes, streams, d_counts, count,
                         d_initial, d_out, d_error, tuning, stream);
}

loom_status loom_sum_rows(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                          int32_t lanes, int32_t width, const int32_t *d_counts, int32_t count, float *d_out,
                          void *stream)
{
    return lane_sum_common(d_values, num_segments, seg_stride, rows, lanes, width, false, d_counts, count, 0, 0,
                           d_out, nullptr, nullptr, stream);
}

loom_status loom_sum_rows_ex(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                             int32_t lanes, int32_t width, const int32_t *d_counts, int32_t count, float *d_out,
                             int32_t *d_error, const loom_tuning *tuning, void *stream)
{
    return lane_sum_common(d_values, num_segments, seg_stride, rows, lanes, width, false, d_counts, count, 0, 0,
                           d_out, d_error, tuning, stream);
}

loom_status loom_sum_guarded_rows(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                                  int32_t lanes, const int32_t *d_counts, int32_t count, int32_t columns,
                                  int32_t active_lanes, float *d_out, void *stream)
{
    return lane_sum_common(d_values, num_segments, seg_stride, rows, lanes, 4, true, d_counts, count, columns,
                           active_lanes, d_out, nullptr, nullptr, stream);
}

loom_status loom_sum_guarded_rows_ex(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                                     int32_t lanes, const int32_t *d_counts, int32_t count, int32_t columns,
                                     int32_t active_lanes, float *d_out, int32_t *d_error, const loom_tuning *tuning,
                                     void *stream)
{
    return lane_sum_common(d_values, num_segments, seg_stride, rows, lanes, 4, true, d_counts, count, columns,
                           active_lanes, d_out, d_error, tuning, stream);
}

loom_status loom_routed_combine(const int32_t *d_ids, const float *d_weights, const float *d_payload, int64_t tokens,
                                int32_t routes, int32_t rows, int32_t width, float *d_out, void *stream)
{
    return routed_common(d_ids, d_weights, d_payload, tokens, routes, rows, width, d_out, nullptr, nullptr, stream);
}

loom_status loom_routed_combine_ex(const int32_t *d_ids, const float *d_weights, const float *d_payload,
                                   int64_t tokens, int32_t routes, int32_t rows, int32_t width, float *d_out,
                                   int32_t *d_error, const loom_tuning *tuning, void *stream)
{
    return routed_common(d_ids, d_weights, d_payload, tokens, routes, rows, width, d_out, d_error, tuning, stream);
}

loom_status loom_stage_rows(const float *h_values, float *d_values, int64_t num_segments, int64_t seg_stride,
                            int32_t rows, int32_t lanes, const int32_t *d_counts, int32_t count, void *stream)
{
    if (num_segments < 0 || rows < 0 || lanes < 1 || seg_stride < 0 || (int64_t)rows * lanes >= (1ll << 31))
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride < (int64_t)rows * lanes)
        return LOOM_ERR_SHAPE;
    if (num_segments > 1 && seg_stride > 0 && num_segments - 1 > (INT64_MAX - (int64_t)rows * lanes) / seg_stride)
        return LOOM_ERR_SHAPE;
    if (!d_counts && (count < 0 || count > rows))
        return LOOM_ERR_RANGE;
    loom_launch L;
    loom_status st = stage_geometry(num_segments, rows, lanes, &L);
    if (st != LOOM_OK)
        return st;
    if (num_segments == 0 || rows == 0)
        return LOOM_OK;
    if (!h_values || !d_values)
        return LOOM_ERR_NULL;
    if (misaligned(h_values, 4) || misaligned(d_values, 4) || misaligned(d_counts, 4))
        return LOOM_ERR_ALIGN;
    if (!device_readable(h_values) || (d_counts && !device_readable(d_counts)))
        return LOOM_ERR_ARG;
    StageParams p;
    p.src = h_values;
    p.dst = d_values;
    p.num_units = num_segments;
    p.unit_stride = seg_stride;
    p.chunks_per_unit = stage_chunks_per_unit(rows, lanes);
    p.rows = rows;
    p.lanes = lanes;
    p.counts = d_counts;
    p.count_scalar = count;
    p.vec4 = !misaligned(h_values, 16) && !misaligned(d_values, 16) && (seg_stride % 4 == 0 || num_segments == 1);
    const cudaError_t e = launch_stage_rows(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

loom_status loom_stream_floor(const void *d_src, int64_t bytes, int32_t schedule, int32_t depth,
                              int32_t ctas_per_sm, uint64_t *d_sink, int32_t *d_error, void *stream)
{
    if (bytes < 0 || bytes % 16 != 0)
        return LOOM_ERR_SHAPE;
    const bool loads = schedule == LOOM_FLOOR_GRID_STRIDE || schedule == LOOM_FLOOR_WARP_RANGE;
    if ((!loads && schedule != LOOM_FLOOR_BULK_RING) || (loads && depth != 4 && depth != 8) ||
        (!loads && (depth < 1 || depth > LOOM_MAX_DEPTH)) || ctas_per_sm < 1 || ctas_per_sm > 32)
        return LOOM_ERR_ARG;
    if (!d_sink || (bytes > 0 && !d_src))
        return LOOM_ERR_NULL;
    if (misaligned(d_src, 16) || misaligned(d_sink, 8) || misaligned(d_error, 4))
        return LOOM_ERR_ALIGN;
    if (bytes == 0)
        return LOOM_OK;
    int64_t sms = 0;
    const loom_status st = current_sm_count(&sms);
    if (st != LOOM_OK)
        return st;
    const cudaError_t e = launch_stream_floor(d_src, bytes, schedule, depth, ctas_per_sm, (int32_t)sms, d_sink,
                                              d_error, DEFAULT_WAIT_NS, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LOOM_ERR_CUDA;
    }
    return LOOM_OK;
}

loom_status loom_i8_unpack(const int32_t *d_packed, int64_t n_words, float *d_out, void *stream)
{
    if (n_words < 0)
        return LOOM_ERR_SHAPE;
    loom_launch L;
    const int64_t wl[1] = {n_words};
    loom_status st = loom_launch_config(LOOM_OP_I8_UNPACK, wl, 1, &L);
    if (st != LOOM_OK)
        return st;
    if (n_words == 0)
        return LOOM_OK;
    if (!d_packed || !d_out)
        return LOOM_ERR_NULL;
    if (misaligned(d_packed, 4) || misaligned(d_out, 4))
        return LOOM_ERR_ALIGN;
    cudaError_t e = launch_unpack(d_packed, n_words, d_out, L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LOOM_OK : LOOM_ERR_CUDA;
}

}  // extern "C"
