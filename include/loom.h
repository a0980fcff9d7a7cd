/*
 * loom.h -- C ABI of libloom, a GB300 (sm_103a) library for the streaming
 * reductions described in the Loom documentation pages (ROCm hrx-system):
 *
 *   [P1] "Tune loop unrolling and pipelining"
 *   [P3] "Kernels and launch configuration"
 *
 *  1. the ragged full-tile f32 row sum: a dynamic row count is split into
 *     exact tiles, every full-tile row is reduced across its lanes and added
 *     to a carried sum, and the partial final tile is summed separately
 *     ([P1] "Derive full tiles from a ragged loop");
 *  2. packed signed-byte dequantisation with dot accumulation
 *     ([P1] "Apply the same controls to a packed dot product");
 *  3. the pages' other streaming examples: their own packed dot (f16 record
 *     scales, f32 activations, an ordered f32 sum), per-lane column sums
 *     (sum_rows, sum_vector_rows), guarded ragged rows and the routed row
 *     combine -- each a fixed sequence of f32 operations, defined to the bit;
 *  4. an upload of ragged row-sum inputs that moves only the active rows.
 *
 * Conventions for every entry point
 *  - Pointers prefixed d_ are device pointers owned by the caller; the library
 *    never allocates, frees or retains them and keeps no global mutable state
 *    (two exceptions, documented at their entry points: the fixed scratch of
 *    loom_i8_dequant_dot_noalloc, and a process-wide cache of tensor maps and
 *    device attributes), so calls may be made from several host threads.
 *  - Every kernel is launched as a programmatic dependent of the previous
 *    kernel on the stream and waits for it before touching memory: stream
 *    order holds as for any launch.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; the return value covers argument validation and
 *    the launch only.  Faults found on the device are reported through the
 *    optional error word (LOOM_DEVERR_* bits, atomically OR-ed; the caller
 *    zeroes it) and, for results that could not be computed, NaN outputs.
 *  - Empty work (no segments, no rows, empty batch) returns LOOM_OK and
 *    launches nothing.
 *  - Results do not depend on the read-ahead depth, the stream or earlier
 *    calls: the same inputs give the same bits.
 */
#ifndef LOOM_H
#define LOOM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LOOM_ABI_VERSION 4

typedef enum loom_status {
    LOOM_OK = 0,
    LOOM_ERR_NULL = -1,    /* a required pointer is NULL */
    LOOM_ERR_ALIGN = -2,   /* a pointer is not aligned to its element size */
    LOOM_ERR_SHAPE = -3,   /* a size, stride or tile is outside the supported range */
    LOOM_ERR_RANGE = -4,   /* a host-side count is outside [0, rows] */
    LOOM_ERR_CUDA = -5,    /* the CUDA runtime refused the launch */
    LOOM_ERR_TIMEOUT = -6, /* a device wait ran out (reported via the error word) */
    LOOM_ERR_ARG = -7      /* any other invalid argument (unknown op, bad tuning) */
} loom_status;

/* Bits of the device error word. */
#define LOOM_DEVERR_COUNT_RANGE 0x1 /* a device count was outside [0, rows]; clamped */
#define LOOM_DEVERR_TIMEOUT 0x2     /* a staged copy did not land in time; NaN results */

typedef enum loom_op {
    LOOM_OP_I8_UNPACK = 0,       /* workload {n_words} */
    LOOM_OP_FULL_TILE_SUM = 1,   /* workload {rows, lanes, staged (0/1), depth, warps_per_cta,
                                    chunk_bytes} */
    LOOM_OP_ROW_SUM_BATCHED = 2, /* workload {num_segments, rows, lanes, staged (0/1), depth,
                                    warps_per_cta, units_per_warp, chunk_bytes} */
    LOOM_OP_I8_DEQUANT_DOT = 3,  /* workload {n_rows, k, batch, staged (0/1), depth,
                                    warps_per_cta, ctas_per_sm (batch <= 2 kernel), engine (0 auto, 1 dp4a,
                                    2 tensor), workspace (0/1, default 1), sm_count (0 =
                                    the current device), tc_units_per_stage,
                                    tc_a_buffers, tc_pipelines, tc_schedule} */
    LOOM_OP_PACKED_DOT = 4,      /* workload {problems, records, lanes, streams, aligned (0/1:
                                    inputs 16-byte aligned, default 1), depth,
                                    records_per_stage, sm_count (0 = the current device)} */
    LOOM_OP_LANE_SUMS = 5,       /* workload {num_segments, rows, lanes, width (1 or 4), aligned
                                    (0/1, default 1), depth, warps_per_cta, units_per_warp,
                                    chunk_bytes}; also the guarded rows (width 4) */
    LOOM_OP_ROUTED_COMBINE = 6,  /* workload {tokens, routes, rows, width, aligned (0/1, default
                                    1), depth, warps_per_cta} */
    LOOM_OP_STAGE_ROWS = 7       /* workload {num_segments, rows, lanes} */
} loom_op;

/* Launch geometry of one kernel launch.  `units_per_cta` logical work units
 * (words, segments or output rows) map onto each CTA; the grid is the
 * ceiling division of the workload by it, and units past the workload in the
 * last CTA do no loads and no stores.  The tensor-core dot runs one CTA per
 * SM instead: with few 128-row bands, a cluster of cluster[0] CTAs per band
 * (each an equal share of the band's 128-k units); otherwise min(work units,
 * SMs) CTAs, each an equal contiguous share -- at most units_per_cta -- of the
 * list of 128-row x 128-k weight units (of whole bands without a workspace). */
typedef struct loom_launch {
    uint32_t grid[3];
    uint32_t block[3];
    uint32_t cluster[3];    /* {1,1,1}, or {C,1,1} when the tensor-core dot gives each band a
                               cluster of C CTAs */
    uint32_t subgroup_size; /* 32 */
    uint32_t smem_bytes;    /* dynamic shared memory per CTA */
    uint32_t units_per_cta;
    uint32_t kernel;        /* LOOM_KERNEL_* selected for this workload */
} loom_launch;

#define LOOM_KERNEL_UNPACK 1
#define LOOM_KERNEL_ROWSUM_STAGED 2 /* bulk-copy read-ahead ring per warp */
#define LOOM_KERNEL_ROWSUM_DIRECT 3 /* plain loads (unaligned inputs) */
#define LOOM_KERNEL_DOT_STAGED_K 4  /* lanes across k, batch <= 2: a block of rows per CTA (units_per_cta =
                                       rows), its 8 KiB row pieces shared out evenly over the warps */
#define LOOM_KERNEL_DOT_STAGED_B 5  /* lanes across the batch, batch > 2 */
#define LOOM_KERNEL_DOT_DIRECT 6    /* plain loads (unaligned or k % 16 != 0) */
#define LOOM_KERNEL_DOT_TENSOR 7    /* tcgen05 MMA on exact f16 copies, batch 3..16 per pass;
                                       one CTA per SM, a cluster per band or whole bands */
#define LOOM_KERNEL_DOT_TENSOR_SPLIT 8 /* the same kernel over equal shares of all units, then
                                          a finishing kernel for the bands split between CTAs
                                          (two launches per pass) */
#define LOOM_KERNEL_PACKED_STAGED 9  /* packed dot: up to seven CTAs per SM (as many as
                                        their rings fit) over tiles of 256 lanes, two lanes per
                                        consumer thread (units_per_cta = tiles), one 3-D TMA
                                        read-ahead ring per CTA */
#define LOOM_KERNEL_PACKED_DIRECT 10 /* packed dot: plain loads */
#define LOOM_KERNEL_LANESUM_STAGED 11 /* per-lane sums: bulk-copy read-ahead ring per warp */
#define LOOM_KERNEL_LANESUM_DIRECT 12 /* per-lane sums: plain loads */
#define LOOM_KERNEL_ROUTED_STAGED 13  /* routed combine: bulk-copy ring of payload pieces per warp */
#define LOOM_KERNEL_ROUTED_DIRECT 14  /* routed combine: plain loads */
#define LOOM_KERNEL_STAGE_ROWS 15     /* upload of ragged rows: one CTA per 8 KiB of a segment */
#define LOOM_KERNEL_ROWSUM_SEGMENTS 17 /* 32-lane segments that fit the ring (128 x rows <=
                                          chunk_bytes, default 8 KiB): one bulk copy and one wait
                                          per segment, whole segments back to back in a byte ring
                                          per warp, up to `depth` in flight; the same bits as
                                          LOOM_KERNEL_ROWSUM_STAGED */
#define LOOM_KERNEL_DOT_TENSOR_ROWS 16 /* tcgen05 MMA on exact f16 copies, batch 3..16 per pass; one
                                          CTA per SM owning whole rows (units_per_cta = rows),
                                          two k ranges per MMA; one launch, no workspace */

/* Maximum read-ahead depth (staged chunks in flight per warp or CTA). */
#define LOOM_MAX_DEPTH 8

/*
 * Host launch-configuration routine: maps a workload to a launch without
 * touching the device (the tensor-core dot reads the SM count of the current
 * device unless the workload gives one).  [P3] "A kernel owns two signatures" and "Workload is
 * not workgroup count": the workload scalars alone determine the grid by
 * ceiling division; for LOOM_OP_I8_UNPACK 1009 words give 4 CTAs of 256.
 * `workload` holds `n_workload` scalars as listed for each loom_op; trailing
 * optional entries may be left out: staged defaults to 1, the schedule
 * entries (depth, warps_per_cta, units/rows per warp, chunk_bytes) to the
 * library's defaults (also selected by 0).
 * Errors: NULL out/workload -> LOOM_ERR_NULL; unknown op or too few entries
 * -> LOOM_ERR_ARG; negative or unsupported sizes -> LOOM_ERR_SHAPE.
 */
loom_status loom_launch_config(loom_op op, const int64_t *workload, int32_t n_workload,
                               loom_launch *out);

/*
 * One segment.  [P1] "Derive full tiles from a ragged loop": with
 * F = tile_size * floor(count / tile_size) and t = count - F,
 *   *d_final_row  = F,  *d_tail_count = t,
 *   *d_full_sum   = initial + sum over rows r < F, lanes l of values[r][l],
 *   *d_tail_sum   = sum over rows F <= r < count, lanes l of values[r][l].
 * d_values: f32 [rows][lanes], row-major, contiguous, 4-byte aligned
 * (16-byte alignment selects the bulk-copy path; it is never required).
 * Sums are accumulated without rounding loss (error-free double-word f32)
 * and rounded once, so they are within one f32 rounding of the exact sum.
 * Errors: NULL -> LOOM_ERR_NULL; misaligned -> LOOM_ERR_ALIGN; rows < 0,
 * lanes not 1 or 32, tile_size outside [1, 64], rows*lanes >= 2^31 ->
 * LOOM_ERR_SHAPE; count outside [0, rows] -> LOOM_ERR_RANGE.
 */
loom_status loom_full_tile_sum(const float *d_values, int32_t rows, int32_t lanes, int32_t count,
                               float initial, int32_t tile_size, int32_t *d_final_row,
                               int32_t *d_tail_count, float *d_full_sum, float *d_tail_sum,
                               void *stream);

/*
 * num_segments independent segments, each exactly loom_full_tile_sum above.
 * Segment s holds f32 [rows][lanes] at d_values + s * seg_stride (elements);
 * its count is d_counts[s] and its initial sum d_initial[s] (0 when
 * d_initial is NULL).  Outputs are four arrays of num_segments entries
 * (structure of arrays).  Wide ragged rows are the case lanes = 1: each row
 * is a segment of `rows` one-lane records with its active length as count.
 * A device count outside [0, rows] is clamped into range and sets
 * LOOM_DEVERR_COUNT_RANGE in *d_error (d_error may be NULL).
 * Errors: as loom_full_tile_sum, plus seg_stride < rows*lanes (when
 * num_segments > 1) or num_segments < 0 -> LOOM_ERR_SHAPE.
 */
loom_status loom_row_sum_batched(const float *d_values, int64_t num_segments, int64_t seg_stride,
                                 int32_t rows, int32_t lanes, const int32_t *d_counts,
                                 const float *d_initial, int32_t tile_size, int32_t *d_final_row,
                                 int32_t *d_tail_count, float *d_full_sum, float *d_tail_sum,
                                 int32_t *d_error, void *stream);

/*
 * Dequantised dot products.  [P1] "Apply the same controls to a packed dot
 * product": packed words are unpacked into signed bytes and accumulated as a
 * dot product; here every weight row r has scale d_scale_w[r] and every
 * activation vector b has scale d_scale_x[b]:
 *   acc[r][b] = sum_k W[r][k] * X[b][k]                  (int32, exact)
 *   y[r][b]   = (float)acc[r][b] * (d_scale_w[r] * d_scale_x[b])   (f32)
 * d_w_packed: int32 [n_rows][k/4]; d_x_packed: int32 [batch][k/4].  Word j
 * of a row holds elements 4j..4j+3, element 4j+i in bits [8i, 8i+7] as a
 * signed byte (the little-endian int8 array viewed as int32 words).
 * d_y: f32 [n_rows][batch]; d_acc: int32 [n_rows][batch] or NULL.
 * d_workspace / workspace_bytes: see loom_i8_dequant_dot_workspace_bytes
 * (NULL / 0 is always valid).
 * Errors: NULL -> LOOM_ERR_NULL; misaligned (the workspace: to 256 bytes) ->
 * LOOM_ERR_ALIGN; k % 4 != 0, k > 131068 (|acc| must stay below 2^31) or
 * negative sizes -> LOOM_ERR_SHAPE; a workspace shorter than its query ->
 * LOOM_ERR_ARG.
 */
loom_status loom_i8_dequant_dot(const int32_t *d_w_packed, const float *d_scale_w, int32_t n_rows,
                                int32_t k, const int32_t *d_x_packed, const float *d_scale_x,
                                int32_t batch, float *d_y, int32_t *d_acc, void *d_workspace,
                                int64_t workspace_bytes, void *stream);

/*
 * Bytes of the workspace that lets loom_i8_dequant_dot split 128-row bands
 * of W between CTAs that are not in one cluster, on the current device (0
 * when the tensor-core kernel is not taken: batch < 3, k < 16 or k % 16 !=
 * 0).  It is the most any schedule uses; with few bands the call gives each
 * band a cluster of CTAs and uses none of it.  The size grows with the CTAs
 * of the launch, at most one per SM, so the query for the largest problem
 * (n_rows = INT32_MAX) gives a workspace that serves every call on the device.  With many bands, splitting
 * spreads the weights evenly over the SMs; without a workspace each CTA then
 * takes whole bands.
 * The workspace (d_workspace, caller-owned device memory, 256-byte aligned,
 * any contents) holds the partial sums of the split bands between the
 * streaming kernel and a second, finishing kernel that the call launches
 * after it on the same stream.  Calls that may run at the same time (other
 * streams, other host threads) must not share one workspace.
 * workspace_bytes smaller than this size -> LOOM_ERR_ARG; d_workspace NULL ->
 * no split (one launch).
 * Errors: NULL bytes -> LOOM_ERR_NULL; sizes as for loom_i8_dequant_dot ->
 * LOOM_ERR_SHAPE; no usable device -> LOOM_ERR_CUDA.
 */
loom_status loom_i8_dequant_dot_workspace_bytes(int32_t n_rows, int32_t k, int32_t batch,
                                                int64_t *bytes);

/*
 * loom_i8_dequant_dot without a caller workspace and without any device
 * allocation.  The Loom pages have no counterpart of this entry point: it is
 * a deployment variant of the call above.  The bands of W are split between
 * CTAs through scratch that the library holds in a fixed device array (8 MiB
 * on each device that loads the library, held until the process exits);
 * results are the same bits as loom_i8_dequant_dot.  The first call on a
 * device (and again after its context has been re-created) looks up the
 * array's device address with cudaGetSymbolAddress, which may load the
 * module: make that first call before any stream capture.  The scratch is
 * shared by every call on a device, so calls that may run at the same time
 * (other streams, other host threads) must be serialised by the caller.
 * Errors: as loom_i8_dequant_dot; a problem whose split workspace would not
 * fit the fixed scratch -> LOOM_ERR_ARG; no usable device -> LOOM_ERR_CUDA.
 */
loom_status loom_i8_dequant_dot_noalloc(const int32_t *d_w_packed, const float *d_scale_w,
                                        int32_t n_rows, int32_t k, const int32_t *d_x_packed,
                                        const float *d_scale_x, int32_t batch, float *d_y,
                                        int32_t *d_acc, void *stream);

/*
 * The packed signed-byte dot of the pages' streaming example, for `problems`
 * independent instances (the pages time one instance per dispatch over many
 * dispatches; here one call takes them all).
 * [P1] "Apply the same controls to a packed dot product": lane l of an
 * instance owns one output.  For every record r < count it reads the packed
 * word fields[r][l] (four signed bytes, element j = bits 8j..8j+7), the f16
 * scale scales[r][l] and four f32 activations rhs[r][l mod streams][0..3];
 * the bytes become f32, are multiplied by the scale, and the dot product
 * with the activations advances the lane's f32 sum in record order.  Each of
 * the four products enters the sum as one fused multiply-add, in element
 * order (the reading taken of the pages' ordered dot step), so the result is
 * defined to the bit.  The sum starts from d_initial (or 0).
 * Layout (caller-owned device memory, row-major): d_fields int32
 * [problems][records][lanes]; d_scales f16 bit patterns [problems][records]
 * [lanes]; d_rhs f32 [problems][records][streams][4]; d_counts int32
 * [problems] (NULL: `count` for every instance); d_initial f32
 * [problems][lanes] (NULL: 0); d_out f32 [problems][lanes].
 * Schedule: with lanes a multiple of 8, at most 64 streams and 16-byte
 * aligned inputs, CTAs (up to seven per SM) walk tiles of 256 lanes of one
 * instance, two lanes per thread, fed by one read-ahead ring of 3-D TMA copies
 * per CTA; else 256 lanes per CTA with plain loads (same bits).
 * Errors: NULL required pointer -> LOOM_ERR_NULL; pointers not 4-byte (fields,
 * rhs, initial, out) or 2-byte (scales) aligned -> LOOM_ERR_ALIGN; negative
 * sizes, streams < 1, or more than 65535 instances -> LOOM_ERR_SHAPE; host
 * count outside [0, records] -> LOOM_ERR_RANGE.  Device counts outside
 * [0, records] are clamped and flagged (LOOM_DEVERR_COUNT_RANGE, _ex only).
 */
loom_status loom_packed_dot(const int32_t *d_fields, const uint16_t *d_scales, const float *d_rhs,
                            int32_t problems, int32_t records, int32_t lanes, int32_t streams,
                            const int32_t *d_counts, int32_t count, const float *d_initial,
                            float *d_out, void *stream);

/*
 * Per-lane f32 sums of independent segments: the pages' sum_rows (width 1)
 * and sum_vector_rows (width 4).
 * [P1] "Keep one checked source for experiments": work-item `lane` sums its
 * column of rows [0, count), an f32 carried sum from zero, one row per trip
 * in row order (the pages' check cases print the expected sums for an iota
 * input).  [P1] "Give each motif its own schedule": each row holds a
 * four-element vector per lane, reduced into the carried sum one element at
 * a time in element order (the reading taken).  The results are defined to
 * the bit.
 * Layout: segment s at d_values + s * seg_stride, rows x lanes x width f32
 * row-major (lanes 1..32); d_counts int32 [num_segments] (NULL: `count` for
 * all); d_out f32 [num_segments][lanes].  One warp per segment, its active
 * rows streamed through a ring of bulk copies (16-byte aligned values and
 * segment starts, lanes * width a multiple of 4), else plain loads.
 * Errors: NULL -> LOOM_ERR_NULL; pointers not 4-byte aligned ->
 * LOOM_ERR_ALIGN; bad sizes or strides -> LOOM_ERR_SHAPE; host count outside
 * [0, rows] -> LOOM_ERR_RANGE.  Device counts outside [0, rows] are clamped.
 */
loom_status loom_sum_rows(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                          int32_t lanes, int32_t width, const int32_t *d_counts, int32_t count, float *d_out,
                          void *stream);

/*
 * Guarded ragged rows of independent segments: the pages' sum_guarded_rows.
 * [P1] "Keep guards and inner loops in the source": the row range is
 * rounded up to a multiple of four; each trip adds to the lane's f32 carried
 * sum the identity for a row at or past the count (such rows are never
 * read), else the f32 sum from zero of the row's first `columns` (0..4)
 * components, each of them the identity on lanes at or past `active_lanes`.
 * Layout: segment s at d_values + s * seg_stride, rows x lanes x 4 f32;
 * d_counts / count, d_out and errors as loom_sum_rows; columns outside
 * [0, 4] or active_lanes outside [0, lanes] -> LOOM_ERR_SHAPE.
 */
loom_status loom_sum_guarded_rows(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                                  int32_t lanes, const int32_t *d_counts, int32_t count, int32_t columns,
                                  int32_t active_lanes, float *d_out, void *stream);

/*
 * Routed row combine (a mixture-of-experts combine).
 * [P1] "Separate route and payload lookahead": for each token the routes are
 * visited in order; route r's row id selects a row of d_payload; a missing
 * id (negative) suppresses the route's weight and payload reads and leaves
 * the sum unchanged; otherwise every element of the selected row is
 * multiplied by the route's weight (one f32 product) and added to the
 * token's f32 sum (one f32 addition), which starts at zero.  Product and sum
 * are rounded separately (the reading taken), so the result is defined to
 * the bit.
 * Layout (caller-owned device memory): d_ids int32 and d_weights f32
 * [tokens][routes]; d_payload f32 [rows][width]; d_out f32 [tokens][width].
 * One warp per token; its ids are read once, then its valid routes' row
 * pieces stream through a ring of bulk copies (width a multiple of 4,
 * 16-byte aligned payload and output, at most 32 routes), else plain loads.
 * Errors: NULL -> LOOM_ERR_NULL; pointers not 4-byte aligned ->
 * LOOM_ERR_ALIGN; negative sizes -> LOOM_ERR_SHAPE.  Ids at or past `rows`
 * are treated as missing and flagged (LOOM_DEVERR_COUNT_RANGE, _ex only).
 */
loom_status loom_routed_combine(const int32_t *d_ids, const float *d_weights, const float *d_payload, int64_t tokens,
                                int32_t routes, int32_t rows, int32_t width, float *d_out, void *stream);

/*
 * Upload of ragged row-sum inputs: only the rows the row sums read.  For each
 * segment s, elements [0, count_s * lanes) at h_values + s * seg_stride are
 * copied to the same offsets of d_values; the rest of d_values is not
 * touched.  The pages have no counterpart (their inputs start on the
 * device): the bytes past a segment's count are not inputs of the row sums,
 * and on GB300 the SMs read host memory in place over the host link, so the
 * upload moves only the active prefix of every segment.
 * h_values: memory the device can read -- pinned host memory (cudaHostAlloc,
 * cudaMallocHost, cudaHostRegister), device memory, or any host memory where
 * the device has pageable-memory access; d_values: device memory; d_counts:
 * int32 [num_segments] readable by the device, or NULL (`count` for every
 * segment); counts are clamped to [0, rows].  Asynchronous on `stream`.
 * Errors: NULL -> LOOM_ERR_NULL; pointers not 4-byte aligned ->
 * LOOM_ERR_ALIGN; bad sizes or strides -> LOOM_ERR_SHAPE; host count outside
 * [0, rows] -> LOOM_ERR_RANGE; memory the device cannot read -> LOOM_ERR_ARG.
 */
loom_status loom_stage_rows(const float *h_values, float *d_values, int64_t num_segments, int64_t seg_stride,
                            int32_t rows, int32_t lanes, const int32_t *d_counts, int32_t count, void *stream);

/*
 * Unpack and convert: d_out[4j + i] = (float) signed byte i of d_packed[j].
 * [P1] "Apply the same controls to a packed dot product" (bit-unpack into
 * four 8-bit integers, then signed integer to float).  One thread per word,
 * 256-thread CTAs, grid = ceil(n_words / 256) ([P3] "Over-dispatch safely").
 * Errors: NULL -> LOOM_ERR_NULL; misaligned -> LOOM_ERR_ALIGN;
 * n_words < 0 -> LOOM_ERR_SHAPE.
 */
loom_status loom_i8_unpack(const int32_t *d_packed, int64_t n_words, float *d_out, void *stream);

/* Static description of a status code (never NULL). */
const char *loom_status_string(int32_t status);

/* LOOM_ABI_VERSION of the loaded library. */
int32_t loom_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LOOM_H */
