/*
 * loom_tuning.h -- schedule controls and test hooks of libloom.
 *
 * The _ex entry points take the same arguments as their plain counterparts
 * in loom.h, plus a device error word and an optional loom_tuning.  They
 * exist for schedule experiments (read-ahead depth, serial control, plain
 * loads) and for the limit of device waits; none of these controls changes a
 * result.
 * [P1] = "Tune loop unrolling and pipelining" (Loom pages): the depth is the
 * read-ahead depth of its pipeline(depth) ("Separate depth from unrolling"),
 * depth 1 being the serial control.
 */
#ifndef LOOM_TUNING_H
#define LOOM_TUNING_H

#include "loom.h"

#ifdef __cplusplus
extern "C" {
#endif

#define LOOM_PATH_AUTO 0   /* staged when inputs are 16-byte aligned, else direct; dot:
                              tensor cores for 3..16 vectors when k allows */
#define LOOM_PATH_STAGED 1 /* bulk-copy read-ahead ring (dot: dp4a kernels only);
                              LOOM_ERR_ALIGN if not possible */
#define LOOM_PATH_DIRECT 2 /* plain loads, no shared-memory staging */
#define LOOM_PATH_TENSOR 3 /* dot only: the tensor-core kernel for every batch pass;
                              LOOM_ERR_ALIGN / LOOM_ERR_SHAPE when not possible */

typedef struct loom_tuning {
    int32_t depth;          /* staged chunks in flight per warp (per CTA for the tensor-core
                               dot), 1..LOOM_MAX_DEPTH; 0 = default */
    int32_t path;           /* LOOM_PATH_* */
    int32_t units_per_warp; /* row sums: segments per warp, 1..32; dot: CTAs per SM of
                               the batch <= 2 kernel, 1..32 (its rows are spread over
                               that many CTAs on every SM); 0 = default */
    int32_t warps_per_cta;  /* 1, 2, 4 or 8; 0 = default */
    int32_t chunk_bytes;    /* row sums: bytes per staged chunk, a multiple of 512 in
                               [512, 32768]; 0 = default */
    int64_t wait_ns;        /* limit of each device wait in ns; 0 = default (1 s).  A wait
                               that runs out ends the kernel with NaN results and
                               LOOM_DEVERR_TIMEOUT in the error word; the device stays usable */
    /* tensor-core dot schedule (depth above = its shared-memory stages) */
    int32_t tc_units_per_stage; /* 128-k weight units per stage, 1 .. converter groups of a
                                   pipeline; 0 = default (one per group) */
    int32_t tc_a_buffers;       /* f16 A buffers per pipeline in tensor memory, at least twice
                                   the converter groups less one; 0 = default (that minimum);
                                   the rest of the pipeline's columns hold accumulators */
    int32_t tc_pipelines;       /* pipelines per CTA (one CTA per SM): 1 (four converter groups,
                                   all 512 tensor-memory columns) or 2 (two groups and 256
                                   columns each, the halves of the CTA's units); 0 = 2 */
    int32_t tc_schedule;        /* how rows of W map onto CTAs: 0 choose; 1 whole 128-row
                                   bands per CTA; 2 equal shares of all units, split bands
                                   finished by a second kernel (needs the workspace, else
                                   LOOM_ERR_ARG); 3 a cluster of CTAs per band (when the SMs
                                   allow at least two per band, else as 1); 4 ceil(n_rows /
                                   SMs) whole rows per CTA, in blocks of up to 64 (depth even,
                                   2..8; tc_a_buffers 2 or 3; tc_units_per_stage 0 or 1 and
                                   tc_pipelines 0 or 2, else LOOM_ERR_ARG).  Choosing takes 4
                                   where blocks hold 32 rows or more and k >= 2048 */
} loom_tuning;

/* loom_row_sum_batched with tuning (NULL = defaults).  Extra errors:
 * out-of-range tuning -> LOOM_ERR_ARG; LOOM_PATH_STAGED on unaligned input
 * -> LOOM_ERR_ALIGN. */
loom_status loom_row_sum_batched_ex(const float *d_values, int64_t num_segments,
                                    int64_t seg_stride, int32_t rows, int32_t lanes,
                                    const int32_t *d_counts, const float *d_initial,
                                    int32_t tile_size, int32_t *d_final_row, int32_t *d_tail_count,
                                    float *d_full_sum, float *d_tail_sum, int32_t *d_error,
                                    const loom_tuning *tuning, void *stream);

/* loom_i8_dequant_dot with a device error word (may be NULL) and tuning.
 * Extra errors: a tensor-core schedule that does not fit (shared or tensor
 * memory) -> LOOM_ERR_ARG. */
loom_status loom_i8_dequant_dot_ex(const int32_t *d_w_packed, const float *d_scale_w,
                                   int32_t n_rows, int32_t k, const int32_t *d_x_packed,
                                   const float *d_scale_x, int32_t batch, float *d_y,
                                   int32_t *d_acc, void *d_workspace, int64_t workspace_bytes,
                                   int32_t *d_error, const loom_tuning *tuning, void *stream);

/* loom_packed_dot with tuning (NULL = defaults): depth = stages of the read-ahead
 * ring (1 = the serial control), units_per_warp = records per stage (1..32),
 * path = LOOM_PATH_STAGED / LOOM_PATH_DIRECT to force one (LOOM_ERR_ALIGN or
 * LOOM_ERR_SHAPE when the staged path cannot take the inputs).  Extra errors:
 * a tuning value out of range -> LOOM_ERR_ARG. */
loom_status loom_packed_dot_ex(const int32_t *d_fields, const uint16_t *d_scales, const float *d_rhs,
                               int32_t problems, int32_t records, int32_t lanes, int32_t streams,
                               const int32_t *d_counts, int32_t count, const float *d_initial,
                               float *d_out, int32_t *d_error, const loom_tuning *tuning, void *stream);

/* loom_sum_rows and loom_sum_guarded_rows with tuning (NULL = defaults): depth,
 * warps_per_cta, units_per_warp (segments per warp), chunk_bytes and path as for
 * the row sums; d_error gets LOOM_DEVERR_* bits. */
loom_status loom_sum_rows_ex(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                             int32_t lanes, int32_t width, const int32_t *d_counts, int32_t count, float *d_out,
                             int32_t *d_error, const loom_tuning *tuning, void *stream);
loom_status loom_sum_guarded_rows_ex(const float *d_values, int64_t num_segments, int64_t seg_stride, int32_t rows,
                                     int32_t lanes, const int32_t *d_counts, int32_t count, int32_t columns,
                                     int32_t active_lanes, float *d_out, int32_t *d_error, const loom_tuning *tuning,
                                     void *stream);

/* loom_routed_combine with tuning (NULL = defaults): depth = row pieces in flight per
 * warp, warps_per_cta, path (LOOM_PATH_STAGED on inputs it cannot take ->
 * LOOM_ERR_SHAPE / LOOM_ERR_ALIGN); d_error gets LOOM_DEVERR_* bits. */
loom_status loom_routed_combine_ex(const int32_t *d_ids, const float *d_weights, const float *d_payload,
                                   int64_t tokens, int32_t routes, int32_t rows, int32_t width, float *d_out,
                                   int32_t *d_error, const loom_tuning *tuning, void *stream);

/* Schedules of loom_stream_floor. */
#define LOOM_FLOOR_GRID_STRIDE 0 /* grid-stride 16-byte loads, `depth` (4 or 8) in flight per thread */
#define LOOM_FLOOR_WARP_RANGE 1  /* one contiguous range per warp, 16-byte loads, `depth` (4 or 8) in
                                    flight per lane */
#define LOOM_FLOOR_BULK_RING 2   /* one warp per CTA, a ring of `depth` (1..8) 8 KiB stages filled by
                                    bulk copies */

/* Measurement probe, not a step of the method: one launch that reads `bytes`
 * of device memory at d_src once (16-byte loads or bulk copies) and keeps
 * nothing of it.  Its time is what one launch that
 * moves that many bytes takes on this device -- launch, ramp and tail
 * included -- and is the reference each kernel's single-launch time is set
 * against.  `ctas_per_sm` (1..32) CTAs per SM of the current device, 256
 * threads each (32 for LOOM_FLOOR_BULK_RING).  d_sink: a device word that is
 * written only when the checksum of the loaded words equals a fixed constant
 * (so that no load can be dropped); d_error (may be NULL) gets
 * LOOM_DEVERR_TIMEOUT if a bulk copy did not land within the default wait.
 * Errors: NULL d_sink or d_src (bytes > 0) -> LOOM_ERR_NULL; d_src not 16-byte
 * or d_sink not 8-byte aligned -> LOOM_ERR_ALIGN; bytes < 0 or not a multiple
 * of 16 -> LOOM_ERR_SHAPE; unknown schedule, depth or ctas_per_sm ->
 * LOOM_ERR_ARG. */
loom_status loom_stream_floor(const void *d_src, int64_t bytes, int32_t schedule, int32_t depth,
                              int32_t ctas_per_sm, uint64_t *d_sink, int32_t *d_error, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LOOM_TUNING_H */
