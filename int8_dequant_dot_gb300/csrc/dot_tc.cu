// dot_tc.cu -- batched dequantised dot products on the 5th-generation tensor
// cores (tcgen05, sm_103a).
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section "Apply
// the same controls to a packed dot product"): packed signed bytes are
// unpacked and accumulated as dot products; here weights W[n_rows][k] and up
// to 16 activation vectors X[b][k], int32 accumulation, per-row and
// per-vector scales in the epilogue.
//
// Design
//  * The product is a skinny GEMM D[128 x 16] += A[128 x 16] * B[16 x 16]^T
//    per instruction (tcgen05.mma kind::f16, M = 128, N = 16, K = 16).
//    int8 has no fast tensor path on sm_103a, but every int8 value is exact
//    in f16, every product of two is exact in the f32 accumulator, and a sum
//    of at most 1024 products stays within |2^24|, where f32 holds every
//    integer.  One f32 accumulator (16 TMEM columns) takes the products of at
//    most eight 128-k units (8 x 128 = 1024 per element); epilogue warps turn
//    each finished accumulator into int32 and add it to their running sums,
//    so the int32 result is exact and tensor memory holds only a small ring
//    of accumulators whatever k is.
//  * Conversion int8 -> f16 is exact and cheap: a byte b becomes the f16 bit
//    pattern 0x6400 | (b + 128) (the value 1024 + b + 128) by a byte permute,
//    and one packed f16 subtraction of 1152 leaves b.
//  * The weights stream once.  The work is a list of units -- 128 rows x 128
//    k of W -- ordered band by band (a band is 128 rows), k fastest.  A
//    persistent grid of one CTA per SM splits that list into equal contiguous
//    ranges (stream-K), so every SM moves the same number of bytes whatever
//    the number of bands.  Each CTA runs two independent pipelines on the two
//    halves of its range; each has its own ring of shared-memory stages (2-D
//    TMA copies of one or two units of 128 rows x 128 bytes, 128-byte
//    swizzle, plus the matching activation columns), eight converter warps,
//    an MMA thread, four epilogue warps and half of the tensor memory.  The
//    converters of a pipeline take one unit of a stage per group of four warps
//    -- each thread a whole row, whose bytes the swizzle keeps conflict-free --
//    convert, and write the f16 A operand straight into tensor memory with
//    tcgen05.st; the activations become a 128-byte-swizzled K-major f16 B tile
//    in shared memory.
//  * One thread per pipeline issues the MMAs; tcgen05.commit releases A/B
//    buffers and hands finished accumulators to the epilogue warps.
//  * A band shared by the two pipelines is merged in shared memory by the
//    second to finish it.  A band split between CTAs leaves one record of
//    int32 partial sums per CTA in a caller-owned workspace; a small second
//    kernel, launched as a programmatic dependent of the first, adds the
//    records of each split band in CTA order, applies the scales and writes
//    the outputs, so the streaming kernel ends without any cross-CTA
//    handshake.  With no workspace every CTA takes whole bands instead.
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT,
//    every role stops at its next wait, issued copies and MMAs are allowed to
//    finish, records are still written (marked invalid), tensor memory is
//    freed and the affected outputs are NaN.
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace loom {
namespace {

using tc::i8x4_to_f16x4;
using tc::lds128;
using tc::mbar_arrive;
using tc::smem_desc_sw128;
using tc::sts128;
using tc::tma_load_2d;

constexpr int TC_M = 128;                    // rows per band (MMA M)
constexpr int TC_N = 16;                     // vectors per pass (MMA N)
constexpr int TC_KU = 128;                   // k (bytes) per unit
constexpr int TC_KSLICES = TC_KU / 16;       // MMAs per unit (K = 16 each)
constexpr int TC_UNITS_PER_GROUP = 8;        // units per f32 accumulator: 8 x 128 products
// Warps of a pipeline with g converter groups (four warps each, one per
// tensor-memory sub-partition): 4 g converters, four epilogue warps (one per
// sub-partition), the producer and the MMA issuer.
constexpr int TC_EPI_WARPS = 4;
__host__ __device__ constexpr int tc_pipe_warps(int groups) { return 4 * groups + TC_EPI_WARPS + 2; }
constexpr int TC_MAX_PIPES = 2;
constexpr int TC_MAX_GROUPS = 4;
constexpr int TC_MAX_CLUSTER = 4;                        // CTAs sharing one band
constexpr int TC_THREADS = 32 * 2 * tc_pipe_warps(2);   // the largest CTA: two pipelines of two groups
constexpr uint32_t TC_TMEM_COLS = 512;                   // the whole SM: one CTA per SM
constexpr uint32_t TC_W_BOX = TC_M * TC_KU;          // 16 KiB of weights per unit
constexpr uint32_t TC_X_UNIT = TC_N * TC_KU;         // 2 KiB of activations per unit
constexpr uint32_t TC_B_BYTES = TC_N * TC_KU * 2;    // f16 activation tile of one unit, 4 KiB
constexpr uint32_t TC_A_COLS = 64;                   // TMEM columns of one f16 A buffer
constexpr uint32_t TC_ACC_COLS = TC_N;               // TMEM columns of one f32 accumulator
constexpr int TC_MAX_ACC = 16;
constexpr int TC_WHOLE = 0;     // every CTA takes whole bands (no workspace)
constexpr int TC_SPLIT = 1;     // equal shares of the unit list; split bands finished by a second kernel
constexpr int TC_CLUSTER = 2;   // a cluster of CTAs per band, merged through distributed shared memory
constexpr uint32_t TC_EPI_BAR = 1;                   // named barriers 1, 2: epilogue warps of pipeline 0, 1
constexpr uint32_t TC_REC_HDR = 16;                   // record header: validity word + padding
constexpr uint32_t TC_REC_BYTES = TC_REC_HDR + 128 * 16 * 4;   // one split segment's partial sums
// instruction descriptor: D f32, A/B f16, both K-major, N = 16, M = 128
constexpr uint32_t TC_IDESC = tc::idesc_f16(TC_M, TC_N);

struct TcParams {
    const float *scale_w;
    const float *scale_x;
    float *y;
    int32_t *acc;
    int32_t *error;
    char *records;        // [grid][2] records: validity header, then int32 [128][16] partial sums,
                          // or NULL (no split)
    int32_t n_rows, batch, y_stride;
    int32_t units_per_band;   // ceil(k / 128)
    int64_t total_units;      // bands * units_per_band
    int32_t quantum;          // units per partition step: 1, or units_per_band (whole bands)
    int32_t depth;            // shared-memory stages per pipeline
    int32_t ups;              // units per stage (1 or 2)
    int32_t na;               // f16 A buffers per pipeline in tensor memory
    int32_t ng;               // f32 accumulators per pipeline in tensor memory
    int32_t pipes;            // pipelines per CTA (1 or 2)
    int32_t groups;           // converter groups per pipeline (= units per stage)
    int32_t mode;             // TC_WHOLE, TC_SPLIT or TC_CLUSTER (how bands map onto CTAs)
    int32_t cluster;          // CTAs per band in TC_CLUSTER mode
    uint32_t cta_area;        // shared memory in front of the pipelines
    uint32_t pipe_cols;       // tensor-memory columns of one pipeline
    uint32_t pipe_bytes;      // shared memory of one pipeline
    uint64_t wait_ns;
    int32_t inject_stall;
};

// Shared memory of one pipeline (1024-aligned): its stage ring, B tiles and barriers.
struct Layout {
    uint32_t base;
    int S, ups, na, ng, groups;
    __device__ uint32_t stage_bytes() const { return (uint32_t)ups * (TC_W_BOX + TC_X_UNIT); }
    __device__ uint32_t stage(int s) const { return base + (uint32_t)s * stage_bytes(); }
    // activations of unit bx of stage s: [16 vectors][128 bytes]
    __device__ uint32_t xtile(int s, int bx) const { return stage(s) + (uint32_t)ups * TC_W_BOX + (uint32_t)bx * TC_X_UNIT; }
    __device__ uint32_t btile(int a) const { return base + (uint32_t)S * stage_bytes() + (uint32_t)a * TC_B_BYTES; }
    __device__ uint32_t bars() const { return btile(na); }
    __device__ uint32_t full(int s) const { return bars() + 8 * s; }
    __device__ uint32_t empty(int s) const { return bars() + 8 * (S + s); }
    __device__ uint32_t aready(int a) const { return bars() + 8 * (2 * S + a); }
    __device__ uint32_t afree(int a) const { return bars() + 8 * (2 * S + na + a); }
    __device__ uint32_t gfull(int g) const { return bars() + 8 * (2 * S + 2 * na + g); }
    __device__ uint32_t gfree(int g) const { return bars() + 8 * (2 * S + 2 * na + ng + g); }
    __device__ uint32_t done() const { return bars() + 8 * (2 * S + 2 * na + 2 * ng); }
    __device__ int n_bars() const { return 2 * S + 2 * na + 2 * ng + 1; }
    // i-th barrier of the list above and its arrival count
    __device__ void bar_init(int i) const
    {
        uint32_t count;
        if (i < S) count = 1;
        else if (i < 2 * S) count = 4 * groups;                 // every converter warp
        else if (i < 2 * S + na) count = 4;                    // the four warps of one unit
        else if (i < 2 * S + 2 * na) count = 1;
        else if (i < 2 * S + 2 * na + ng) count = 1;
        else if (i < 2 * S + 2 * na + 2 * ng) count = TC_EPI_WARPS;
        else count = 1;
        dev::mbar_init(bars() + 8 * i, count);
    }
};

// Shared memory of the whole CTA, in front of the pipelines.
// Flags, the vector scales, the two pipelines' merge slots and, in a
// cluster's first CTA, one slot per other CTA of the cluster.
uint32_t tc_cta_area(int cluster)
{
    const uint32_t slots = 2u + (uint32_t)(cluster > 1 ? cluster - 1 : 0);
    return 1024u + ((slots * TC_REC_BYTES + 1023u) & ~1023u);
}

struct CtaArea {
    uint32_t base;
    __device__ uint32_t tmem_slot() const { return base; }
    __device__ uint32_t abort_flag() const { return base + 4; }
    __device__ uint32_t merge_ctr() const { return base + 8; }
    __device__ uint32_t second(int p) const { return base + 16 + 4 * p; }   // merge order, per pipeline
    __device__ uint32_t sx(int p) const { return base + 64 + 64 * p; }       // the pass's vector scales
    __device__ uint32_t cluster_in() const { return base + 192; }            // the other ranks' partials arrived
    __device__ uint32_t merge(int p) const { return base + 1024 + (uint32_t)p * TC_REC_BYTES; }
    __device__ uint32_t cslot(int r) const { return base + 1024 + (uint32_t)(2 + r) * TC_REC_BYTES; }
};

uint32_t tc_pipe_bytes(int S, int ups, int na, int ng)
{
    const uint32_t b = (uint32_t)S * ups * (TC_W_BOX + TC_X_UNIT) + (uint32_t)na * TC_B_BYTES +
                       8u * (2 * S + 2 * na + 2 * ng + 1);
    return (b + 1023u) & ~1023u;
}

uint32_t tc_smem_bytes(int pipes, int cluster, int S, int ups, int na, int ng)
{
    return 1024u + tc_cta_area(cluster) + (uint32_t)pipes * tc_pipe_bytes(S, ups, na, ng);
}

// ---- PTX wrappers ----------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Arrive on a barrier of another CTA of the cluster, releasing this thread's
// (and, through the preceding CTA barrier, its warps') shared-memory stores.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void epi_barrier(int p)
{
    asm volatile("bar.sync %0, %1;" ::"r"(TC_EPI_BAR + p), "n"(32 * TC_EPI_WARPS) : "memory");
}

// bar.sync of the epilogue warps that also returns the AND of `v` over them.
__device__ __forceinline__ bool epi_barrier_and(int p, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(TC_EPI_BAR + p), "n"(32 * TC_EPI_WARPS)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(TC_IDESC), "r"(accumulate)
        : "memory");
}

// The same, accumulating (the enable-input predicate as an immediate).
__device__ __forceinline__ void tc_mma_acc(uint32_t d, uint32_t a, uint64_t bdesc)
{
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a), "l"(bdesc),
                 "r"(TC_IDESC)
                 : "memory");
}

__device__ __forceinline__ bool aborted(const CtaArea &C) { return tc::aborted(C.abort_flag()); }

__device__ __forceinline__ void set_abort(const CtaArea &C, const TcParams &q) { tc::set_abort(C.abort_flag(), q.error); }

__device__ __forceinline__ bool role_wait(const CtaArea &C, const TcParams &q, uint32_t bar, uint32_t parity)
{
    return tc::role_wait(C.abort_flag(), q.error, q.wait_ns, bar, parity);
}

__device__ __forceinline__ bool warp_wait(const CtaArea &C, const TcParams &q, uint32_t bar, uint32_t parity)
{
    return tc::warp_wait(C.abort_flag(), q.error, q.wait_ns, bar, parity);
}

// ---- work partition ----------------------------------------------------------
// n / d for n >= 0, d > 0: one 32-bit division when both fit (64-bit division
// is a long instruction sequence, and these sit on the start-up path).
__device__ __forceinline__ int64_t div64(int64_t n, int64_t d)
{
    if ((((uint64_t)n) | ((uint64_t)d)) < (1ull << 32))
        return (int64_t)((uint32_t)n / (uint32_t)d);
    return n / d;
}

// CTA c of G takes units [begin(c), begin(c + 1)): equal shares of the unit
// list, in steps of `quantum` units.
__device__ __forceinline__ int64_t part_begin(const TcParams &q, int64_t c, int64_t G)
{
    const int64_t steps = div64(q.total_units, q.quantum);
    return q.quantum * div64(steps * c, G);
}

// The CTA whose range holds unit u (split partitions: quantum 1).  CTA c
// starts at floor(T c / G), so it is the largest c with T c < (u + 1) G.
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t T, int64_t G) { return div64((u + 1) * G - 1, T); }

// Walks a CTA's units stage by stage: up to `ups` units of one band.
struct StageWalk {
    int64_t u, u1, band;
    int32_t kb, ub, ups;
    __device__ StageWalk(int64_t u0_, int64_t u1_, int32_t ub_, int32_t ups_)
        : u(u0_), u1(u1_), band(div64(u0_, ub_)), kb((int32_t)(u0_ - div64(u0_, ub_) * ub_)), ub(ub_), ups(ups_)
    {
    }
    __device__ bool more() const { return u < u1; }
    __device__ int count() const
    {
        const int64_t left = u1 - u;
        const int c = ups < ub - kb ? ups : ub - kb;
        return left < c ? (int)left : c;
    }
    __device__ void next(int c)
    {
        u += c;
        kb += c;
        if (kb == ub) {
            kb = 0;
            ++band;
        }
    }
};

// Scale and store the sums of one row (all vectors of this pass); sw is the
// row's scale, the vector scales are read from shared memory.
__device__ __forceinline__ void store_row(const TcParams &q, uint32_t sx_at, int64_t row, float sw,
                                          const int32_t (&sum)[TC_N], bool valid)
{
    if (row >= q.n_rows)
        return;
#pragma unroll
    for (int b = 0; b < TC_N; ++b) {
        if (b < q.batch) {
            float sx;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sx) : "r"(sx_at + 4 * b));
            const int64_t o = row * q.y_stride + b;
            q.y[o] = valid ? __fmul_rn(__int2float_rn(sum[b]), __fmul_rn(sw, sx)) : __int_as_float(0x7fc00000);
            if (q.acc)
                q.acc[o] = valid ? sum[b] : INT32_MIN;
        }
    }
}

// Intra-CTA arrival for the band the two pipelines share (release: this
// pipeline's partial sums in shared memory; acquire: the other's).
__device__ __forceinline__ uint32_t arrive_merge(uint32_t ctr)
{
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(ctr) : "memory");
    return old;
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    dot_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                  const TcParams q)
{
    extern __shared__ unsigned char smem_raw[];
    // Set-up (barriers, tensor memory, the tensor maps' prefetch) may run while
    // the previous kernel on the stream drains; the first global access of each
    // role -- the producer's first copy, the epilogue's first scale load -- waits
    // for it (wait_previous_kernel).  The MMA and converter warps touch only
    // shared and tensor memory.  The next kernel (the finishing kernel, when
    // bands are split) is let in at teardown.
    const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
    const CtaArea C{base};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int PW = tc_pipe_warps(q.groups);
    const int CONV = 4 * q.groups;             // converter warps of a pipeline
    const int EPI0 = CONV;                     // its first epilogue warp
    const int PRODUCER = EPI0 + TC_EPI_WARPS;
    const int MMA = PRODUCER + 1;
    const int p = warp / PW;                   // pipeline
    const int w = warp % PW;                   // role within the pipeline
    Layout L;
    L.base = base + q.cta_area + (uint32_t)p * q.pipe_bytes;
    L.S = q.depth;
    L.ups = q.ups;
    L.na = q.na;
    L.ng = q.ng;
    L.groups = q.groups;
    const int S = q.depth, NA = q.na, NG = q.ng;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int32_t UB = q.units_per_band;
    // this CTA's units, and the halves of its pipelines
    int64_t U0, U1;
    uint32_t crank = 0;
    if (q.mode == TC_CLUSTER) {
        crank = cluster_rank();   // cluster b = blockIdx.x / C takes band b
        const int64_t b0 = (int64_t)(blockIdx.x / q.cluster) * UB;
        U0 = b0 + (int64_t)UB * crank / q.cluster;
        U1 = b0 + (int64_t)UB * (crank + 1) / q.cluster;
    } else {
        U0 = part_begin(q, cta, G);
        U1 = part_begin(q, cta + 1, G);
    }
    const int64_t M = q.pipes == 2 ? U0 + (U1 - U0) / 2 : U0;
    const int64_t u0 = (q.pipes == 2 && p == 0) ? U0 : M;
    const int64_t u1 = (q.pipes == 2 && p == 0) ? M : U1;
    const int64_t ou0 = p == 0 ? M : U0;       // the other pipeline's units (empty with one pipeline)
    const int64_t ou1 = q.pipes == 2 ? (p == 0 ? U1 : M) : ou0;

    // ---- set-up: barriers, flags, tensor memory ------------------------------
    // Each producer initialises its pipeline's barriers and at once issues the
    // copies of its first stages (they need nothing else), so the weights are
    // on their way while the rest of the CTA sets up.
    const uint64_t wpol = dev::l2_evict_first_policy();
    const uint64_t xpol = dev::l2_evict_last_policy();
    int issued = 0;        // producer: stages issued
    if (w == PRODUCER && p < q.pipes) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
        }
        for (int i = lane; i < L.n_bars(); i += 32)
            L.bar_init(i);
        dev::fence_barrier_init();
        __syncwarp();
        dev::wait_previous_kernel();
        if (lane == 0 && !q.inject_stall) {
            int i = 0;
            for (StageWalk sw(u0, u1, UB, q.ups); sw.more() && i < S; ++i) {
                const int cnt = sw.count();
                dev::mbar_arrive_expect_tx(L.full(i), cnt * (TC_W_BOX + TC_X_UNIT));
                for (int bx = 0; bx < cnt; ++bx) {
                    tma_load_2d(L.stage(i) + bx * TC_W_BOX, &tmw, (sw.kb + bx) * TC_KU,
                                (int32_t)(sw.band * TC_M), L.full(i), wpol);
                    tma_load_2d(L.xtile(i, bx), &tmx, (sw.kb + bx) * TC_KU, 0, L.full(i), xpol);
                }
                sw.next(cnt);
            }
            issued = i;
        }
    }
    if (threadIdx.x == 0) {
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(C.abort_flag()) : "memory");
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(C.merge_ctr()) : "memory");
        if (q.mode == TC_CLUSTER && crank == 0) {
            dev::mbar_init(C.cluster_in(), (uint32_t)(q.cluster - 1));   // one arrival per other rank
            dev::fence_barrier_init();
        }
    }
    if (p == 0 && w == PRODUCER) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(C.tmem_slot()),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (q.mode == TC_CLUSTER)
        cluster_sync();   // rank 0's barrier is initialised before any rank arrives on it
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(C.tmem_slot()));
    tmem += (uint32_t)p * q.pipe_cols;   // this pipeline's columns
    const uint32_t acc_col = (uint32_t)NA * TC_A_COLS;

    if (p >= q.pipes) {
        // no second pipeline: its warps only meet the final barrier
    } else if (w == PRODUCER) {
        // ---- producer: 2-D TMA of weight units and activation columns --------
        if (lane == 0) {
            int i = 0;
            for (StageWalk sw(u0, u1, UB, q.ups); sw.more(); ++i) {
                const int cnt = sw.count();
                const int s = i % S;
                if (i < S) {   // issued during set-up (none when stalled on purpose)
                    sw.next(cnt);
                    continue;
                }
                if (!role_wait(C, q, L.empty(s), ((i / S) - 1) & 1))
                    break;
                if (!q.inject_stall) {
                    dev::mbar_arrive_expect_tx(L.full(s), cnt * (TC_W_BOX + TC_X_UNIT));
                    for (int bx = 0; bx < cnt; ++bx) {
                        tma_load_2d(L.stage(s) + bx * TC_W_BOX, &tmw, (sw.kb + bx) * TC_KU,
                                    (int32_t)(sw.band * TC_M), L.full(s), wpol);
                        tma_load_2d(L.xtile(s, bx), &tmx, (sw.kb + bx) * TC_KU, 0, L.full(s), xpol);
                    }
                    ++issued;
                }
                sw.next(cnt);
            }
            // every copy issued must land before the CTA may leave (bounded)
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                dev::mbar_wait_bounded(L.full(j % S), (j / S) & 1, q.wait_ns);
        }
        __syncwarp();
    } else if (w == MMA) {
        // ---- MMA issuer: accumulator g takes up to 8 units of one band ------------
        // This thread shares its scheduler with converter warps, so the loop
        // keeps its own work small: descriptors and barrier addresses are
        // formed once, buffer indices and phases advance by increments.
        if (lane == 0) {
            const uint64_t bdesc0 = smem_desc_sw128(L.btile(0));   // + (byte offset >> 4) per tile and slice
            const uint32_t aready0 = L.aready(0), afree0 = L.afree(0);
            const uint32_t gfull0 = L.gfull(0), gfree0 = L.gfree(0);
            int a = 0, gs = 0;                 // A buffer and accumulator of the next unit / group
            uint32_t aph = 0, gph = 0;         // their barrier phase parities
            int g = 0;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok;) {
                const int64_t e = min(u1, (div64(u, UB) + 1) * UB);   // end of this band's segment
                for (int64_t gu = u; gu < e && ok; gu += TC_UNITS_PER_GROUP) {
                    if (g >= NG && !role_wait(C, q, gfree0 + 8 * gs, gph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const int n_in = (int)min((int64_t)TC_UNITS_PER_GROUP, e - gu);
                    const uint32_t d = tmem + acc_col + gs * TC_ACC_COLS;
                    for (int m = 0; m < n_in; ++m) {
                        if (!role_wait(C, q, aready0 + 8 * a, aph)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)a * (TC_B_BYTES >> 4));
                        const uint32_t ta = tmem + (uint32_t)a * TC_A_COLS;
                        tc_mma(d, ta, bd, m != 0 ? 1u : 0u);
#pragma unroll
                        for (int kk = 1; kk < TC_KSLICES; ++kk)
                            tc_mma_acc(d, ta + kk * 8, bd + (uint64_t)(((kk >> 2) * 2048 + (kk & 3) * 32) >> 4));
                        tc::commit(afree0 + 8 * a);   // A/B buffer a is free once these MMAs complete
                        if (++a == NA) {
                            a = 0;
                            aph ^= 1u;
                        }
                    }
                    if (!ok)
                        break;
                    tc::commit(gfull0 + 8 * gs);   // accumulator gs is final once these complete
                    ++g;
                    if (++gs == NG) {
                        gs = 0;
                        gph ^= 1u;
                    }
                }
                u = e;
            }
            tc::commit(L.done());   // every MMA issued by this thread has completed
        }
        __syncwarp();
    } else if (w < CONV) {
        // ---- converters: warp w owns tile rows 32 (w % 4) .. +31 (its TMEM lanes)
        // of unit h = w / 4 of each stage (whole 128-byte rows).  Both units of
        // a stage are read at once, so the stage goes back to the producer
        // after one round of loads.
        const int sub = w & 3;
        const int h = w >> 2;
        const int t = 32 * sub + lane;   // tile row
        const uint32_t tlane = (uint32_t)(32 * sub) << 16;
        bool ok = true;
        int i = 0, j0 = 0;
        for (StageWalk sw(u0, u1, UB, q.ups); sw.more() && ok; ++i) {
            const int cnt = sw.count();
            const int s = i % S;
            if (!warp_wait(C, q, L.full(s), (i / S) & 1)) {
                ok = false;
                break;
            }
            const bool mine = h < cnt;
            int4 wv[8];
            int4 xv = make_int4(0, 0, 0, 0);
            if (mine) {
                // a weight row (128 bytes, 128-byte swizzle) and a 16-byte piece of
                // the activations: vector t / 8, k = 16 (t % 8) .. +15 of this unit
                const uint32_t wrow = L.stage(s) + h * TC_W_BOX + t * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    wv[c] = lds128(wrow + ((c ^ (t & 7)) << 4));
                xv = lds128(L.xtile(s, h) + (t >> 3) * TC_KU + (t & 7) * 16);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(L.empty(s));   // this warp is done with stage s
            if (mine) {
                const int j = j0 + h;
                const int a = j % NA;
                if (j >= NA && !warp_wait(C, q, L.afree(a), ((j / NA) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                // A operand: 128 f16 of row t -> 64 TMEM columns of buffer a
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[16];
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int4 &v = wv[part * 2 + c2];
                        i8x4_to_f16x4((uint32_t)v.x, r[c2 * 8 + 0], r[c2 * 8 + 1]);
                        i8x4_to_f16x4((uint32_t)v.y, r[c2 * 8 + 2], r[c2 * 8 + 3]);
                        i8x4_to_f16x4((uint32_t)v.z, r[c2 * 8 + 4], r[c2 * 8 + 5]);
                        i8x4_to_f16x4((uint32_t)v.w, r[c2 * 8 + 6], r[c2 * 8 + 7]);
                    }
                    tc::st16(tmem + tlane + a * TC_A_COLS + part * 16, r);
                }
                // B operand: the activation piece into the K-major 128-byte-swizzled
                // f16 tile (two 64-k atoms of 16 rows)
                {
                    const int n = t >> 3, c8 = t & 7;
                    uint32_t hx[8];
                    i8x4_to_f16x4((uint32_t)xv.x, hx[0], hx[1]);
                    i8x4_to_f16x4((uint32_t)xv.y, hx[2], hx[3]);
                    i8x4_to_f16x4((uint32_t)xv.z, hx[4], hx[5]);
                    i8x4_to_f16x4((uint32_t)xv.w, hx[6], hx[7]);
                    const uint32_t atom = L.btile(a) + (c8 >> 2) * 2048 + (n >> 3) * 1024 + (n & 7) * 128;
                    const int c0 = 2 * (c8 & 3);
                    sts128(atom + (((c0) ^ (n & 7)) << 4), hx[0], hx[1], hx[2], hx[3]);
                    sts128(atom + (((c0 + 1) ^ (n & 7)) << 4), hx[4], hx[5], hx[6], hx[7]);
                }
                tc::wait_st();
                tc::fence_async_smem();
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(L.aready(a));
            }
            j0 += cnt;
            sw.next(cnt);
        }
    } else {
        // ---- epilogue warps: accumulators -> int32 row sums -> outputs ------------
        const int sub = w & 3;
        const int t = 32 * sub + lane;   // tile row
        const uint32_t tlane = (uint32_t)(32 * sub) << 16;
        const bool leader = w == EPI0 && lane == 0;
        dev::wait_previous_kernel();
        // the pass's vector scales, one copy per pipeline
        if (w == EPI0 && lane < TC_N) {
            const float v = lane < q.batch ? __ldg(q.scale_x + lane) : 0.f;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(C.sx(p) + 4 * lane), "f"(v) : "memory");
        }
        epi_barrier(p);
        bool ok = true;
        int g = 0;
        for (int64_t u = u0; u < u1;) {
            const int64_t band = div64(u, UB);
            const int64_t blo = band * UB, bhi = blo + UB;
            const int64_t e = min(u1, bhi);
            const int64_t row = band * TC_M + t;
            const float sw = row < q.n_rows ? __ldg(q.scale_w + row) : 0.f;   // in flight during the drain
            int32_t isum[TC_N];
#pragma unroll
            for (int b = 0; b < TC_N; ++b)
                isum[b] = 0;
            for (int64_t gu = u; gu < e; gu += TC_UNITS_PER_GROUP, ++g) {
                if (!ok)
                    continue;
                const int gs = g % NG;
                if (!warp_wait(C, q, L.gfull(gs), (g / NG) & 1)) {
                    ok = false;
                    continue;
                }
                tc::fence_after();
                uint32_t v[16];
                tc::ld16(tmem + tlane + acc_col + gs * TC_ACC_COLS, v);
#pragma unroll
                for (int b = 0; b < TC_N; ++b)
                    isum[b] += __float2int_rn(__uint_as_float(v[b]));
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(L.gfree(gs));
            }
            bool valid = ok && !aborted(C);
            u = e;
            if (blo >= u0 && bhi <= u1) {
                store_row(q, C.sx(p), row, sw, isum, valid);   // this pipeline holds the whole band
                continue;
            }
            // ---- the band the two pipelines share: the second to finish adds both
            if ((blo > ou0 ? blo : ou0) < (bhi < ou1 ? bhi : ou1)) {
                const uint32_t mine = C.merge(p);
#pragma unroll
                for (int b = 0; b < TC_N; b += 4)
                    sts128(mine + TC_REC_HDR + (t * TC_N + b) * 4, (uint32_t)isum[b], (uint32_t)isum[b + 1],
                           (uint32_t)isum[b + 2], (uint32_t)isum[b + 3]);
                valid = epi_barrier_and(p, valid);
                if (leader) {
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(mine), "r"(valid ? 1u : 0u) : "memory");
                    const uint32_t second = arrive_merge(C.merge_ctr());
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(C.second(p)), "r"(second) : "memory");
                }
                epi_barrier(p);
                uint32_t second;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(second) : "r"(C.second(p)));
                if (!second)
                    continue;   // the other pipeline finishes this band
                const uint32_t other = C.merge(p ^ 1);
                uint32_t hdr;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(hdr) : "r"(other));
                valid = valid && hdr != 0;
#pragma unroll
                for (int b = 0; b < TC_N; b += 4) {
                    const int4 v4 = lds128(other + TC_REC_HDR + (t * TC_N + b) * 4);
                    isum[b] += v4.x;
                    isum[b + 1] += v4.y;
                    isum[b + 2] += v4.z;
                    isum[b + 3] += v4.w;
                }
            }
            if (blo >= U0 && bhi <= U1) {
                store_row(q, C.sx(p), row, sw, isum, valid);   // this CTA holds the whole band
                continue;
            }
            if (q.mode == TC_CLUSTER) {
                // ---- the CTAs of a cluster share one band: rank 0 adds them in rank order
                if (crank != 0) {
                    const uint32_t slot = map_to_rank(C.cslot((int)crank - 1), 0);
#pragma unroll
                    for (int b = 0; b < TC_N; b += 4)
                        st_cluster_v4(slot + TC_REC_HDR + (t * TC_N + b) * 4, (uint32_t)isum[b],
                                      (uint32_t)isum[b + 1], (uint32_t)isum[b + 2], (uint32_t)isum[b + 3]);
                    valid = epi_barrier_and(p, valid);   // every row is stored before the release below
                    if (leader) {
                        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(slot), "r"(valid ? 1u : 0u) : "memory");
                        mbar_arrive_remote(map_to_rank(C.cluster_in(), 0));
                    }
                    continue;
                }
                bool got = mbar_try_wait_cluster(C.cluster_in(), 0);
                if (!got) {
                    const uint64_t t0 = dev::global_ns();
                    for (uint32_t i = 1; !got; ++i) {
                        got = mbar_try_wait_cluster(C.cluster_in(), 0);
                        if (!got && (i & 15u) == 0 && dev::global_ns() - t0 > q.wait_ns)
                            break;
                    }
                }
                if (!got) {
                    set_abort(C, q);
                    valid = false;
                }
                for (int r = 0; r + 1 < q.cluster; ++r) {
                    const uint32_t at = C.cslot(r);
                    uint32_t hdr;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(hdr) : "r"(at));
                    valid = valid && hdr != 0;
#pragma unroll
                    for (int b = 0; b < TC_N; b += 4) {
                        const int4 v4 = lds128(at + TC_REC_HDR + (t * TC_N + b) * 4);
                        isum[b] += v4.x;
                        isum[b + 1] += v4.y;
                        isum[b + 2] += v4.z;
                        isum[b + 3] += v4.w;
                    }
                }
                store_row(q, C.sx(p), row, sw, isum, valid);
                continue;
            }
            // ---- a band split between CTAs: this CTA's record of it (the
            // finishing kernel adds the records of every CTA sharing the band)
            const int64_t rec = 2 * cta + (band == div64(U0, UB) ? 0 : 1);
            char *rp = q.records + rec * TC_REC_BYTES;
            int4 *dst = reinterpret_cast<int4 *>(rp + TC_REC_HDR + t * TC_N * 4);
#pragma unroll
            for (int b = 0; b < TC_N; b += 4)
                __stcg(dst + b / 4, make_int4(isum[b], isum[b + 1], isum[b + 2], isum[b + 3]));
            const bool all_ok = epi_barrier_and(p, valid);
            if (leader)
                __stcg(reinterpret_cast<int4 *>(rp), make_int4(all_ok ? 1 : 0, 0, 0, 0));
        }
    }

    // ---- teardown: tensor memory is freed only after every MMA has completed
    tc::fence_before();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the finishing kernel may start
    if (p == 0 && w == PRODUCER) {
        if (lane < q.pipes) {
            Layout Lp = L;
            Lp.base = base + q.cta_area + (uint32_t)lane * q.pipe_bytes;
            dev::mbar_wait_bounded(Lp.done(), 0, q.wait_ns);
        }
        __syncwarp();
        tc::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
    }
    if (q.mode == TC_CLUSTER)
        cluster_sync();   // no CTA leaves while another may still write its shared memory
}

// ---- finishing kernel for bands split between CTAs ------------------------------
struct FinishParams {
    const char *records;
    const float *scale_w;
    const float *scale_x;
    float *y;
    int32_t *acc;
    int32_t n_rows, batch, y_stride;
    int32_t units_per_band;
    int64_t total_units;   // T of the streaming launch
    int64_t grid;          // its CTA count
    int64_t bands;
};

constexpr int TC_FIN_THREADS = 4 * TC_M;   // four threads per row, four vectors each

// Band b of a streaming launch of G CTAs over T units (one unit per partition
// step) is split when its first and last units belong to different CTAs;
// each of them left a record of its partial sums (record 2c for the band of
// CTA c's first unit, 2c + 1 for the other).  One CTA per band adds the
// records in CTA order, scales and stores.
__global__ void __launch_bounds__(TC_FIN_THREADS) dot_tc_finish_kernel(const FinishParams f)
{
    __shared__ int64_t span[3];   // first and last CTA of the band, and cf's record index
    dev::follow_previous_kernel();   // the streaming kernel's records are complete
    const int r_in = threadIdx.x >> 2;                    // row within the band
    const int quad = threadIdx.x & 3;                      // vectors 4 quad .. 4 quad + 3
    const int64_t T = f.total_units, G = f.grid;
    const int64_t UB = f.units_per_band;
    for (int64_t band = blockIdx.x; band < f.bands; band += gridDim.x) {
        if (threadIdx.x == 0) {
            const int64_t cf = owner_of(band * UB, T, G);
            span[0] = cf;
            span[1] = owner_of((band + 1) * UB - 1, T, G);
            // the first CTA's record: its head if its range starts at the band, else its tail;
            // every later CTA starts inside the band (its head record)
            span[2] = 2 * cf + (div64(T * cf, G) == band * UB ? 0 : 1);
        }
        __syncthreads();
        const int64_t cf = span[0], cl = span[1], r0 = span[2];
        __syncthreads();
        if (cf == cl)
            continue;   // one CTA held the whole band and wrote its outputs
        const int64_t row = band * TC_M + r_in;
        const bool live = row < f.n_rows;
        // scales first: their loads overlap the records'
        const float sw = live ? __ldg(f.scale_w + row) : 0.f;
        float sx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            sx[i] = 4 * quad + i < f.batch ? __ldg(f.scale_x + 4 * quad + i) : 0.f;
        int32_t tot[4] = {0, 0, 0, 0};
        bool valid = true;
        // the records of up to four CTAs at a time, all loads in flight together
        for (int64_t c0 = cf; c0 <= cl; c0 += 4) {
            int4 v[4];
            int hdr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t c = c0 + i;
                v[i] = make_int4(0, 0, 0, 0);
                hdr[i] = 1;
                if (c <= cl) {
                    const int64_t r = c == cf ? r0 : 2 * c;
                    const char *rp = f.records + r * TC_REC_BYTES;
                    v[i] = __ldcg(reinterpret_cast<const int4 *>(rp + TC_REC_HDR + (r_in * TC_N + 4 * quad) * 4));
                    hdr[i] = __ldcg(reinterpret_cast<const int *>(rp));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                tot[0] += v[i].x;
                tot[1] += v[i].y;
                tot[2] += v[i].z;
                tot[3] += v[i].w;
                valid &= hdr[i] != 0;
            }
        }
        if (!live)
            continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = 4 * quad + i;
            if (b < f.batch) {
                const int64_t o = row * f.y_stride + b;
                f.y[o] = valid ? __fmul_rn(__int2float_rn(tot[i]), __fmul_rn(sw, sx[i])) : __int_as_float(0x7fc00000);
                if (f.acc)
                    f.acc[o] = valid ? tot[i] : INT32_MIN;
            }
        }
    }
}

// ---- host side ------------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

bool encode_2d_u8_uncached(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle)
{
    EncodeTiled enc = encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host work per call is kept small: the last few tensor maps are reused while
// their tensor and box are the same (encoding is a driver call).
struct MapEntry {
    const void *base;
    uint64_t inner, outer;
    uint32_t box_inner, box_outer;
    CUtensorMapSwizzle swizzle;
    CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[8];
int g_maps_used = 0, g_maps_next = 0;

}  // namespace

bool encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                             uint32_t box_outer, CUtensorMapSwizzle swizzle)
{
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_maps_used; ++i) {
        const MapEntry &m = g_maps[i];
        if (m.base == base && m.inner == inner && m.outer == outer && m.box_inner == box_inner &&
            m.box_outer == box_outer && m.swizzle == swizzle) {
            *map = m.map;
            return true;
        }
    }
    if (!encode_2d_u8_uncached(map, base, inner, outer, box_inner, box_outer, swizzle))
        return false;
    MapEntry &m = g_maps[g_maps_next];
    m = MapEntry{base, inner, outer, box_inner, box_outer, swizzle, *map};
    g_maps_next = (g_maps_next + 1) % 8;
    g_maps_used = g_maps_used < 8 ? g_maps_used + 1 : 8;
    return true;
}

namespace {

// The kernel's dynamic shared-memory limit, raised once per device to the
// largest size asked for so far.
std::atomic<int> g_smem_limit[64];

cudaError_t ensure_smem_limit(uint32_t bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(dot_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    int cur = g_smem_limit[dev].load(std::memory_order_acquire);
    if ((int)bytes <= cur)
        return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(dot_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) {
        while (cur < (int)bytes && !g_smem_limit[dev].compare_exchange_weak(cur, (int)bytes))
            ;
    }
    return e;
}

// cudaOccupancyMaxActiveClusters answers, per device and launch shape.
struct ClusterFit {
    int dev;
    uint32_t smem;
    int threads, cluster, n;
};
std::mutex g_fit_mu;
ClusterFit g_fits[16];
int g_fits_used = 0;


// Shared memory per CTA: at least 120 KiB, more than half of the SM's, so
// that one CTA runs per SM and finds all 512 tensor-memory columns free
// (tcgen05.alloc would otherwise wait for another CTA to finish).
constexpr uint32_t TC_MIN_SMEM = 120u * 1024u;
constexpr uint32_t TC_MAX_SMEM = 227u * 1024u;

int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }

}  // namespace

bool dot_tc_eligible(bool aligned, int32_t k, int32_t batch_pass)
{
    return aligned && k >= 16 && (k % 16) == 0 && batch_pass >= 1 && batch_pass <= TC_N;
}

int dot_tc_threads(int pipes) { return 32 * pipes * tc_pipe_warps(pipes == 2 ? 2 : TC_MAX_GROUPS); }

int dot_tc_rows_per_band() { return TC_M; }

// Resolve the schedule of one tensor-core launch.  cfg fields of 0 take the
// defaults: two pipelines per CTA, two units per stage, two stages, three A
// buffers per pipeline (the rest of its tensor memory holds accumulators).
// Rows map onto CTAs in one of four ways (cfg.schedule, 0 = choose):
//  * whole rows per CTA (dot_tc_rows.cu) when n_rows / SMs fills at least half
//    of the 64 rows of a block and k has 16 units or more: no partial sums
//    leave a CTA;
//  * a cluster of C CTAs per band (C = 2..4) when that keeps every SM busy --
//    or, with no workspace, at least three quarters of them: no cross-SM
//    traffic at all;
//  * equal shares of the whole unit list (stream-K) when a workspace is given;
//  * whole bands per CTA otherwise.
bool dot_tc_plan(int64_t n_rows, int32_t k, int64_t sm_count, const DotTcConfig &cfg, bool split,
                 DotTcPlan *out)
{
    // whole rows per CTA, where the rows fill the tensor-memory lanes well (dot_tc_rows.cu)
    if (cfg.schedule == 4)
        return dot_tc_rows_plan(n_rows, k, sm_count, cfg, true, out);
    if (cfg.schedule == 0 && dot_tc_rows_plan(n_rows, k, sm_count, cfg, false, out))
        return true;
    const int pipes = cfg.pipes ? cfg.pipes : 2;
    if (pipes < 1 || pipes > TC_MAX_PIPES)
        return false;
    const int groups = pipes == 2 ? 2 : TC_MAX_GROUPS;   // converter groups per pipeline
    const int ups = cfg.units_per_stage ? cfg.units_per_stage : groups;
    if (ups < 1 || ups > groups || sm_count < 1 || cfg.schedule < 0 || cfg.schedule > 4)
        return false;
    const int depth = cfg.depth ? cfg.depth : (ups >= 2 ? 2 : 4);
    const uint32_t cols = TC_TMEM_COLS / (uint32_t)pipes;
    const int na = cfg.a_bufs ? cfg.a_bufs : 2 * groups - 1;
    // A group's consecutive units are at most 2 groups - 1 apart (a stage cut
    // short by a band's end is skipped by the groups past its units); with
    // fewer A buffers than that a group could wait on a barrier phase two
    // ahead of the last one completed.
    if (depth < 1 || depth > LOOM_MAX_DEPTH || na < 2 * groups - 1 ||
        (uint32_t)na * TC_A_COLS + 2 * TC_ACC_COLS > cols)
        return false;
    int ng = (int)((cols - (uint32_t)na * TC_A_COLS) / TC_ACC_COLS);
    ng = ng > TC_MAX_ACC ? TC_MAX_ACC : ng;
    const int64_t bands = (n_rows + TC_M - 1) / TC_M;
    const int32_t ub = (k + TC_KU - 1) / TC_KU;
    const int64_t total = bands * ub;

    // CTAs per band for the cluster schedule: each CTA keeps at least one unit per pipeline
    int64_t c = bands > 0 ? sm_count / bands : 0;
    c = c > TC_MAX_CLUSTER ? TC_MAX_CLUSTER : c;
    c = c > ub / pipes ? ub / pipes : c;
    int mode;
    if (cfg.schedule == 1)
        mode = TC_WHOLE;
    else if (cfg.schedule == 2)
        mode = TC_SPLIT;
    else if (cfg.schedule == 3)
        mode = TC_CLUSTER;
    else if (c >= 2 && (split ? bands * c == sm_count : 4 * bands * c >= 3 * sm_count))
        mode = TC_CLUSTER;   // every SM busy (or, with no workspace, most of them)
    else
        mode = split ? TC_SPLIT : TC_WHOLE;
    if (mode == TC_SPLIT && !split)
        return false;   // the split schedule needs the workspace
    if (mode == TC_CLUSTER && c < 2)
        mode = TC_WHOLE;   // one CTA per band already
    const int cluster = mode == TC_CLUSTER ? (int)c : 1;

    uint32_t smem = tc_smem_bytes(pipes, cluster, depth, ups, na, ng);
    if (smem > TC_MAX_SMEM)
        return false;
    smem = smem < TC_MIN_SMEM ? TC_MIN_SMEM : smem;
    const int32_t quantum = mode == TC_SPLIT ? 1 : ub;
    const int64_t steps = total / quantum;
    if (mode == TC_CLUSTER)
        out->grid = bands * cluster;
    else
        out->grid = steps < sm_count ? steps : sm_count;
    out->quantum = quantum;
    out->units_per_band = ub;
    out->total_units = total;
    out->depth = depth;
    out->ups = ups;
    out->na = na;
    out->ng = ng;
    out->pipes = pipes;
    out->groups = groups;
    out->mode = mode;
    out->cluster = cluster;
    out->cta_area = tc_cta_area(cluster);
    out->pipe_cols = cols;
    out->pipe_bytes = tc_pipe_bytes(depth, ups, na, ng);
    out->smem_bytes = smem;
    out->split = mode == TC_SPLIT;
    out->sm_count = sm_count;
    return true;
}

// Workspace of a split launch: two partial-sum records (validity header +
// sums) per CTA, every one written before it is read, so the workspace needs
// no initialisation.
int64_t dot_tc_workspace_bytes(const DotTcPlan &plan)
{
    return plan.split ? align256(plan.grid * 2 * (int64_t)TC_REC_BYTES) : 0;
}

// Whether every cluster of a cluster-schedule plan is resident at once on the
// current device (clusters need their CTAs' SMs inside one GPC, so fewer may
// fit than SMs / cluster).
bool dot_tc_cluster_fits(const DotTcPlan &plan)
{
    if (plan.mode != TC_CLUSTER)
        return true;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const int threads = dot_tc_threads(plan.pipes);
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        for (int i = 0; i < g_fits_used; ++i) {
            const ClusterFit &f = g_fits[i];
            if (f.dev == dev && f.smem == plan.smem_bytes && f.threads == threads && f.cluster == plan.cluster)
                return (int64_t)f.n * plan.cluster >= plan.grid;
        }
    }
    if (ensure_smem_limit(plan.smem_bytes) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)dot_tc_threads(plan.pipes), 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeClusterDimension;
    ca[0].val.clusterDim.x = (unsigned)plan.cluster;
    ca[0].val.clusterDim.y = 1;
    ca[0].val.clusterDim.z = 1;
    cfg.attrs = ca;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dot_tc_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        if (g_fits_used < 16)
            g_fits[g_fits_used++] = ClusterFit{dev, plan.smem_bytes, threads, plan.cluster, n};
    }
    return (int64_t)n * plan.cluster >= plan.grid;
}

cudaError_t launch_dot_tc(const DotParams &p, const DotTcPlan &plan, cudaStream_t stream)
{
    if (plan.mode == DOT_TC_ROWS)
        return launch_dot_tc_rows(p, plan, stream);
    if (plan.grid == 0)
        return cudaSuccess;
    const int64_t k = (int64_t)p.k_words * 4;
    CUtensorMap tmw, tmx;
    if (!encode_tensor_map_2d_u8(&tmw, p.w, (uint64_t)k, (uint64_t)p.n_rows, TC_KU, TC_M, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d_u8(&tmx, p.x, (uint64_t)k, (uint64_t)p.batch, TC_KU, TC_N, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcParams q;
    q.scale_w = p.scale_w;
    q.scale_x = p.scale_x;
    q.y = p.y;
    q.acc = p.acc;
    q.error = p.error;
    q.records = nullptr;
    if (plan.split) {
        if (!p.workspace || p.workspace_bytes < dot_tc_workspace_bytes(plan))
            return cudaErrorInvalidValue;
        q.records = static_cast<char *>(p.workspace);
    }
    q.n_rows = p.n_rows;
    q.batch = p.batch;
    q.y_stride = p.y_stride;
    q.units_per_band = plan.units_per_band;
    q.total_units = plan.total_units;
    q.quantum = plan.quantum;
    q.depth = plan.depth;
    q.ups = plan.ups;
    q.na = plan.na;
    q.ng = plan.ng;
    q.pipes = plan.pipes;
    q.groups = plan.groups;
    q.mode = plan.mode;
    q.cluster = plan.cluster;
    q.cta_area = plan.cta_area;
    q.pipe_cols = plan.pipe_cols;
    q.pipe_bytes = plan.pipe_bytes;
    q.wait_ns = p.wait_ns;
    q.inject_stall = p.inject_stall;

    cudaError_t e = ensure_smem_limit(plan.smem_bytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)dot_tc_threads(plan.pipes), 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute ca[2];
    ca[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see follow_previous_kernel
    ca[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = ca;
    cfg.numAttrs = 1;
    if (plan.mode == TC_CLUSTER) {
        ca[1].id = cudaLaunchAttributeClusterDimension;
        ca[1].val.clusterDim.x = (unsigned)plan.cluster;
        ca[1].val.clusterDim.y = 1;
        ca[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    e = cudaLaunchKernelEx(&cfg, dot_tc_kernel, tmw, tmx, q);
    if (e != cudaSuccess || !plan.split)
        return e;

    // bands split between CTAs: the finishing kernel, a programmatic dependent
    // (its CTAs are scheduled as the streaming CTAs retire)
    FinishParams f;
    f.records = q.records;
    f.scale_w = p.scale_w;
    f.scale_x = p.scale_x;
    f.y = p.y;
    f.acc = p.acc;
    f.n_rows = p.n_rows;
    f.batch = p.batch;
    f.y_stride = p.y_stride;
    f.units_per_band = plan.units_per_band;
    f.total_units = plan.total_units;
    f.grid = plan.grid;
    f.bands = plan.total_units / plan.units_per_band;
    cudaLaunchConfig_t fc = {};
    fc.gridDim = dim3((unsigned)(f.bands < 4096 ? f.bands : 4096), 1, 1);
    fc.blockDim = dim3(TC_FIN_THREADS, 1, 1);
    fc.stream = stream;
    cudaLaunchAttribute fa[1];
    fa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    fa[0].val.programmaticStreamSerializationAllowed = 1;
    fc.attrs = fa;
    fc.numAttrs = 1;
    return cudaLaunchKernelEx(&fc, dot_tc_finish_kernel, f);
}

}  // namespace loom
