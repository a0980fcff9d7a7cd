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
//    persistent grid of two CTAs per SM splits that list into equal
//    contiguous ranges (stream-K), so every SM moves the same number of
//    bytes whatever the number of bands.  A 2-D TMA copy brings one or two
//    units per stage (128 rows x 128 bytes each, 128-byte swizzle) plus the
//    matching activation columns into a ring of `depth` shared-memory
//    stages.  Eight converter warps -- two per tensor-memory sub-partition,
//    each half of every row -- read their bytes (the swizzle keeps the reads
//    conflict-free), convert, and write the f16 A operand straight into
//    tensor memory with tcgen05.st; the activations become a 128-byte-
//    swizzled K-major f16 B tile in shared memory.
//  * One thread issues the MMAs; tcgen05.commit releases A/B buffers and
//    hands finished accumulators to the epilogue warps.
//  * A band split between CTAs is finished through a caller-owned workspace:
//    each contributing CTA stores its int32 partial sums, then bumps a
//    counter; the last to arrive adds all partials in CTA order, applies the
//    scales, writes the outputs and resets the counter to zero.  Integer
//    partial sums make the result independent of the arrival order.  With no
//    workspace every CTA takes whole bands instead.
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT,
//    every role stops at its next wait, issued copies and MMAs are allowed to
//    finish, split bands still reach their counters (so the workspace is left
//    clean), tensor memory is freed and the affected outputs are NaN.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

constexpr int TC_M = 128;                    // rows per band (MMA M)
constexpr int TC_N = 16;                     // vectors per pass (MMA N)
constexpr int TC_KU = 128;                   // k (bytes) per unit
constexpr int TC_KSLICES = TC_KU / 16;       // MMAs per unit (K = 16 each)
constexpr int TC_UNITS_PER_GROUP = 8;        // units per f32 accumulator: 8 x 128 products
constexpr int TC_CONV_WARPS = 8;             // two per TMEM sub-partition, each half a row
constexpr int TC_EPI_WARP0 = TC_CONV_WARPS;  // four epilogue warps, one per sub-partition
constexpr int TC_EPI_WARPS = 4;
constexpr int TC_PRODUCER_WARP = TC_EPI_WARP0 + TC_EPI_WARPS;
constexpr int TC_MMA_WARP = TC_PRODUCER_WARP + 1;
constexpr int TC_THREADS = 32 * (TC_MMA_WARP + 1);
constexpr uint32_t TC_W_BOX = TC_M * TC_KU;          // 16 KiB of weights per unit
constexpr uint32_t TC_X_UNIT = TC_N * TC_KU;         // 2 KiB of activations per unit
constexpr uint32_t TC_B_BYTES = TC_N * TC_KU * 2;    // f16 activation tile of one unit, 4 KiB
constexpr uint32_t TC_A_COLS = 64;                   // TMEM columns of one f16 A buffer
constexpr uint32_t TC_ACC_COLS = TC_N;               // TMEM columns of one f32 accumulator
constexpr int TC_MAX_UPS = 2;                        // units per stage
constexpr int TC_MAX_ACC = 16;
constexpr uint32_t TC_EPI_BAR = 1;                   // named barrier of the epilogue warps
constexpr uint32_t TC_REC_HDR = 16;                   // record header: validity word + padding
constexpr uint32_t TC_REC_BYTES = TC_REC_HDR + 128 * 16 * 4;   // one split segment's partial sums
// instruction descriptor: D f32, A/B f16, both K-major, N = 16, M = 128
constexpr uint32_t TC_IDESC = (1u << 4) | ((TC_N >> 3) << 17) | ((TC_M >> 4) << 24);

struct TcParams {
    const float *scale_w;
    const float *scale_x;
    float *y;
    int32_t *acc;
    int32_t *error;
    uint32_t *counters;   // [2 x SMs] split-band arrival counters, or NULL (no split)
    char *records;        // [grid][2] records: validity header, then int32 [128][16] partial sums
    int32_t n_rows, batch, y_stride;
    int32_t units_per_band;   // ceil(k / 128)
    int64_t total_units;      // bands * units_per_band
    int32_t quantum;          // units per partition step: 1, or units_per_band (whole bands)
    int32_t depth;            // shared-memory stages
    int32_t ups;              // units per stage (1 or 2)
    int32_t na;               // f16 A buffers in tensor memory
    int32_t ng;               // f32 accumulators in tensor memory
    uint32_t tmem_cols;
    uint64_t wait_ns;
    int32_t inject_stall;
};

struct Layout {
    uint32_t base;   // 1024-aligned shared address
    int S, ups, na, ng;
    __device__ uint32_t stage_bytes() const { return (uint32_t)ups * (TC_W_BOX + TC_X_UNIT); }
    __device__ uint32_t stage(int s) const { return base + (uint32_t)s * stage_bytes(); }
    __device__ uint32_t xtile(int s) const { return stage(s) + (uint32_t)ups * TC_W_BOX; }
    __device__ uint32_t btile(int a) const { return base + (uint32_t)S * stage_bytes() + (uint32_t)a * TC_B_BYTES; }
    __device__ uint32_t bars() const { return btile(na); }
    __device__ uint32_t full(int s) const { return bars() + 8 * s; }
    __device__ uint32_t empty(int s) const { return bars() + 8 * (S + s); }
    __device__ uint32_t aready(int a) const { return bars() + 8 * (2 * S + a); }
    __device__ uint32_t afree(int a) const { return bars() + 8 * (2 * S + na + a); }
    __device__ uint32_t gfull(int g) const { return bars() + 8 * (2 * S + 2 * na + g); }
    __device__ uint32_t gfree(int g) const { return bars() + 8 * (2 * S + 2 * na + ng + g); }
    __device__ uint32_t done() const { return bars() + 8 * (2 * S + 2 * na + 2 * ng); }
    __device__ uint32_t tmem_slot() const { return done() + 8; }
    __device__ uint32_t abort_flag() const { return done() + 12; }
    __device__ uint32_t last_flag() const { return done() + 16; }
    __device__ uint32_t sx() const { return done() + 24; }   // the pass's vector scales, 16 f32
};

uint32_t tc_smem_bytes(int S, int ups, int na, int ng)
{
    return 1024u + (uint32_t)S * ups * (TC_W_BOX + TC_X_UNIT) + (uint32_t)na * TC_B_BYTES +
           8u * (2 * S + 2 * na + 2 * ng + 1) + 16u + 64u;
}

// ---- PTX wrappers ----------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void epi_barrier()
{
    asm volatile("bar.sync %0, %1;" ::"n"(TC_EPI_BAR), "n"(32 * TC_EPI_WARPS) : "memory");
}

// bar.sync of the epilogue warps that also returns the AND of `v` over them.
__device__ __forceinline__ bool epi_barrier_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(TC_EPI_BAR), "n"(32 * TC_EPI_WARPS)
        : "memory");
    return r != 0;
}

// 16-byte copy global (L2) -> shared memory by this thread, completed by cp.async.wait_group.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(TC_IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory descriptor of a K-major operand with 128-byte swizzle:
// start address, leading offset (unused here, 16 B), stride between 8-row
// groups 1024 B, descriptor version 1, layout "128-byte swizzle".
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t start)
{
    return (uint64_t)((start >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Four signed bytes -> two f16x2 words (elements 0,1 and 2,3; low half first).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;   // b + 128 as an unsigned byte
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));   // - 1152
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__device__ __forceinline__ int4 lds128(uint32_t addr)
{
    int4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ bool aborted(const Layout &L)
{
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(L.abort_flag()));
    return v != 0;
}

__device__ __forceinline__ void set_abort(const Layout &L, const TcParams &q)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(L.abort_flag()), "r"(1u) : "memory");
    dev::flag_error(q.error, LOOM_DEVERR_TIMEOUT);
}

// Wait for a phase of `bar`; false once the CTA has aborted or the limit
// has passed (which aborts the CTA).
__device__ __forceinline__ bool role_wait(const Layout &L, const TcParams &q, uint32_t bar, uint32_t parity)
{
    if (dev::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = dev::global_ns();
    for (uint32_t i = 1;; ++i) {
        if (dev::mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0) {
            if (aborted(L))
                return false;
            if (dev::global_ns() - t0 > q.wait_ns) {
                set_abort(L, q);
                return false;
            }
        }
    }
}

// The same, agreed by every lane of the warp.
__device__ __forceinline__ bool warp_wait(const Layout &L, const TcParams &q, uint32_t bar, uint32_t parity)
{
    return __all_sync(dev::FULL_MASK, role_wait(L, q, bar, parity));
}

// ---- work partition ----------------------------------------------------------
// CTA c of G takes units [begin(c), begin(c + 1)): equal shares of the unit
// list, in steps of `quantum` units.
__device__ __forceinline__ int64_t part_begin(const TcParams &q, int64_t c, int64_t G)
{
    const int64_t steps = q.total_units / q.quantum;
    return q.quantum * (steps * c / G);
}

// The CTA whose range holds unit u (split partitions: quantum 1).  CTA c
// starts at floor(T c / G), so it is the largest c with T c < (u + 1) G.
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t T, int64_t G) { return ((u + 1) * G - 1) / T; }

// Walks a CTA's units stage by stage: up to `ups` units of one band.
struct StageWalk {
    int64_t u, u1, band;
    int32_t kb, ub, ups;
    __device__ StageWalk(int64_t u0_, int64_t u1_, int32_t ub_, int32_t ups_)
        : u(u0_), u1(u1_), band(u0_ / ub_), kb((int32_t)(u0_ - (u0_ / ub_) * ub_)), ub(ub_), ups(ups_)
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
__device__ __forceinline__ void store_row(const TcParams &q, const Layout &L, int64_t row, float sw,
                                          const int32_t (&sum)[TC_N], bool valid)
{
    if (row >= q.n_rows)
        return;
#pragma unroll
    for (int b = 0; b < TC_N; ++b) {
        if (b < q.batch) {
            float sx;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sx) : "r"(L.sx() + 4 * b));
            const int64_t o = row * q.y_stride + b;
            q.y[o] = valid ? __fmul_rn(__int2float_rn(sum[b]), __fmul_rn(sw, sx)) : __int_as_float(0x7fc00000);
            if (q.acc)
                q.acc[o] = valid ? sum[b] : INT32_MIN;
        }
    }
}

// Counter increment with release (this CTA's partial sums, ordered before it
// by the epilogue barrier, become visible with it) and acquire (the last to
// arrive sees every other partial).
__device__ __forceinline__ uint32_t arrive_counter(uint32_t *ctr)
{
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctr) : "memory");
    return old;
}

__global__ void __launch_bounds__(TC_THREADS, 2)
    dot_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                  const TcParams q)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = dev::smem_u32(smem_raw);
    Layout L;
    L.base = (raw + 1023u) & ~1023u;
    L.S = q.depth;
    L.ups = q.ups;
    L.na = q.na;
    L.ng = q.ng;
    const int S = q.depth, NA = q.na, NG = q.ng;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t u0 = part_begin(q, cta, G);
    const int64_t u1 = part_begin(q, cta + 1, G);
    const int32_t UB = q.units_per_band;

    // ---- set-up: barriers, flags, tensor memory ------------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            dev::mbar_init(L.full(s), 1);
            dev::mbar_init(L.empty(s), TC_CONV_WARPS);
        }
        for (int a = 0; a < NA; ++a) {
            dev::mbar_init(L.aready(a), TC_CONV_WARPS / 2);   // the four warps of one unit
            dev::mbar_init(L.afree(a), 1);
        }
        for (int g = 0; g < NG; ++g) {
            dev::mbar_init(L.gfull(g), 1);
            dev::mbar_init(L.gfree(g), TC_EPI_WARPS);
        }
        dev::mbar_init(L.done(), 1);
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(L.abort_flag()) : "memory");
        dev::fence_barrier_init();
    }
    if (warp == TC_MMA_WARP && lane < TC_N) {
        const float v = lane < q.batch ? __ldg(q.scale_x + lane) : 0.f;
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(L.sx() + 4 * lane), "f"(v) : "memory");
    }
    if (warp == TC_PRODUCER_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(L.tmem_slot()),
                     "r"(q.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(L.tmem_slot()));
    const uint32_t acc_col = (uint32_t)NA * TC_A_COLS;

    if (warp == TC_PRODUCER_WARP) {
        // ---- producer: 2-D TMA of weight units and activation columns --------
        if (lane == 0) {
            const uint64_t wpol = dev::l2_evict_first_policy();
            const uint64_t xpol = dev::l2_evict_last_policy();
            int issued = 0;
            int i = 0;
            for (StageWalk sw(u0, u1, UB, q.ups); sw.more(); ++i) {
                const int cnt = sw.count();
                const int s = i % S;
                if (i >= S && !role_wait(L, q, L.empty(s), ((i / S) - 1) & 1))
                    break;
                if (!q.inject_stall) {
                    dev::mbar_arrive_expect_tx(L.full(s), cnt * TC_W_BOX + q.ups * TC_X_UNIT);
                    for (int bx = 0; bx < cnt; ++bx)
                        tma_load_2d(L.stage(s) + bx * TC_W_BOX, &tmw, (sw.kb + bx) * TC_KU,
                                    (int32_t)(sw.band * TC_M), L.full(s), wpol);
                    tma_load_2d(L.xtile(s), &tmx, sw.kb * TC_KU, 0, L.full(s), xpol);
                    ++issued;
                }
                sw.next(cnt);
            }
            // every copy issued must land before the CTA may leave (bounded)
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                dev::mbar_wait_bounded(L.full(j % S), (j / S) & 1, q.wait_ns);
        }
        __syncwarp();
    } else if (warp == TC_MMA_WARP) {
        // ---- MMA issuer: accumulator g takes up to 8 units of one band ------------
        if (lane == 0) {
            int j = 0, g = 0;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok;) {
                const int64_t e = min(u1, (u / UB + 1) * UB);   // end of this band's segment
                for (int64_t gu = u; gu < e && ok; gu += TC_UNITS_PER_GROUP) {
                    const int gs = g % NG;
                    if (g >= NG && !role_wait(L, q, L.gfree(gs), ((g / NG) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const int n_in = (int)min((int64_t)TC_UNITS_PER_GROUP, e - gu);
                    const uint32_t d = tmem + acc_col + gs * TC_ACC_COLS;
                    for (int m = 0; m < n_in; ++m, ++j) {
                        const int a = j % NA;
                        if (!role_wait(L, q, L.aready(a), (j / NA) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < TC_KSLICES; ++kk) {
                            const uint64_t bdesc = smem_desc_sw128(L.btile(a) + (kk >> 2) * 2048 + (kk & 3) * 32);
                            tc_mma(d, tmem + a * TC_A_COLS + kk * 8, bdesc, (m | kk) != 0 ? 1u : 0u);
                        }
                        tc_commit(L.afree(a));   // A/B buffer a is free once these MMAs complete
                    }
                    if (!ok)
                        break;
                    tc_commit(L.gfull(gs));   // accumulator gs is final once these complete
                    ++g;
                }
                u = e;
            }
            tc_commit(L.done());   // every MMA issued by this thread has completed
        }
        __syncwarp();
    } else if (warp < TC_CONV_WARPS) {
        // ---- converters: warp w owns tile rows 32 (w % 4) .. +31 (its TMEM lanes)
        // of unit h = w / 4 of each stage (whole 128-byte rows).  Both units of
        // a stage are read at once, so the stage goes back to the producer
        // after one round of loads.
        const int sub = warp & 3;
        const int h = warp >> 2;
        const int t = 32 * sub + lane;   // tile row
        const uint32_t tlane = (uint32_t)(32 * sub) << 16;
        const uint32_t xrow = (uint32_t)q.ups * TC_KU;   // bytes per activation row in a stage
        bool ok = true;
        int i = 0, j0 = 0;
        for (StageWalk sw(u0, u1, UB, q.ups); sw.more() && ok; ++i) {
            const int cnt = sw.count();
            const int s = i % S;
            if (!warp_wait(L, q, L.full(s), (i / S) & 1)) {
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
                xv = lds128(L.xtile(s) + (t >> 3) * xrow + h * TC_KU + (t & 7) * 16);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(L.empty(s));   // this warp is done with stage s
            if (mine) {
                const int j = j0 + h;
                const int a = j % NA;
                if (j >= NA && !warp_wait(L, q, L.afree(a), ((j / NA) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // A operand: 128 f16 of row t -> 64 TMEM columns of buffer a
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[16];
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int4 &w = wv[part * 2 + c2];
                        i8x4_to_f16x4((uint32_t)w.x, r[c2 * 8 + 0], r[c2 * 8 + 1]);
                        i8x4_to_f16x4((uint32_t)w.y, r[c2 * 8 + 2], r[c2 * 8 + 3]);
                        i8x4_to_f16x4((uint32_t)w.z, r[c2 * 8 + 4], r[c2 * 8 + 5]);
                        i8x4_to_f16x4((uint32_t)w.w, r[c2 * 8 + 6], r[c2 * 8 + 7]);
                    }
                    tc_st16(tmem + tlane + a * TC_A_COLS + part * 16, r);
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
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(L.aready(a));
            }
            j0 += cnt;
            sw.next(cnt);
        }
    } else {
        // ---- epilogue warps: accumulators -> int32 row sums -> outputs ------------
        const int sub = warp & 3;
        const int t = 32 * sub + lane;   // tile row
        const uint32_t tlane = (uint32_t)(32 * sub) << 16;
        const int64_t T = q.total_units;
        bool ok = true;
        int g = 0;
        for (int64_t u = u0; u < u1;) {
            const int64_t band = u / UB;
            const int64_t e = min(u1, (band + 1) * UB);
            int32_t isum[TC_N];
#pragma unroll
            for (int b = 0; b < TC_N; ++b)
                isum[b] = 0;
            for (int64_t gu = u; gu < e; gu += TC_UNITS_PER_GROUP, ++g) {
                if (!ok)
                    continue;
                const int gs = g % NG;
                if (!warp_wait(L, q, L.gfull(gs), (g / NG) & 1)) {
                    ok = false;
                    continue;
                }
                tc_fence_after();
                uint32_t v[16];
                tc_ld16(tmem + tlane + acc_col + gs * TC_ACC_COLS, v);
#pragma unroll
                for (int b = 0; b < TC_N; ++b)
                    isum[b] += __float2int_rn(__uint_as_float(v[b]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(L.gfree(gs));
            }
            const int64_t row = band * TC_M + t;
            const float sw = row < q.n_rows ? __ldg(q.scale_w + row) : 0.f;
            const bool whole = u == band * UB && e == (band + 1) * UB;
            if (whole) {
                store_row(q, L, row, sw, isum, ok && !aborted(L));
                u = e;
                continue;
            }
            // ---- a split band: store the partial sums, then count this CTA in
            const int64_t rec = 2 * cta + (u == u0 ? 0 : 1);
            char *rp = q.records + rec * TC_REC_BYTES;
            int4 *dst = reinterpret_cast<int4 *>(rp + TC_REC_HDR + t * TC_N * 4);
#pragma unroll
            for (int b = 0; b < TC_N; b += 4)
                __stcg(dst + b / 4, make_int4(isum[b], isum[b + 1], isum[b + 2], isum[b + 3]));
            const bool all_ok = epi_barrier_and(ok && !aborted(L));
            const int64_t cf = owner_of(band * UB, T, G);
            const int64_t cl = owner_of((band + 1) * UB - 1, T, G);
            if (warp == TC_EPI_WARP0 && lane == 0) {
                __stcg(reinterpret_cast<int4 *>(rp), make_int4(all_ok ? 1 : 0, 0, 0, 0));
                // the barrier above ordered every row's stores before this release
                const uint32_t before = arrive_counter(q.counters + cf);
                const uint32_t last = before == (uint32_t)(cl - cf) ? 1u : 0u;
                if (last)
                    q.counters[cf] = 0u;   // every contributor has counted in
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(L.last_flag()), "r"(last) : "memory");
            }
            epi_barrier();
            uint32_t last;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(last) : "r"(L.last_flag()));
            if (last) {
                // the last contributor adds every partial in CTA order
                int32_t total[TC_N];
#pragma unroll
                for (int b = 0; b < TC_N; ++b)
                    total[b] = 0;
                bool valid = true;
                if (e == u1 && all_ok) {
                    // this CTA's last segment (and no role gave up): its stage ring
                    // is idle, so every thread copies its row of each record (and
                    // one header) into it with cp.async, all in flight at once
                    const int cap = (int)((uint32_t)S * L.stage_bytes() / TC_REC_BYTES);
                    for (int64_t c0 = cf; c0 <= cl; c0 += cap) {
                        const int n = (int)min((int64_t)cap, cl - c0 + 1);
                        for (int m = 0; m < n; ++m) {
                            const int64_t c = c0 + m;
                            const int64_t r = 2 * c + (part_begin(q, c, G) / UB == band ? 0 : 1);
                            const char *src = q.records + r * TC_REC_BYTES;
                            const uint32_t at = L.base + (uint32_t)m * TC_REC_BYTES;
#pragma unroll
                            for (int b = 0; b < TC_N; b += 4)
                                cp_async16(at + TC_REC_HDR + (t * TC_N + b) * 4, src + TC_REC_HDR + (t * TC_N + b) * 4);
                            if (t == 0)
                                cp_async16(at, src);
                        }
                        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
                        epi_barrier();   // every thread's copies have landed
                        for (int m = 0; m < n; ++m) {
                            const uint32_t at = L.base + (uint32_t)m * TC_REC_BYTES;
                            uint32_t hdr;
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(hdr) : "r"(at));
                            valid &= hdr != 0;
#pragma unroll
                            for (int b = 0; b < TC_N; b += 4) {
                                const int4 v4 = lds128(at + TC_REC_HDR + (t * TC_N + b) * 4);
                                total[b] += v4.x;
                                total[b + 1] += v4.y;
                                total[b + 2] += v4.z;
                                total[b + 3] += v4.w;
                            }
                        }
                        epi_barrier();   // the ring is read before the next round lands
                    }
                } else {
                    for (int64_t c = cf; c <= cl; ++c) {
                        const int64_t r = 2 * c + (part_begin(q, c, G) / UB == band ? 0 : 1);
                        const char *src = q.records + r * TC_REC_BYTES;
                        const int hdr = __ldcg(reinterpret_cast<const int *>(src));
                        const int4 *sp = reinterpret_cast<const int4 *>(src + TC_REC_HDR + t * TC_N * 4);
#pragma unroll
                        for (int b = 0; b < TC_N; b += 4) {
                            const int4 v4 = __ldcg(sp + b / 4);
                            total[b] += v4.x;
                            total[b + 1] += v4.y;
                            total[b + 2] += v4.z;
                            total[b + 3] += v4.w;
                        }
                        valid &= hdr != 0;
                    }
                }
                store_row(q, L, row, sw, total, valid);
            }
            u = e;
        }
    }

    // ---- teardown: tensor memory is freed only after every MMA has completed
    tc_fence_before();
    __syncthreads();
    if (warp == TC_PRODUCER_WARP) {
        if (lane == 0)
            dev::mbar_wait_bounded(L.done(), 0, q.wait_ns);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(q.tmem_cols)
                     : "memory");
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

bool encode_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
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

// Shared memory per CTA, sized so that every CTA resident on an SM finds its
// tensor memory free (tcgen05.alloc would otherwise wait for another CTA to
// finish): with 256 columns each CTA asks for more than a third of the SM's
// shared memory (at most two CTAs, which together fit the 512 columns); with
// 512 columns, for more than half (one CTA per SM).
constexpr uint32_t TC_MIN_SMEM_2 = 80u * 1024u;
constexpr uint32_t TC_MAX_SMEM_2 = 113u * 1024u;
constexpr uint32_t TC_MIN_SMEM_1 = 120u * 1024u;
constexpr uint32_t TC_MAX_SMEM_1 = 227u * 1024u;


int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }

}  // namespace

bool dot_tc_eligible(bool aligned, int32_t k, int32_t batch_pass)
{
    return aligned && k >= 16 && (k % 16) == 0 && batch_pass >= 1 && batch_pass <= TC_N;
}

int dot_tc_threads() { return TC_THREADS; }

int dot_tc_rows_per_band() { return TC_M; }

// Resolve the schedule of one tensor-core launch.  cfg fields of 0 take the
// defaults: two CTAs per SM, two units per stage, two stages, three A
// buffers (the remaining tensor memory holds the accumulators).
bool dot_tc_plan(int64_t n_rows, int32_t k, int64_t sm_count, const DotTcConfig &cfg, bool split,
                 DotTcPlan *out)
{
    const int cps = cfg.ctas_per_sm ? cfg.ctas_per_sm : 2;
    const int ups = cfg.units_per_stage ? cfg.units_per_stage : 2;
    if ((cps != 1 && cps != 2) || ups < 1 || ups > TC_MAX_UPS || sm_count < 1)
        return false;
    const int depth = cfg.depth ? cfg.depth : (ups == 2 ? 2 : 4);
    const uint32_t cols = cps == 2 ? 256u : 512u;
    const int na = cfg.a_bufs ? cfg.a_bufs : (cps == 2 ? 3 : 4);
    // two converter groups fill consecutive units at once: with one A buffer a
    // group could wait on a barrier phase two ahead of the last it saw
    if (depth < 1 || depth > LOOM_MAX_DEPTH || na < 2 || (uint32_t)na * TC_A_COLS + 2 * TC_ACC_COLS > cols)
        return false;
    int ng = (int)((cols - (uint32_t)na * TC_A_COLS) / TC_ACC_COLS);
    ng = ng > TC_MAX_ACC ? TC_MAX_ACC : ng;
    uint32_t smem = tc_smem_bytes(depth, ups, na, ng);
    const uint32_t lo = cps == 2 ? TC_MIN_SMEM_2 : TC_MIN_SMEM_1;
    const uint32_t hi = cps == 2 ? TC_MAX_SMEM_2 : TC_MAX_SMEM_1;
    if (smem > hi)
        return false;
    smem = smem < lo ? lo : smem;
    const int64_t bands = (n_rows + TC_M - 1) / TC_M;
    const int32_t ub = (k + TC_KU - 1) / TC_KU;
    const int64_t total = bands * ub;
    const int32_t quantum = split ? 1 : ub;
    const int64_t steps = total / quantum;
    const int64_t slots = (int64_t)cps * sm_count;
    out->grid = steps < slots ? steps : slots;
    out->quantum = quantum;
    out->units_per_band = ub;
    out->total_units = total;
    out->depth = depth;
    out->ups = ups;
    out->na = na;
    out->ng = ng;
    out->tmem_cols = cols;
    out->smem_bytes = smem;
    out->split = split;
    out->sm_count = sm_count;
    return true;
}

// Workspace of a split launch: arrival counters for the largest grid the
// device runs (two CTAs per SM) at offset 0 -- a fixed place, so calls of
// any shape find them at zero -- then two partial-sum records (validity
// header + sums) per CTA of this grid, rewritten by every call.
static int64_t tc_counter_bytes(int64_t sm_count) { return align256(2 * sm_count * 4); }

int64_t dot_tc_workspace_bytes(const DotTcPlan &plan)
{
    return tc_counter_bytes(plan.sm_count) + align256(plan.grid * 2 * (int64_t)TC_REC_BYTES);
}

cudaError_t launch_dot_tc(const DotParams &p, const DotTcPlan &plan, cudaStream_t stream)
{
    if (plan.grid == 0)
        return cudaSuccess;
    const int64_t k = (int64_t)p.k_words * 4;
    CUtensorMap tmw, tmx;
    if (!encode_2d_u8(&tmw, p.w, (uint64_t)k, (uint64_t)p.n_rows, TC_KU, TC_M, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d_u8(&tmx, p.x, (uint64_t)k, (uint64_t)p.batch, (uint32_t)(TC_KU * plan.ups), TC_N,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcParams q;
    q.scale_w = p.scale_w;
    q.scale_x = p.scale_x;
    q.y = p.y;
    q.acc = p.acc;
    q.error = p.error;
    q.counters = nullptr;
    q.records = nullptr;
    if (plan.split) {
        if (!p.workspace || p.workspace_bytes < dot_tc_workspace_bytes(plan))
            return cudaErrorInvalidValue;
        char *ws = static_cast<char *>(p.workspace);
        q.counters = reinterpret_cast<uint32_t *>(ws);
        q.records = ws + tc_counter_bytes(plan.sm_count);
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
    q.tmem_cols = plan.tmem_cols;
    q.wait_ns = p.wait_ns;
    q.inject_stall = p.inject_stall;

    cudaError_t e = cudaFuncSetAttribute(dot_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem_bytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, dot_tc_kernel, tmw, tmx, q);
}

}  // namespace loom
