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
//    integer.  The eight K = 16 slices of a stage go to eight separate f32
//    accumulators (so consecutive MMAs are independent), and a block of 64
//    stages shares one set of eight: each accumulator then sums 64 x 16 =
//    1024 products.  The accumulators are converted to int32 and added in the
//    epilogue, so the int32 result is exact.
//  * Conversion int8 -> f16 is exact and cheap: a byte b becomes the f16 bit
//    pattern 0x6400 | (b + 128) (the value 1024 + b + 128) by a byte permute,
//    and one packed f16 subtraction of 1152 leaves b.
//  * The weights stream once: a 2-D TMA copy brings a 128-row x 128-byte
//    tile (128-byte swizzle) into a ring of `depth` shared-memory stages.
//    Eight converter warps -- two per tensor-memory sub-partition, each half
//    of every row -- read their bytes (the swizzle keeps the reads
//    conflict-free), convert, and write the f16 operand straight into tensor
//    memory with tcgen05.st: the A operand never goes back
//    through shared memory, so shared-memory traffic stays at two bytes per
//    weight byte.  The activation tile is converted into a 128-byte-swizzled
//    K-major f16 tile in shared memory (the B operand).
//  * One thread issues the MMAs; tcgen05.commit releases the A/B buffers and
//    finally signals the epilogue.
//  * Each 128-row tile is split along k over a cluster of four CTAs (two for
//    short k; 256 CTAs for 8192 rows, two per SM, whose pipelines overlap);
//    the other CTAs hand their int32 partial sums to the first through
//    distributed shared memory, which adds them in rank order and applies the
//    scales.  No global scratch, no atomics, deterministic.
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT,
//    the kernel skips the remaining work, still meets every cluster barrier,
//    lets issued copies and MMAs finish, frees its tensor memory and writes
//    NaN results.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

constexpr int TC_M = 128;                  // rows per tile (MMA M)
constexpr int TC_N = 16;                   // vectors per pass (MMA N)
constexpr int TC_KS = 128;                 // k (bytes) per stage
constexpr int TC_KSLICES = TC_KS / 16;     // MMAs per stage (K = 16 each)
constexpr int TC_STAGES_PER_BLOCK = 64;    // stages whose products share accumulators
constexpr int TC_CONV_WARPS = 8;           // two per TMEM sub-partition, each half a row
constexpr int TC_PRODUCER_WARP = TC_CONV_WARPS;
constexpr int TC_MMA_WARP = TC_CONV_WARPS + 1;
constexpr int TC_THREADS = 32 * (TC_CONV_WARPS + 2);
constexpr uint32_t TC_W_BYTES = TC_M * TC_KS;          // 16 KiB
constexpr uint32_t TC_X_BYTES = TC_N * TC_KS;          // 2 KiB
constexpr uint32_t TC_STAGE_BYTES = TC_W_BYTES + TC_X_BYTES;   // 18 KiB (1024-aligned)
constexpr uint32_t TC_B_BYTES = TC_N * TC_KS * 2;      // f16 activation tile, 4 KiB
constexpr uint32_t TC_RED_BYTES = TC_M * TC_N * 4;     // int32 partials of one peer CTA
constexpr uint32_t TC_A_COLS = 64;                     // TMEM columns of one f16 A buffer
// instruction descriptor: D f32, A/B f16, both K-major, N = 16, M = 128
constexpr uint32_t TC_IDESC = (1u << 4) | ((TC_N >> 3) << 17) | ((TC_M >> 4) << 24);

struct TcParams {
    const float *scale_w;
    const float *scale_x;
    float *y;
    int32_t *acc;
    int32_t *error;
    int32_t n_rows, batch, y_stride;
    int32_t stages_total;   // ceil(k / 128)
    int32_t depth;          // shared-memory stages
    int32_t a_bufs;         // f16 A buffers in tensor memory (2 or 4)
    uint32_t tmem_cols;
    uint64_t wait_ns;
    int32_t inject_stall;
};

// Bytes of the stage ring; it also holds the hand-over buffers at the end.
__host__ __device__ constexpr uint32_t tc_ring_bytes(int S, int peers)
{
    return ((uint32_t)S * TC_STAGE_BYTES > (uint32_t)peers * (TC_RED_BYTES + TC_M * 4))
               ? (uint32_t)S * TC_STAGE_BYTES
               : (((uint32_t)peers * (TC_RED_BYTES + TC_M * 4) + 1023u) & ~1023u);
}

struct Layout {
    uint32_t base;  // 1024-aligned shared address
    int S;
    int peers;      // cluster size - 1
    __device__ uint32_t stage(int s) const { return base + s * TC_STAGE_BYTES; }
    __device__ uint32_t btile(int a) const { return base + tc_ring_bytes(S, peers) + a * TC_B_BYTES; }
    // The hand-over buffers reuse the stage ring once every stage is consumed.
    __device__ uint32_t red() const { return base; }
    __device__ uint32_t red_ok() const { return red() + peers * TC_RED_BYTES; }
    __device__ uint32_t bars() const { return base + tc_ring_bytes(S, peers) + 2 * TC_B_BYTES; }
    __device__ uint32_t full(int s) const { return bars() + 8 * s; }
    __device__ uint32_t empty(int s) const { return bars() + 8 * (S + s); }
    __device__ uint32_t aready(int a) const { return bars() + 8 * (2 * S + a); }
    __device__ uint32_t afree(int a) const { return bars() + 8 * (2 * S + 4 + a); }
    __device__ uint32_t done() const { return bars() + 8 * (2 * S + 8); }
    __device__ uint32_t tmem_slot() const { return bars() + 8 * (2 * S + 9); }
    __device__ uint32_t abort_flag() const { return tmem_slot() + 4; }
};

uint32_t tc_smem_bytes(int S, int cs)
{
    return 1024 + tc_ring_bytes(S, cs - 1) + 2 * TC_B_BYTES + 8 * (2 * S + 9) + 16;
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

template <int CS>
__global__ void __launch_bounds__(TC_THREADS, 1)
    dot_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                  const TcParams q)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = dev::smem_u32(smem_raw);
    Layout L;
    L.base = (raw + 1023u) & ~1023u;
    L.S = q.depth;
    L.peers = CS - 1;
    const int S = q.depth;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int32_t row0 = (int32_t)(blockIdx.x / CS) * TC_M;
    const int32_t per_rank = (q.stages_total + CS - 1) / CS;
    const int32_t s_begin = (int32_t)rank * per_rank;
    const int32_t ns = max(0, min(q.stages_total, s_begin + per_rank) - s_begin);
    const int ng = TC_KSLICES * ((ns + TC_STAGES_PER_BLOCK - 1) / TC_STAGES_PER_BLOCK);   // accumulators

    // ---- set-up: barriers, abort flag, tensor memory --------------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            dev::mbar_init(L.full(s), 1);
            dev::mbar_init(L.empty(s), TC_CONV_WARPS);
        }
        for (int a = 0; a < 4; ++a) {
            dev::mbar_init(L.aready(a), TC_CONV_WARPS);
            dev::mbar_init(L.afree(a), 1);
        }
        dev::mbar_init(L.done(), 1);
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(L.abort_flag()) : "memory");
        dev::fence_barrier_init();
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
    cluster_sync();   // both CTAs of the pair are running before any remote access
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(L.tmem_slot()));
    const int NA = q.a_bufs;
    const uint32_t acc_col = NA * TC_A_COLS;

    bool ok = true;   // this thread's role finished its part
    int32_t isum[TC_N];
#pragma unroll
    for (int b = 0; b < TC_N; ++b)
        isum[b] = 0;

    if (warp == TC_PRODUCER_WARP) {
        // ---- producer: 2-D TMA of the weight and activation tiles ------------
        int issued = 0;
        if (lane == 0) {
            const uint64_t wpol = dev::l2_evict_first_policy();
            const uint64_t xpol = dev::l2_evict_last_policy();
            for (int i = 0; i < ns; ++i) {
                const int s = i % S;
                if (i >= S && !dev::mbar_wait_bounded(L.empty(s), ((i / S) - 1) & 1, q.wait_ns)) {
                    set_abort(L, q);
                    break;
                }
                if (aborted(L))
                    break;
                if (!q.inject_stall) {
                    const int32_t kx = (s_begin + i) * TC_KS;
                    dev::mbar_arrive_expect_tx(L.full(s), TC_STAGE_BYTES);
                    tma_load_2d(L.stage(s), &tmw, kx, row0, L.full(s), wpol);
                    tma_load_2d(L.stage(s) + TC_W_BYTES, &tmx, kx, 0, L.full(s), xpol);
                    ++issued;
                }
            }
            // every copy issued must land before the CTA may leave (bounded)
            for (int i = max(0, issued - S); i < issued; ++i)
                dev::mbar_wait_bounded(L.full(i % S), (i / S) & 1, q.wait_ns);
        }
        __syncwarp();
    } else if (warp == TC_MMA_WARP) {
        // ---- MMA issuer ----------------------------------------------------------
        if (lane == 0) {
            for (int i = 0; i < ns; ++i) {
                const int a = i % NA;
                if (!dev::mbar_wait_bounded(L.aready(a), (i / NA) & 1, q.wait_ns) || aborted(L)) {
                    set_abort(L, q);
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + acc_col + TC_N * TC_KSLICES * (i / TC_STAGES_PER_BLOCK);
                const uint32_t accumulate = (i % TC_STAGES_PER_BLOCK) == 0 ? 0u : 1u;
#pragma unroll
                for (int kk = 0; kk < TC_KSLICES; ++kk) {
                    const uint64_t bdesc = smem_desc_sw128(L.btile(a) + (kk >> 2) * 2048 + (kk & 3) * 32);
                    tc_mma(d0 + TC_N * kk, tmem + a * TC_A_COLS + kk * 8, bdesc, accumulate);
                }
                tc_commit(L.afree(a));   // A/B buffer a is free once these MMAs complete
            }
            tc_commit(L.done());   // all MMAs issued by this thread complete
        }
        __syncwarp();
    } else {
        // ---- converters: warp w owns tile rows 32 (w % 4) .. +31 (its TMEM lanes)
        // and half h = w / 4 of each row's 128 bytes; warps with h = 0 also
        // convert the activation tile.
        const int sub = warp & 3;
        const int h = warp >> 2;
        const int t = 32 * sub + lane;   // tile row
        const uint32_t tlane = (uint32_t)(32 * sub) << 16;
        for (int i = 0; i < ns; ++i) {
            const int s = i % S;
            const int a = i % NA;
            bool w_ok = dev::mbar_wait_bounded(L.full(s), (i / S) & 1, q.wait_ns);
            if (w_ok && i >= NA)
                w_ok = dev::mbar_wait_bounded(L.afree(a), ((i / NA) - 1) & 1, q.wait_ns);
            if (!__all_sync(dev::FULL_MASK, w_ok) || aborted(L)) {
                ok = false;
                break;
            }
            // half a weight row (64 bytes, 128-byte swizzle) and, for h = 0, a 16-byte
            // piece of the activations
            int4 wv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                wv[c] = lds128(L.stage(s) + t * 128 + (((4 * h + c) ^ (t & 7)) << 4));
            int4 xv = make_int4(0, 0, 0, 0);
            if (h == 0)
                xv = lds128(L.stage(s) + TC_W_BYTES + t * 16);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(L.empty(s));   // this warp is done with stage s
            // A operand: 64 f16 of row t -> 32 TMEM columns of buffer a
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t r[16];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int4 &w = wv[part * 2 + c2];
                    i8x4_to_f16x4((uint32_t)w.x, r[c2 * 8 + 0], r[c2 * 8 + 1]);
                    i8x4_to_f16x4((uint32_t)w.y, r[c2 * 8 + 2], r[c2 * 8 + 3]);
                    i8x4_to_f16x4((uint32_t)w.z, r[c2 * 8 + 4], r[c2 * 8 + 5]);
                    i8x4_to_f16x4((uint32_t)w.w, r[c2 * 8 + 6], r[c2 * 8 + 7]);
                }
                tc_st16(tmem + tlane + a * TC_A_COLS + 32 * h + part * 16, r);
            }
            // B operand: activations of vector n = t / 8, k = 16 (t % 8) .. +15, into
            // the K-major 128-byte-swizzled f16 tile (two 64-k atoms of 16 rows).
            if (h == 0) {
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
        // ---- epilogue part 1 (warps with h = 0): the f32 groups to int32 --------
        bool done_ok = ok && h == 0 && dev::mbar_wait_bounded(L.done(), 0, q.wait_ns);
        done_ok = __all_sync(dev::FULL_MASK, done_ok);
        if (done_ok && !aborted(L)) {
            tc_fence_after();
            for (int g = 0; g < ng; ++g) {
                uint32_t v[16];
                tc_ld16(tmem + tlane + acc_col + TC_N * g, v);
#pragma unroll
                for (int b = 0; b < TC_N; ++b)
                    isum[b] += __float2int_rn(__uint_as_float(v[b]));
            }
        } else if (h == 0) {
            ok = false;
        }
        if (!ok)
            set_abort(L, q);
    }

    // Every CTA of the cluster is past its stage ring (and its copies have
    // landed) before the ring memory of the first CTA receives the partials.
    tc_fence_before();
    cluster_sync();
    if (warp < TC_CONV_WARPS) {
        const int h = warp >> 2;
        const int t = 32 * (warp & 3) + lane;
        // the other CTAs of the cluster hand their partial sums to the first
        if (rank >= 1 && h == 0) {
            const uint32_t dst = map_to_rank(L.red() + (rank - 1) * TC_RED_BYTES + t * TC_N * 4, 0);
#pragma unroll
            for (int b = 0; b < TC_N; b += 4)
                st_cluster_v4(dst + b * 4, isum[b], isum[b + 1], isum[b + 2], isum[b + 3]);
            const uint32_t okdst = map_to_rank(L.red_ok() + (rank - 1) * TC_M * 4 + t * 4, 0);
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(okdst), "r"(ok && !aborted(L) ? 1u : 0u)
                         : "memory");
        }
    }

    // ---- hand-over and teardown ---------------------------------------------------
    tc_fence_before();
    cluster_sync();   // partial sums of rank 1 are visible in rank 0's shared memory
    tc_fence_after();
    if (rank == 0 && threadIdx.x < TC_M) {
        const int t = threadIdx.x;
        bool valid = ok && !aborted(L);
#pragma unroll
        for (int r = 0; r < CS - 1; ++r) {
            uint32_t peer_ok;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(peer_ok) : "r"(L.red_ok() + r * TC_M * 4 + t * 4));
            valid = valid && peer_ok != 0;
        }
        const int32_t row = row0 + t;
        if (row < q.n_rows) {
            const float sw = __ldg(q.scale_w + row);
#pragma unroll
            for (int b = 0; b < TC_N; ++b) {
                if (b < q.batch) {
                    int32_t total = isum[b];   // peers added in rank order
#pragma unroll
                    for (int r = 0; r < CS - 1; ++r) {
                        uint32_t other;
                        asm volatile("ld.shared.u32 %0, [%1];"
                                     : "=r"(other)
                                     : "r"(L.red() + r * TC_RED_BYTES + (t * TC_N + b) * 4));
                        total += (int32_t)other;
                    }
                    const int64_t o = (int64_t)row * q.y_stride + b;
                    q.y[o] = valid ? __fmul_rn(__int2float_rn(total), __fmul_rn(sw, __ldg(q.scale_x + b)))
                                   : __int_as_float(0x7fc00000);
                    if (q.acc)
                        q.acc[o] = valid ? total : INT32_MIN;
                }
            }
        }
    }
    // tensor memory is freed only after every MMA of this CTA has completed
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

// Cluster size: four CTAs share a tile's k when each still gets a long
// stream (two CTAs per SM then overlap their pipelines), else two.
int tc_cluster(int32_t k) { return (k + TC_KS - 1) / TC_KS >= 64 ? 4 : 2; }

// f32 accumulators of one CTA (16 columns each)
int32_t tc_groups(int32_t k)
{
    const int32_t stages = (k + TC_KS - 1) / TC_KS;
    const int cs = tc_cluster(k);
    const int32_t per_rank = (stages + cs - 1) / cs;
    return TC_KSLICES * ((per_rank + TC_STAGES_PER_BLOCK - 1) / TC_STAGES_PER_BLOCK);
}

// Two A buffers: conversion of stage i + 1 overlaps the MMAs of stage i
// (four measured slower on GB300: the 512-column allocation it needs costs
// more than the extra overlap buys).
int tc_a_bufs(int32_t) { return 2; }

uint32_t tc_tmem_cols(int32_t k)
{
    return tc_a_bufs(k) * TC_A_COLS + TC_N * tc_groups(k) <= 256 ? 256u : 512u;
}

// Shared memory per CTA, sized so that every CTA resident on an SM finds its
// tensor memory free: a CTA that would wait in tcgen05.alloc while holding a
// cluster partner at a cluster barrier elsewhere could close a cycle of
// waits.  With 256 columns each CTA asks for more than a third of the SM's
// shared memory (at most two CTAs, which together fit the 512 columns); with
// 512 columns, for more than half (one CTA per SM).
constexpr uint32_t TC_MIN_SMEM_256 = 80u * 1024u;
constexpr uint32_t TC_MIN_SMEM_512 = 120u * 1024u;

}  // namespace

bool dot_tc_eligible(bool aligned, int32_t k, int32_t batch_pass)
{
    if (!aligned || k < 16 || (k % 16) != 0 || batch_pass < 1 || batch_pass > TC_N)
        return false;
    return 2 * TC_A_COLS + TC_N * tc_groups(k) <= 512;
}

uint32_t dot_tc_smem_bytes(int depth, int32_t k)
{
    const uint32_t b = tc_smem_bytes(depth, tc_cluster(k));
    const uint32_t floor = tc_tmem_cols(k) == 512u ? TC_MIN_SMEM_512 : TC_MIN_SMEM_256;
    return b > floor ? b : floor;
}

int dot_tc_rows_per_cluster() { return TC_M; }

int dot_tc_cluster(int32_t k) { return tc_cluster(k); }

cudaError_t launch_dot_tc(const DotParams &p, const loom_launch &L, cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    const int64_t k = (int64_t)p.k_words * 4;
    CUtensorMap tmw, tmx;
    if (!encode_2d_u8(&tmw, p.w, (uint64_t)k, (uint64_t)p.n_rows, TC_KS, TC_M, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d_u8(&tmx, p.x, (uint64_t)k, (uint64_t)p.batch, TC_KS, TC_N, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    TcParams q;
    q.scale_w = p.scale_w;
    q.scale_x = p.scale_x;
    q.y = p.y;
    q.acc = p.acc;
    q.error = p.error;
    q.n_rows = p.n_rows;
    q.batch = p.batch;
    q.y_stride = p.y_stride;
    q.stages_total = (int32_t)((k + TC_KS - 1) / TC_KS);
    q.depth = p.depth;
    q.a_bufs = tc_a_bufs((int32_t)k);
    q.tmem_cols = tc_tmem_cols((int32_t)k);
    if (L.smem_bytes < (q.tmem_cols == 512u ? TC_MIN_SMEM_512 : TC_MIN_SMEM_256))
        return cudaErrorInvalidValue;   // too many CTAs per SM for the tensor memory
    q.wait_ns = p.wait_ns;
    q.inject_stall = p.inject_stall;

    const int cs = tc_cluster((int32_t)k);
    auto kernel = cs == 4 ? dot_tc_kernel<4> : dot_tc_kernel<2>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid[0], 1, 1);
    cfg.blockDim = dim3(L.block[0], 1, 1);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((int)L.cluster[0] != cs)
        return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, kernel, tmw, tmx, q);
}

}  // namespace loom
