// dot_tc_rows.cu -- batched dequantised dot products on the 5th-generation
// tensor cores with each CTA owning whole rows of W (tcgen05, sm_103a).
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section "Apply
// the same controls to a packed dot product"): packed signed bytes are
// unpacked and accumulated as dot products; here weights W[n_rows][k] and up
// to 16 activation vectors X[b][k], int32 accumulation, per-row and
// per-vector scales in the epilogue:
//   acc[r][b] = sum_k W[r][k] X[b][k],   y[r][b] = (float)acc[r][b] * (sw[r] * sx[b]).
//
// Design
//  * A persistent grid of at most one CTA per SM.  CTA c owns rows
//    [c RPC, (c + 1) RPC) for the whole of k, RPC = ceil(n_rows / SMs) (8192
//    rows on 152 SMs: 54 each), so every row's sum is finished inside one CTA:
//    no partial sums go through global memory and no second kernel runs.  A
//    CTA takes its rows in blocks of at most 64.
//  * The MMA's 128 tensor-memory lanes (M = 128) carry a block twice: lanes
//    0..63 its rows over one k range, lanes 64..127 the same rows over
//    another.  The B operand has 32 columns, the 16 vectors over the first
//    range and then over the second; of a lane's 32 accumulator columns the
//    16 of its own range are the wanted sums, the other 16 (cross terms) are
//    never read.  k is cut into two halves of whole 128-byte units, one per
//    pipeline of the CTA; a stage of a pipeline holds two neighbouring units
//    of its half, the first for lanes 0..63 and the second for lanes 64..127
//    (each row then reads 256 contiguous bytes per stage), so over the stages
//    each lane half sums every other unit of the pipeline's half.
//  * A pipeline: a producer thread (per stage, 2-D TMA copies of the two
//    128-byte units of k of the block's rows, 128-byte swizzle, and the two
//    matching 16 x 128-byte activation boxes); two converter
//    groups of four warps taking alternate stages (each thread one tensor-
//    memory lane: int8 -> f16 of one row's 128 bytes into tensor memory with
//    tcgen05.st, and two 16-byte pieces of activations into the 128-byte-
//    swizzled K-major f16 B tile); an MMA thread (tcgen05.mma kind::f16,
//    M 128, N 32, K 16, A from tensor memory, B by descriptor); four
//    epilogue warps.
//  * Exactness: int8 -> f16 is exact; one f32 accumulator sums the products
//    of at most eight units (1024 per element, |sum| <= 2^24, where f32 holds
//    every integer); the epilogue converts each finished accumulator to int32
//    and adds it to its running sums, so acc is exact for any k.
//  * At the end of a block the eight epilogue warps of the CTA put their
//    int32 sums of the four parts of k (two pipelines x two lane halves) in
//    shared memory; each row's four are added, scaled and stored.
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT,
//    every role stops at its next wait, issued copies and MMAs are allowed to
//    finish, tensor memory is freed and the affected outputs are NaN (acc
//    INT32_MIN).
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace loom {
namespace {

constexpr int RB_MAX_ROWS = 64;                 // rows per block: half the lanes
constexpr int RB_VEC = 16;                      // vectors per pass
constexpr int RB_N = 2 * RB_VEC;                // MMA N: the vectors over two k ranges
constexpr int RB_KU = 128;                      // k (bytes) per unit
constexpr int RB_KSLICES = RB_KU / 16;          // MMAs per unit (K = 16 each)
constexpr int RB_UNITS_PER_GROUP = 8;           // units per f32 accumulator: 8 x 128 products
constexpr int RB_GROUPS = 2;                    // converter groups per pipeline (alternate stages)
constexpr int RB_PIPES = 2;
constexpr int RB_EPI_WARPS = 4;
constexpr int RB_PIPE_WARPS = 4 * RB_GROUPS + RB_EPI_WARPS + 2;   // + producer, MMA issuer
constexpr int RB_THREADS = 32 * RB_PIPES * RB_PIPE_WARPS;
constexpr uint32_t RB_TMEM_COLS = 512;          // the whole SM: one CTA per SM
constexpr uint32_t RB_PIPE_COLS = RB_TMEM_COLS / RB_PIPES;
constexpr uint32_t RB_A_COLS = 64;              // one f16 A buffer: 128 k per lane
constexpr uint32_t RB_ACC_COLS = RB_N;          // one f32 accumulator
constexpr uint32_t RB_X_BOX = RB_VEC * RB_KU;   // 2 KiB of activations per range and unit
constexpr uint32_t RB_B_BYTES = RB_N * RB_KU * 2;   // f16 B tile of one stage, 8 KiB
constexpr uint32_t RB_B_KBLOCK = RB_N * 128;        // bytes of one 64-k block of the B tile
constexpr uint32_t RB_MERGE_BYTES = 4 * RB_MAX_ROWS * RB_VEC * 4;   // int32 [part of k][row][vector]
constexpr uint32_t RB_AREA = 1024;              // tensor-memory slot, abort word, vector scales
constexpr uint32_t RB_EPI_BAR = 1;              // named barrier of the CTA's eight epilogue warps
constexpr uint32_t RB_IDESC = tc::idesc_f16(128, RB_N);
constexpr uint32_t RB_MIN_SMEM = 120u * 1024u;  // more than half the SM: one CTA per SM
constexpr uint32_t RB_MAX_SMEM = 227u * 1024u;

struct RowsParams {
    const float *scale_w;
    const float *scale_x;
    float *y;
    int32_t *acc;
    int32_t *error;
    int32_t n_rows, batch, y_stride;
    int32_t rpc;          // rows per CTA
    int32_t br;           // rows per block (the weight boxes' height), <= 64
    int32_t uq;           // stages per block of each pipeline (two 128-byte units of k each)
    int32_t depth;        // shared-memory stages per pipeline (even)
    int32_t na, ng;       // f16 A buffers and f32 accumulators per pipeline
    uint32_t wbox;        // shared memory of one weight box (1024-aligned)
    uint32_t stage_bytes;
    uint32_t pipe_bytes;
    uint64_t wait_ns;
    int32_t inject_stall;
};

// Shared memory of one pipeline: stage ring, B tiles, barriers.
struct Pipe {
    uint32_t base;
    int S, na, ng;
    uint32_t wbox, stage_bytes;
    __device__ uint32_t stage(int s) const { return base + (uint32_t)s * stage_bytes; }
    __device__ uint32_t wtile(int s, int h) const { return stage(s) + (uint32_t)h * wbox; }
    __device__ uint32_t xtile(int s, int h) const { return stage(s) + 2 * wbox + (uint32_t)h * RB_X_BOX; }
    __device__ uint32_t btile(int a) const { return base + (uint32_t)S * stage_bytes + (uint32_t)a * RB_B_BYTES; }
    __device__ uint32_t bars() const { return btile(na); }
    __device__ uint32_t full(int s) const { return bars() + 8 * s; }
    __device__ uint32_t empty(int s) const { return bars() + 8 * (S + s); }
    __device__ uint32_t aready(int a) const { return bars() + 8 * (2 * S + a); }
    __device__ uint32_t afree(int a) const { return bars() + 8 * (2 * S + na + a); }
    __device__ uint32_t gfull(int g) const { return bars() + 8 * (2 * S + 2 * na + g); }
    __device__ uint32_t gfree(int g) const { return bars() + 8 * (2 * S + 2 * na + ng + g); }
    __device__ uint32_t done() const { return bars() + 8 * (2 * S + 2 * na + 2 * ng); }
    __device__ int n_bars() const { return 2 * S + 2 * na + 2 * ng + 1; }
    __device__ void bar_init(int i) const
    {
        uint32_t count = 1;                                        // full, afree, gfull, done
        if ((i >= S && i < 2 * S) || (i >= 2 * S && i < 2 * S + na))
            count = 4;                                             // empty, aready: a group's warps
        else if (i >= 2 * S + 2 * na + ng && i < 2 * S + 2 * na + 2 * ng)
            count = RB_EPI_WARPS;                                  // gfree
        dev::mbar_init(bars() + 8 * i, count);
    }
};

uint32_t rb_pipe_bytes(int S, int na, int ng, uint32_t stage_bytes)
{
    const uint32_t b = (uint32_t)S * stage_bytes + (uint32_t)na * RB_B_BYTES + 8u * (2 * S + 2 * na + 2 * ng + 1);
    return (b + 1023u) & ~1023u;
}

uint32_t rb_smem_bytes(uint32_t pipe_bytes) { return 1024u + RB_AREA + RB_MERGE_BYTES + RB_PIPES * pipe_bytes; }

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync %0, %1;" ::"n"(RB_EPI_BAR), "n"(32 * RB_PIPES * RB_EPI_WARPS) : "memory"); }

// bar.sync of the eight epilogue warps that also returns the AND of `v` over them.
__device__ __forceinline__ bool epi_barrier_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(RB_EPI_BAR), "n"(32 * RB_PIPES * RB_EPI_WARPS)
        : "memory");
    return r != 0;
}

// Where a 16-byte piece of activations -- 16 int8 of B row nn at k = 16 c8 of
// the unit -- goes as f16 in the K-major 128-byte-swizzled B tile: the row's
// offset in the tile and the offsets of its two 16-byte chunks within the row.
struct BPiece {
    uint32_t row, c0, c1;
    __device__ BPiece(int nn, int c8)
        : row((uint32_t)(c8 >> 2) * RB_B_KBLOCK + (uint32_t)(nn >> 3) * 1024 + (uint32_t)(nn & 7) * 128),
          c0((uint32_t)((2 * (c8 & 3)) ^ (nn & 7)) << 4), c1((uint32_t)((2 * (c8 & 3) + 1) ^ (nn & 7)) << 4)
    {
    }
};

__device__ __forceinline__ void put_b(uint32_t at, const BPiece &bp, const int4 &v)
{
    uint32_t h[8];
    tc::i8x4_to_f16x4((uint32_t)v.x, h[0], h[1]);
    tc::i8x4_to_f16x4((uint32_t)v.y, h[2], h[3]);
    tc::i8x4_to_f16x4((uint32_t)v.z, h[4], h[5]);
    tc::i8x4_to_f16x4((uint32_t)v.w, h[6], h[7]);
    tc::sts128(at + bp.c0, h[0], h[1], h[2], h[3]);
    tc::sts128(at + bp.c1, h[4], h[5], h[6], h[7]);
}

__global__ void __launch_bounds__(RB_THREADS, 1)
    dot_tc_rows_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                       const RowsParams q)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t tmem_slot = base, abort_word = base + 4, sx_at = base + 64;
    const uint32_t merge = base + RB_AREA;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int p = warp / RB_PIPE_WARPS;      // pipeline
    const int w = warp % RB_PIPE_WARPS;      // role within it
    const int sub = warp & 3;                // this warp's tensor-memory lanes: 32 sub .. 32 sub + 31
    constexpr int EPI0 = 4 * RB_GROUPS;
    constexpr int PRODUCER = EPI0 + RB_EPI_WARPS;
    constexpr int MMA = PRODUCER + 1;
    const uint32_t pipes0 = base + RB_AREA + RB_MERGE_BYTES;
    Pipe P{pipes0 + (uint32_t)p * q.pipe_bytes, q.depth, q.na, q.ng, q.wbox, q.stage_bytes};
    const int S = q.depth, NA = q.na, NG = q.ng, UQ = q.uq, BR = q.br;
    // this CTA's rows, its blocks, and each pipeline's stages (one unit of k of a block each)
    const int32_t r0 = (int32_t)blockIdx.x * q.rpc;
    const int32_t rc = min(q.rpc, q.n_rows - r0);
    const int nblk = (rc + BR - 1) / BR;
    const int J = nblk * UQ;
    const int32_t kp = p * (2 * UQ) * RB_KU;     // first byte of k of this pipeline's half

    // ---- set-up: barriers, flags, tensor memory ------------------------------
    // Each producer initialises its pipeline's barriers and at once issues the
    // copies of its first stages, so the weights are on their way while the
    // rest of the CTA sets up.  Only the producers' copies and the epilogue's
    // scale loads and stores touch global memory, each after the previous
    // kernel on the stream has completed (wait_previous_kernel).
    const uint64_t wpol = dev::l2_evict_first_policy();
    const uint64_t xpol = dev::l2_evict_last_policy();   // activations: re-read by every CTA
    // The producer's cursor: slot, block and unit of the next stage.  Every
    // role walks the stages with counters like these (no division per stage).
    int ps = 0, pb = 0, pu = 0;
    auto issue_next = [&]() {
        const int32_t k0 = kp + 2 * pu * RB_KU;   // the stage's two units of k, side by side
        const int32_t row = r0 + pb * BR;
        if (!q.inject_stall) {
            dev::mbar_arrive_expect_tx(P.full(ps), 2u * (uint32_t)BR * RB_KU + 2u * RB_X_BOX);
            tc::tma_load_2d(P.wtile(ps, 0), &tmw, k0, row, P.full(ps), wpol);
            tc::tma_load_2d(P.wtile(ps, 1), &tmw, k0 + RB_KU, row, P.full(ps), wpol);
            tc::tma_load_2d(P.xtile(ps, 0), &tmx, k0, 0, P.full(ps), xpol);
            tc::tma_load_2d(P.xtile(ps, 1), &tmx, k0 + RB_KU, 0, P.full(ps), xpol);
        }
        if (++pu == UQ) {
            pu = 0;
            ++pb;
        }
        if (++ps == S)
            ps = 0;
    };
    int issued = 0;
    if (w == PRODUCER) {
        if (lane == 0) {
            tc::prefetch_map(&tmw);
            tc::prefetch_map(&tmx);
        }
        for (int i = lane; i < P.n_bars(); i += 32)
            P.bar_init(i);
        dev::fence_barrier_init();
        __syncwarp();
        dev::wait_previous_kernel();
        if (lane == 0)
            for (int j = 0; j < S && j < J; ++j) {
                issue_next();
                issued += q.inject_stall ? 0 : 1;
            }
    }
    if (threadIdx.x == 0)
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(abort_word) : "memory");
    if (p == 0 && w == PRODUCER) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(RB_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    uint32_t tmem;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tmem_slot));
    tmem += (uint32_t)p * RB_PIPE_COLS;   // this pipeline's columns
    const uint32_t acc_col = (uint32_t)NA * RB_A_COLS;
    const uint32_t tl = (uint32_t)(32 * sub) << 16;   // this warp's lanes in a tensor-memory address
    const int L = 32 * sub + lane;                     // this thread's lane
    const int half = L >> 6;                           // lanes 0..63: a stage's first unit, 64..127: its second
    const int r = L & 63;                              // row within the block

    if (w == PRODUCER) {
        // ---- producer: the stages past the first S as the converters free them ----
        if (lane == 0) {
            uint32_t eph = 0;   // parity of the converters' release of slot ps: ((j / S) - 1) & 1
            for (int j = S; j < J; ++j) {
                if (!tc::role_wait(abort_word, q.error, q.wait_ns, P.empty(ps), eph))
                    break;
                issue_next();
                issued += q.inject_stall ? 0 : 1;
                if (ps == 0)
                    eph ^= 1u;
            }
            // every copy issued must land before the CTA may leave (bounded)
            for (int j = issued > S ? issued - S : 0; j < issued; ++j)
                dev::mbar_wait_bounded(P.full(j % S), (j / S) & 1, q.wait_ns);
        }
        __syncwarp();
    } else if (w == MMA) {
        // ---- MMA issuer: accumulator gs takes up to eight stages of one block ----
        if (lane == 0) {
            const uint64_t bdesc0 = tc::smem_desc_sw128(P.btile(0));
            int a = 0, gs = 0;
            uint32_t aph = 0, gph = 0;
            int g = 0;
            bool ok = true;
            for (int b = 0; b < nblk && ok; ++b) {
                for (int u0 = 0; u0 < UQ; u0 += RB_UNITS_PER_GROUP, ++g) {
                    if (g >= NG && !tc::role_wait(abort_word, q.error, q.wait_ns, P.gfree(gs), gph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const int n_in = min(RB_UNITS_PER_GROUP, UQ - u0);
                    const uint32_t d = tmem + acc_col + (uint32_t)gs * RB_ACC_COLS;
                    for (int m = 0; m < n_in; ++m) {
                        if (!tc::role_wait(abort_word, q.error, q.wait_ns, P.aready(a), aph)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)a * RB_B_BYTES) >> 4);
                        const uint32_t ta = tmem + (uint32_t)a * RB_A_COLS;
#pragma unroll
                        for (int kk = 0; kk < RB_KSLICES; ++kk)
                            tc::mma_f16_ts(d, ta + kk * 8,
                                           bd + (uint64_t)(((kk >> 2) * RB_B_KBLOCK + (kk & 3) * 32) >> 4), RB_IDESC,
                                           (m | kk) != 0 ? 1u : 0u);
                        tc::commit(P.afree(a));   // A buffer and B tile a are free once these complete
                        if (++a == NA) {
                            a = 0;
                            aph ^= 1u;
                        }
                    }
                    if (!ok)
                        break;
                    tc::commit(P.gfull(gs));   // accumulator gs is final once these complete
                    if (++gs == NG) {
                        gs = 0;
                        gph ^= 1u;
                    }
                }
            }
            tc::commit(P.done());   // every MMA issued by this thread has completed
        }
        __syncwarp();
    } else if (w < EPI0) {
        // ---- converters: group h takes stages h, h + 2, ...; thread = lane L ------
        // Weight row r of the stage's unit `half`, and the activation pieces
        // (vector L / 8, 16-byte chunk L % 8) of both units.
        const int h = w >> 2;
        const int n = L >> 3, c8 = L & 7;
        const uint32_t roff = (uint32_t)r * RB_KU, rsw = (uint32_t)(r & 7) << 4;   // 128-byte swizzle
        const uint32_t xoff = (uint32_t)n * RB_KU + (uint32_t)c8 * 16;
        const BPiece bp(n, c8);   // rows n and 16 + n: the same chunk offsets, 2 KiB apart
        int s = h, a = h, qa = 0;   // slot (j % S), A buffer (j % NA) and j / NA of stage j
        uint32_t fph = 0;           // (j / S) & 1
        for (int j = h; j < J; j += RB_GROUPS) {
            if (!tc::warp_wait(abort_word, q.error, q.wait_ns, P.full(s), fph))
                break;
            int4 wv[8];
            if (r < BR) {
                const uint32_t wrow = P.wtile(s, half) + roff;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    wv[c] = tc::lds128(wrow + (((uint32_t)c << 4) ^ rsw));
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    wv[c] = make_int4(0, 0, 0, 0);
            }
            const int4 xa = tc::lds128(P.xtile(s, 0) + xoff);
            const int4 xb = tc::lds128(P.xtile(s, 1) + xoff);
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(P.empty(s));   // this warp is done with stage s
            if (j >= NA && !tc::warp_wait(abort_word, q.error, q.wait_ns, P.afree(a), (uint32_t)(qa & 1) ^ 1u))
                break;
            tc::fence_after();
            // A operand: 128 f16 of this lane's row -> 64 columns of buffer a
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t v[16];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int4 &x = wv[part * 2 + c2];
                    tc::i8x4_to_f16x4((uint32_t)x.x, v[c2 * 8 + 0], v[c2 * 8 + 1]);
                    tc::i8x4_to_f16x4((uint32_t)x.y, v[c2 * 8 + 2], v[c2 * 8 + 3]);
                    tc::i8x4_to_f16x4((uint32_t)x.z, v[c2 * 8 + 4], v[c2 * 8 + 5]);
                    tc::i8x4_to_f16x4((uint32_t)x.w, v[c2 * 8 + 6], v[c2 * 8 + 7]);
                }
                tc::st16(tmem + tl + (uint32_t)a * RB_A_COLS + part * 16, v);
            }
            // B operand: vector n over the first unit is row n, over the second row 16 + n
            put_b(P.btile(a) + bp.row, bp, xa);
            put_b(P.btile(a) + bp.row + 2 * 1024, bp, xb);
            tc::wait_st();
            tc::fence_async_smem();
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(P.aready(a));
            s += RB_GROUPS;
            if (s >= S) {
                s -= S;
                fph ^= 1u;
            }
            a += RB_GROUPS;
            if (a >= NA) {
                a -= NA;
                ++qa;
            }
        }
    } else {
        // ---- epilogue warps: accumulators -> int32 sums -> the four parts of k
        // of each row added in shared memory -> scaled outputs ---------------------
        const int part = 2 * p + half;   // which part of k this lane summed
        const int t = p * (32 * RB_EPI_WARPS) + (w - EPI0) * 32 + lane;   // 0..255 over the CTA
        const int orow = t >> 2;          // output row within the block
        const int ovec = 4 * (t & 3);     // its first of four vectors
        dev::wait_previous_kernel();
        if (p == 0 && w == EPI0 && lane < RB_VEC) {
            const float v = lane < q.batch ? __ldg(q.scale_x + lane) : 0.f;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sx_at + 4 * lane), "f"(v) : "memory");
        }
        bool ok = true;
        int gs = 0;            // accumulator of the next group (g % NG)
        uint32_t gph = 0;      // (g / NG) & 1
        for (int b = 0; b < nblk; ++b) {
            const int32_t row = r0 + b * BR + orow;
            const bool live = orow < BR && b * BR + orow < rc;
            const float sw = live ? __ldg(q.scale_w + row) : 0.f;   // in flight during the block
            int32_t isum[RB_VEC];
#pragma unroll
            for (int v = 0; v < RB_VEC; ++v)
                isum[v] = 0;
            for (int u0 = 0; u0 < UQ; u0 += RB_UNITS_PER_GROUP) {
                const int cur = gs;
                const uint32_t ph = gph;
                if (++gs == NG) {
                    gs = 0;
                    gph ^= 1u;
                }
                if (!ok)
                    continue;
                if (!tc::warp_wait(abort_word, q.error, q.wait_ns, P.gfull(cur), ph)) {
                    ok = false;
                    continue;
                }
                tc::fence_after();
                uint32_t v[16];
                tc::ld16(tmem + tl + acc_col + (uint32_t)cur * RB_ACC_COLS + RB_VEC * half, v);
#pragma unroll
                for (int i = 0; i < RB_VEC; ++i)
                    isum[i] += __float2int_rn(__uint_as_float(v[i]));
                tc::fence_before();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(P.gfree(cur));
            }
            const uint32_t mine = merge + (uint32_t)((part * RB_MAX_ROWS + r) * RB_VEC) * 4;
#pragma unroll
            for (int i = 0; i < RB_VEC; i += 4)
                tc::sts128(mine + 4 * i, (uint32_t)isum[i], (uint32_t)isum[i + 1], (uint32_t)isum[i + 2],
                           (uint32_t)isum[i + 3]);
            const bool valid = epi_barrier_and(ok && !tc::aborted(abort_word));
            if (live) {
                int32_t tot[4] = {0, 0, 0, 0};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int4 v4 = tc::lds128(merge + (uint32_t)((qq * RB_MAX_ROWS + orow) * RB_VEC + ovec) * 4);
                    tot[0] += v4.x;
                    tot[1] += v4.y;
                    tot[2] += v4.z;
                    tot[3] += v4.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int bv = ovec + i;
                    if (bv < q.batch) {
                        float sx;
                        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sx) : "r"(sx_at + 4 * bv));
                        const int64_t o = (int64_t)row * q.y_stride + bv;
                        q.y[o] = valid ? __fmul_rn(__int2float_rn(tot[i]), __fmul_rn(sw, sx))
                                       : __int_as_float(0x7fc00000);
                        if (q.acc)
                            q.acc[o] = valid ? tot[i] : INT32_MIN;
                    }
                }
            }
            epi_barrier();   // the sums are read before the next block writes them
        }
    }

    // ---- teardown: tensor memory is freed only after every MMA has completed
    tc::fence_before();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p == 0 && w == PRODUCER) {
        if (lane < RB_PIPES) {
            Pipe Pl = P;
            Pl.base = pipes0 + (uint32_t)lane * q.pipe_bytes;
            dev::mbar_wait_bounded(Pl.done(), 0, q.wait_ns);
        }
        __syncwarp();
        tc::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(RB_TMEM_COLS)
                     : "memory");
    }
}

// The kernel's dynamic shared-memory limit, raised once per device to the largest size.
std::atomic<int> g_rows_smem_set[64];

cudaError_t rows_smem_limit()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    if (dev >= 0 && dev < 64 && g_rows_smem_set[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(dot_tc_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RB_MAX_SMEM);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        g_rows_smem_set[dev].store(1, std::memory_order_release);
    return e;
}

}  // namespace

// Schedule of the row-block kernel for n_rows x k on `sms` SMs.  cfg: depth
// (even, 2..8; 0 = the deepest of 4 and 2 that fits), a_bufs (2 or 3; 0 = 2);
// units_per_stage must be 0 or 1 and pipes 0 or 2.  Unless `forced`, the
// schedule is taken only where it fills at least half the tensor-memory
// lanes (32 or more rows per block) and k has at least 16 units (each
// pipeline at least four stages).
bool dot_tc_rows_plan(int64_t n_rows, int32_t k, int64_t sms, const DotTcConfig &cfg, bool forced,
                      DotTcPlan *out)
{
    if (n_rows < 1 || sms < 1 || k < 16 || (cfg.units_per_stage != 0 && cfg.units_per_stage != 1) ||
        (cfg.pipes != 0 && cfg.pipes != RB_PIPES))
        return false;
    const int64_t rpc = (n_rows + sms - 1) / sms;
    const int64_t nblk = (rpc + RB_MAX_ROWS - 1) / RB_MAX_ROWS;
    const int64_t br = (rpc + nblk - 1) / nblk;
    const int32_t ub = (k + RB_KU - 1) / RB_KU;
    const int32_t uq = (ub + 3) / 4;   // stages per block: two units each, in each of two pipelines
    if (!forced && (br < RB_MAX_ROWS / 2 || ub < 16))
        return false;
    const int na = cfg.a_bufs ? cfg.a_bufs : 2;
    if (na < 2 || (uint32_t)na * RB_A_COLS + RB_ACC_COLS > RB_PIPE_COLS)
        return false;
    int ng = (int)((RB_PIPE_COLS - (uint32_t)na * RB_A_COLS) / RB_ACC_COLS);
    ng = ng > 16 ? 16 : ng;
    const uint32_t wbox = ((uint32_t)br * RB_KU + 1023u) & ~1023u;
    const uint32_t stage = 2 * wbox + 2 * RB_X_BOX;
    int depth = cfg.depth;
    if (depth == 0) {
        depth = 4;
        if (rb_smem_bytes(rb_pipe_bytes(depth, na, ng, stage)) > RB_MAX_SMEM)
            depth = 2;
    }
    if (depth < 2 || depth > LOOM_MAX_DEPTH || (depth & 1))
        return false;   // the two converter groups must each keep to their own stages
    const uint32_t pipe = rb_pipe_bytes(depth, na, ng, stage);
    uint32_t smem = rb_smem_bytes(pipe);
    if (smem > RB_MAX_SMEM)
        return false;
    smem = smem < RB_MIN_SMEM ? RB_MIN_SMEM : smem;
    *out = DotTcPlan{};
    out->grid = (n_rows + rpc - 1) / rpc;
    out->total_units = n_rows * (int64_t)ub;
    out->units_per_band = ub;
    out->quantum = 1;
    out->depth = depth;
    out->ups = 1;
    out->na = na;
    out->ng = ng;
    out->pipes = RB_PIPES;
    out->groups = RB_GROUPS;
    out->mode = DOT_TC_ROWS;
    out->cluster = 1;
    out->pipe_bytes = pipe;
    out->smem_bytes = smem;
    out->split = false;
    out->sm_count = sms;
    out->rows_per_cta = (int32_t)rpc;
    out->block_rows = (int32_t)br;
    out->stages_per_block = uq;
    out->wbox = wbox;
    out->stage_bytes = stage;
    return true;
}

int dot_tc_rows_threads() { return RB_THREADS; }

cudaError_t launch_dot_tc_rows(const DotParams &p, const DotTcPlan &plan, cudaStream_t stream)
{
    if (plan.grid == 0)
        return cudaSuccess;
    const int64_t k = (int64_t)p.k_words * 4;
    CUtensorMap tmw, tmx;
    if (!encode_tensor_map_2d_u8(&tmw, p.w, (uint64_t)k, (uint64_t)p.n_rows, RB_KU, (uint32_t)plan.block_rows,
                                 CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d_u8(&tmx, p.x, (uint64_t)k, (uint64_t)p.batch, RB_KU, RB_VEC, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    RowsParams q;
    q.scale_w = p.scale_w;
    q.scale_x = p.scale_x;
    q.y = p.y;
    q.acc = p.acc;
    q.error = p.error;
    q.n_rows = p.n_rows;
    q.batch = p.batch;
    q.y_stride = p.y_stride;
    q.rpc = plan.rows_per_cta;
    q.br = plan.block_rows;
    q.uq = plan.stages_per_block;
    q.depth = plan.depth;
    q.na = plan.na;
    q.ng = plan.ng;
    q.wbox = plan.wbox;
    q.stage_bytes = plan.stage_bytes;
    q.pipe_bytes = plan.pipe_bytes;
    q.wait_ns = p.wait_ns;
    q.inject_stall = p.inject_stall;
    cudaError_t e = rows_smem_limit();
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid, 1, 1);
    cfg.blockDim = dim3(RB_THREADS, 1, 1);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see follow_previous_kernel
    ca[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = ca;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dot_tc_rows_kernel, tmw, tmx, q);
}

}  // namespace loom
