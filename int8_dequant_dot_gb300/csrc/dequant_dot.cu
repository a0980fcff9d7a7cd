// dequant_dot.cu -- packed signed-byte dequantised dot products on sm_103a.
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section "Apply
// the same controls to a packed dot product"): each 32-bit field holds four
// signed bytes; they are unpacked, scaled and accumulated as a dot product.
// The workload here uses int8 weights W[n_rows][k] with a scale per row and
// int8 activations X[batch][k] with a scale per vector:
//   acc[r][b] = sum_k W[r][k] * X[b][k]   (int32: exact, order-free)
//   y[r][b]   = (float)acc[r][b] * (scale_w[r] * scale_x[b])
//
// GB300 design
//  * __dp4a does the unpack and four multiply-adds of one packed word in one
//    instruction; accumulation is int32, so results are exact and do not
//    depend on the order of the k terms (|acc| <= 2^14 * k < 2^31).
//  * Weights stream once through HBM.  Each warp owns its rows and a private
//    ring of `depth` shared-memory stages filled by bulk copies (the
//    read-ahead queue); activations are small and stay in L1/L2.
//  * batch <= 2 ("lanes across k"): each CTA owns a block of rows whose 8 KiB
//    pieces its warps share out evenly; every lane takes one 16-byte group of
//    a piece per 512-byte slot, dp4a against the matching activation words,
//    and each warp's share of a row is summed across the warp and added into
//    the row's total in shared memory.
//  * batch > 2 ("lanes across the batch"): eight rows per unit; lane b of
//    each half-warp owns vector b and keeps a slice of its activations in
//    registers, reused for all eight rows; weight words are read from the
//    stage as broadcasts, and the two half-warps split the k range.
//  * Unaligned inputs or k % 16 != 0 take a plain-load kernel.
#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

using dev::FULL_MASK;

__device__ __forceinline__ float dequant(int32_t acc, float sw, float sx)
{
    return __fmul_rn(__int2float_rn(acc), __fmul_rn(sw, sx));
}

__device__ __forceinline__ void dp4a4(int32_t &acc, const int4 &w, const int4 &x)
{
    acc = __dp4a(w.x, x.x, acc);
    acc = __dp4a(w.y, x.y, acc);
    acc = __dp4a(w.z, x.z, acc);
    acc = __dp4a(w.w, x.w, acc);
}

__device__ __forceinline__ void store_result(const DotParams &p, int32_t r, int b, int32_t acc,
                                             bool valid)
{
    const int64_t o = (int64_t)r * p.y_stride + b;
    p.y[o] = valid ? dequant(acc, __ldg(p.scale_w + r), __ldg(p.scale_x + b))
                   : __int_as_float(0x7fc00000);
    if (p.acc)
        p.acc[o] = valid ? acc : INT32_MIN;
}

// Per-warp ring of `depth` stages of `stage_bytes`, with one mbarrier each.
struct Ring {
    uint32_t data0, bar0;
    int depth;
    uint32_t stage_bytes;
    int ps = 0, cs = 0;
    uint32_t cphase = 0;
    uint32_t issued = 0, consumed = 0;

    __device__ void init(int lane)
    {
        if (lane == 0) {
            for (int s = 0; s < depth; ++s)
                dev::mbar_init(bar0 + 8 * s, 1);
            dev::fence_barrier_init();
        }
        __syncwarp();
    }
    __device__ uint32_t pstage() const { return data0 + ps * stage_bytes; }
    __device__ uint32_t pbar() const { return bar0 + 8 * ps; }
    __device__ void pnext()
    {
        ++issued;
        ps = (ps + 1 == depth) ? 0 : ps + 1;
    }
    __device__ bool wait(uint64_t limit_ns)
    {
        const bool landed = dev::mbar_wait_bounded(bar0 + 8 * cs, cphase, limit_ns);
        return __all_sync(FULL_MASK, landed);
    }
    __device__ void cnext()
    {
        __syncwarp();
        ++consumed;
        cs = (cs + 1 == depth) ? 0 : cs + 1;
        cphase ^= (cs == 0) ? 1u : 0u;
    }
    // After a failed wait: let copies already in flight land (bounded).
    __device__ void drain(uint64_t limit_ns, bool any_issued)
    {
        if (!any_issued)
            return;
        int s = cs;
        uint32_t ph = cphase;
        for (uint32_t i = consumed; i < issued; ++i) {
            dev::mbar_wait_bounded(bar0 + 8 * s, ph, limit_ns);
            s = (s + 1 == depth) ? 0 : s + 1;
            ph ^= (s == 0) ? 1u : 0u;
        }
    }
};

// ---------------------------------------------------------------------------
// batch <= 2: lanes across k.  CTA c owns rows [c RPC, (c + 1) RPC) for the
// whole of k.  Its rows are cut into pieces of at most DOT_K_PIECE_WORDS words
// (8 KiB) of one row, numbered chunk by chunk (the first 8 KiB of every row,
// then the next), and warp w of the CTA takes an equal contiguous share of
// the pieces: every warp of every CTA moves the same number of bytes,
// whatever k and the number of rows, and a warp's consecutive pieces share
// their activation words (held in registers for one vector).  A warp streams its
// pieces through its own ring of `depth` bulk-copied stages.  Lane l takes
// words 4l..4l+3 of every 128-word slot of a piece, with the matching
// activation words.  The activations (batch x k bytes, shared by every row)
// are copied once into the CTA's shared memory when they fit (p.x_in_smem);
// else they are read through L1, which measured 2 us slower on 8192 x 16384.
// Each piece ends in one warp-wide sum per vector, added into the row's int32
// total in shared memory; integer additions in any order give the same sum.
// ---------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(256) dot_rows_k_kernel(const DotParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int SLOTS = DOT_K_PIECE_WORDS / 128;   // 128-word slots per piece
    constexpr int DOT_K_SLOT_GROUP = 8 / NB;          // slots whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int32_t r0 = (int32_t)blockIdx.x * p.rows_per_cta;
    if (r0 >= p.n_rows)
        return;   // over-dispatched CTA
    const int nr = min(p.rows_per_cta, p.n_rows - r0);
    const int32_t kw = p.k_words;
    const int32_t P = (kw + DOT_K_PIECE_WORDS - 1) / DOT_K_PIECE_WORDS;   // pieces per row
    const int32_t T = nr * P;
    const int32_t t0 = (int32_t)((int64_t)T * warp / warps);
    const int32_t t1 = (int32_t)((int64_t)T * (warp + 1) / warps);
    const int D = p.depth;
    constexpr uint32_t stage_bytes = DOT_K_PIECE_WORDS * 4;

    // shared memory: the warps' rings, their barriers, the activations' barrier,
    // the row totals [rows_per_cta][NB], then (x_in_smem) the activations
    Ring ring;
    ring.depth = D;
    ring.stage_bytes = stage_bytes;
    ring.data0 = dev::smem_u32(smem) + warp * D * stage_bytes;
    ring.bar0 = dev::smem_u32(smem) + warps * D * stage_bytes + warp * D * 8;
    const uint32_t xbar = dev::smem_u32(smem) + warps * D * (stage_bytes + 8);
    int32_t *rsum = reinterpret_cast<int32_t *>(smem + warps * D * (stage_bytes + 8) + 8);
    const int4 *xs = reinterpret_cast<const int4 *>(smem + dot_k_x_offset(warps, D, p.rows_per_cta));
    for (int i = threadIdx.x; i < nr * NB; i += blockDim.x)
        rsum[i] = 0;
    ring.init(lane);
    const uint64_t policy = dev::l2_evict_first_policy();
    const uint32_t xbytes = (uint32_t)p.batch * (uint32_t)kw * 4u;
    if (threadIdx.x == 0 && p.x_in_smem) {
        dev::mbar_init(xbar, 1);
        dev::fence_barrier_init();
        if (!p.inject_stall && xbytes) {
            dev::mbar_arrive_expect_tx(xbar, xbytes);
            dev::bulk_g2s(dev::smem_u32(xs), p.x, xbytes, xbar, dev::l2_evict_last_policy());
        }
    }
    __syncthreads();

    // Pieces are numbered chunk-major -- piece t is chunk t / nr of row t % nr --
    // so a warp's consecutive pieces share their activation words.  The first
    // piece of this warp: chunk cs0 of row rs.
    const int32_t cs0 = t0 / nr, rs = t0 - cs0 * nr;
    int32_t pt = t0, pr = rs, pc = cs0;   // the producer's next piece
    auto produce = [&]() {
        if (pt >= t1)
            return;
        const int32_t off = pc * DOT_K_PIECE_WORDS;
        if (lane == 0 && !p.inject_stall) {
            const uint32_t bytes = (uint32_t)min(DOT_K_PIECE_WORDS, kw - off) * 4u;
            dev::mbar_arrive_expect_tx(ring.pbar(), bytes);
            dev::bulk_g2s(ring.pstage(), p.w + (int64_t)(r0 + pr) * kw + off, bytes, ring.pbar(), policy);
        }
        ++pt;
        if (++pr == nr) {
            pr = 0;
            ++pc;
        }
        ring.pnext();
    };
    for (int s = 0; s < D; ++s)
        produce();

    // Vectors past the batch (NB rounds it up) re-read vector 0 and are not stored.
    const int4 *x4[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
        x4[b] = (p.x_in_smem ? xs : reinterpret_cast<const int4 *>(p.x)) + (int64_t)(b < p.batch ? b : 0) * (kw >> 2);
    const unsigned char *ring_base = smem + (size_t)warp * D * stage_bytes;
    int32_t acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
        acc[b] = 0;
    int32_t cr = rs, cc = cs0;   // the consumer's piece
    // NB == 1: the activation words of the current chunk held in registers
    // (16 per lane), loaded again only when the chunk changes
    int4 xr[NB == 1 ? SLOTS : 1];
    int32_t xr_chunk = -1;
    bool failed = false;
    // the activations must have landed (a stalled test run issued no copy: its wait runs out)
    if (p.x_in_smem && t0 < t1 && xbytes && !__all_sync(FULL_MASK, dev::mbar_wait_bounded(xbar, 0, p.wait_ns)))
        failed = true;
    for (int32_t t = t0; t < t1 && !failed; ++t) {
        if (!ring.wait(p.wait_ns)) {
            failed = true;
            break;
        }
        const int32_t off = cc * DOT_K_PIECE_WORDS;
        const int32_t m = min(DOT_K_PIECE_WORDS, kw - off);
        const int4 *s4 = reinterpret_cast<const int4 *>(ring_base + ring.cs * stage_bytes) + lane;
        const int4 *xl[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            xl[b] = x4[b] + (off >> 2) + lane;
        // activation words: from shared memory, or through L1
        auto xload = [&](const int4 *a) { return p.x_in_smem ? *a : __ldg(a); };
        if (NB == 1 && m == DOT_K_PIECE_WORDS) {
            if (cc != xr_chunk) {
#pragma unroll
                for (int s = 0; s < SLOTS; ++s)
                    xr[s] = xload(xl[0] + 32 * s);
                xr_chunk = cc;
            }
#pragma unroll
            for (int s = 0; s < SLOTS; ++s)
                dp4a4(acc[0], s4[32 * s], xr[s]);
        } else if (m == DOT_K_PIECE_WORDS) {
            // a whole piece: no bounds tests, so the loads of a group of slots issue together
#pragma unroll
            for (int g = 0; g < SLOTS; g += DOT_K_SLOT_GROUP) {
                int4 wv[DOT_K_SLOT_GROUP], xv[NB][DOT_K_SLOT_GROUP];
#pragma unroll
                for (int s = 0; s < DOT_K_SLOT_GROUP; ++s) {
                    wv[s] = s4[32 * (g + s)];
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        xv[b][s] = xload(xl[b] + 32 * (g + s));
                }
#pragma unroll
                for (int s = 0; s < DOT_K_SLOT_GROUP; ++s)
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        dp4a4(acc[b], wv[s], xv[b][s]);
            }
        } else {
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) {
                if (lane * 4 + 128 * s < m) {
                    const int4 wv = s4[32 * s];
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        dp4a4(acc[b], wv, xload(xl[b] + 32 * s));
                }
            }
        }
        ring.cnext();
        produce();
        // this warp's share of row cr ends with the piece: add it to the row's total
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int32_t sum = dev::warp_sum_i32(acc[b]);
            if (lane == 0)
                atomicAdd(rsum + cr * NB + b, sum);
            acc[b] = 0;
        }
        if (++cr == nr) {
            cr = 0;
            ++cc;
        }
    }
    if (failed) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        ring.drain(p.wait_ns, !p.inject_stall);
    }
    const bool valid = !__syncthreads_or(failed);
    for (int i = threadIdx.x; i < nr * NB; i += blockDim.x) {
        const int r = i / NB, b = i - r * NB;
        if (b < p.batch)
            store_result(p, r0 + r, b, rsum[i], valid);
    }
}

// ---------------------------------------------------------------------------
// batch in (2, 16]: lanes across the batch.  Unit = DOT_B_ROWS rows.
// A stage holds DOT_B_CHUNK_WORDS words of each unit row and of each
// activation vector (one bulk copy per row and per vector).
// Lane (h, b): vector b = lane & 15, half h = lane >> 4.  Within a chunk the
// 16-byte groups alternate between the halves (group g -> half g & 1).
// ---------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(256) dot_staged_b_kernel(const DotParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int warps = blockDim.x >> 5;
    const int b = lane & 15;
    const int h = lane >> 4;
    const int32_t r0 = (int32_t)(((int64_t)blockIdx.x * warps + warp) * DOT_B_ROWS);
    if (r0 >= p.n_rows)
        return;
    const int n = min(DOT_B_ROWS, p.n_rows - r0);
    const int nb = p.batch;
    const int32_t kw = p.k_words;
    const int32_t nchunks = (kw + DOT_B_CHUNK_WORDS - 1) / DOT_B_CHUNK_WORDS;
    const int D = p.depth;
    constexpr uint32_t row_bytes = DOT_B_CHUNK_WORDS * 4;
    constexpr uint32_t stage_bytes = (DOT_B_ROWS + NB) * row_bytes;   // weights, then activations

    Ring ring;
    ring.depth = D;
    ring.stage_bytes = stage_bytes;
    ring.data0 = dev::smem_u32(smem) + warp * D * stage_bytes;
    ring.bar0 = dev::smem_u32(smem) + warps * D * stage_bytes + warp * D * 8;
    ring.init(lane);
    const uint64_t policy = dev::l2_evict_first_policy();
    const uint64_t keep = dev::l2_evict_last_policy();   // activations: re-read by every warp

    int pj = 0;
    auto produce = [&]() {
        if (pj >= nchunks)
            return;
        const int32_t off = pj * DOT_B_CHUNK_WORDS;
        const uint32_t bytes = (uint32_t)min(DOT_B_CHUNK_WORDS, kw - off) * 4u;
        if (!p.inject_stall) {
            if (lane == 0)
                dev::mbar_arrive_expect_tx(ring.pbar(), bytes * (n + nb));
            __syncwarp();
            if (lane < n)
                dev::bulk_g2s(ring.pstage() + lane * row_bytes, p.w + (int64_t)(r0 + lane) * kw + off,
                              bytes, ring.pbar(), policy);
            else if (lane >= DOT_B_ROWS && lane < DOT_B_ROWS + nb)
                dev::bulk_g2s(ring.pstage() + lane * row_bytes,
                              p.x + (int64_t)(lane - DOT_B_ROWS) * kw + off, bytes, ring.pbar(), keep);
        }
        ++pj;
        ring.pnext();
    };
    for (int s = 0; s < D; ++s)
        produce();

    const bool active = b < nb;
    int32_t acc[DOT_B_ROWS];
#pragma unroll
    for (int r = 0; r < DOT_B_ROWS; ++r)
        acc[r] = 0;

    bool failed = false;
    for (int j = 0; j < nchunks; ++j) {
        if (!ring.wait(p.wait_ns)) {
            failed = true;
            break;
        }
        const int32_t off = j * DOT_B_CHUNK_WORDS;
        const int32_t groups = min(DOT_B_CHUNK_WORDS, kw - off) >> 2;  // 16-byte groups
        const unsigned char *stage = smem + (size_t)warp * D * stage_bytes + ring.cs * stage_bytes;
        // This half's groups: g = 2q + h, activations of vector b from the stage.
        constexpr int QMAX = DOT_B_CHUNK_WORDS / 8;
        const int4 *xrow = reinterpret_cast<const int4 *>(stage + (DOT_B_ROWS + (active ? b : 0)) * row_bytes);
        int4 xv[QMAX];
#pragma unroll
        for (int q = 0; q < QMAX; ++q) {
            const int g = 2 * q + h;
            xv[q] = (active && g < groups) ? xrow[g] : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < DOT_B_ROWS; ++r) {
            if (r < n) {
                const int4 *wrow = reinterpret_cast<const int4 *>(stage + r * row_bytes);
#pragma unroll
                for (int q = 0; q < QMAX; ++q) {
                    const int g = 2 * q + h;
                    if (g < groups)
                        dp4a4(acc[r], wrow[g], xv[q]);
                }
            }
        }
        ring.cnext();
        produce();
    }
    if (failed) {
        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        ring.drain(p.wait_ns, !p.inject_stall);
    }
#pragma unroll
    for (int r = 0; r < DOT_B_ROWS; ++r) {
        const int32_t sum = acc[r] + __shfl_xor_sync(FULL_MASK, acc[r], 16);
        if (r < n && h == 0 && active)
            store_result(p, r0 + r, b, sum, !failed);
    }
}

// ---------------------------------------------------------------------------
// Plain loads: any 4-byte aligned input, any k % 4 == 0.  One warp per row.
// ---------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(256, 1) dot_direct_kernel(const DotParams p)
{
    dev::follow_previous_kernel();
    const int lane = threadIdx.x & 31;
    const int32_t r = (int32_t)((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
    if (r >= p.n_rows)
        return;
    const int32_t kw = p.k_words;
    const int32_t *wr = p.w + (int64_t)r * kw;
    int32_t acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
        acc[b] = 0;
    for (int32_t w = lane; w < kw; w += 32) {
        const int32_t wv = __ldg(wr + w);
#pragma unroll
        for (int b = 0; b < NB; ++b)
            if (b < p.batch)
                acc[b] = __dp4a(wv, __ldg(p.x + (int64_t)b * kw + w), acc[b]);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int32_t s = dev::warp_sum_i32(acc[b]);
        if (lane == b && b < p.batch)
            store_result(p, r, b, s, true);
    }
}

// ---------------------------------------------------------------------------
// Unpack: one thread per packed word, 256-thread CTAs.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(UNPACK_BLOCK) unpack_kernel(const int32_t *__restrict__ packed,
                                                              int64_t n_words, float *__restrict__ out)
{
    dev::follow_previous_kernel();
    const int64_t j = (int64_t)blockIdx.x * UNPACK_BLOCK + threadIdx.x;
    if (j >= n_words)
        return;  // over-dispatched invocation: no load, no store
    const uint32_t w = (uint32_t)__ldg(packed + j);
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = (float)(int32_t)(int8_t)(uint8_t)(w >> (8 * i));
    if ((reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
        reinterpret_cast<float4 *>(out)[j] = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[4 * j + i] = v[i];
    }
}

}  // namespace

DotKernel dot_select(bool aligned, int32_t k, int32_t batch_pass)
{
    if (!aligned || (k % 16) != 0)
        return DotKernel::Direct;
    return batch_pass <= 2 ? DotKernel::StagedK : DotKernel::StagedB;
}

int64_t dot_rows_per_cta(DotKernel kind, int64_t n_rows, int warps, int ctas_per_sm, int64_t sms)
{
    switch (kind) {
    case DotKernel::StagedK: {
        // ceil(n_rows / (CTAs per SM x SMs)) rows, so that one wave holds every row
        const int64_t ctas = (int64_t)(ctas_per_sm ? ctas_per_sm : DOT_K_DEFAULT_CTAS_PER_SM) * (sms > 0 ? sms : 1);
        int64_t rpc = (n_rows + ctas - 1) / ctas;
        rpc = rpc < 1 ? 1 : rpc;
        return rpc > DOT_K_MAX_ROWS_PER_CTA ? DOT_K_MAX_ROWS_PER_CTA : rpc;
    }
    case DotKernel::StagedB:
        return (int64_t)warps * DOT_B_ROWS;
    default:
        return warps;
    }
}

uint32_t dot_smem_bytes(DotKernel kind, int depth, int warps, int64_t rows_per_cta)
{
    switch (kind) {
    case DotKernel::StagedK:   // rings, barriers, row totals (the activations are added by the caller)
        return dot_k_x_offset(warps, depth, rows_per_cta);
    case DotKernel::StagedB:
        return (uint32_t)(warps * depth * ((DOT_B_ROWS + DOT_MAX_BATCH_PER_PASS) * DOT_B_CHUNK_WORDS * 4 + 8));
    default:
        return 0;
    }
}

cudaError_t launch_dot(const DotParams &p, DotKernel kind, const loom_launch &L, cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    const int nb = p.batch;
    switch (kind) {
    case DotKernel::Tensor:
        return cudaErrorInvalidValue;   // launched by launch_dot_tc with its schedule
    case DotKernel::StagedK:
        return nb == 1 ? launch_with(dot_rows_k_kernel<1>, L, stream, p) : launch_with(dot_rows_k_kernel<2>, L, stream, p);
    case DotKernel::StagedB:
        return launch_with(dot_staged_b_kernel<16>, L, stream, p);
    default:
        if (nb <= 1)
            return launch_with(dot_direct_kernel<1>, L, stream, p);
        if (nb <= 4)
            return launch_with(dot_direct_kernel<4>, L, stream, p);
        return launch_with(dot_direct_kernel<16>, L, stream, p);
    }
}

cudaError_t launch_unpack(const int32_t *packed, int64_t n_words, float *out, const loom_launch &L,
                          cudaStream_t stream)
{
    if (L.grid[0] == 0)
        return cudaSuccess;
    return launch_with(unpack_kernel, L, stream, packed, n_words, out);
}

}  // namespace loom
