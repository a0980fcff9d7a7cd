// packed_dot.cu -- the pages' own packed signed-byte dot: f16 per-record
// scales, f32 activations, an ordered f32 accumulation per output lane.
//
// Method (Loom pages, "Tune loop unrolling and pipelining", section "Apply
// the same controls to a packed dot product"): lane l of an instance owns one
// output.  For each record r < count it reads the packed word fields[r][l]
// (four signed bytes), the f16 scale scales[r][l] and four f32 activations
// rhs[r][l mod streams][0..3]; the bytes are converted to f32 and scaled, and
// the dot product with the activations advances the lane's f32 sum.  The
// records are a recurrence: their order fixes the result.
//
// Reading of the dot step: the four products enter the sum in element order,
// each as one fused multiply-add.  int8 x f16 fits in 19 significant bits,
// so the scaled bytes are exact in f32 and only the fused steps round.
//
// GB300 design
//  * Many independent instances per launch (the pages benchmark one instance
//    per dispatch, many dispatches per measurement).  The staged path cuts
//    them into tiles of 256 lanes of one instance and runs a grid of up to
//    seven CTAs per SM (as many as their rings and registers allow) over the
//    tile list (tile c, c + G, ...; 1024 tiles of the 128 x 2048-lane workload
//    take one each), where CTAs of 512 lanes ran in 1.7 waves.
//  * One producer thread streams every stage of every tile of its CTA
//    through one ring of `depth` stages -- `rps` records of the tile's words
//    (1 KiB per record), scales (512 B) and the instance's activation row
//    (16 B per stream) as three 3-D TMA copies on the stage's mbarrier;
//    words and scales evict-first, activations (read by every tile of the
//    instance) evict-last -- so a CTA's next tile is already in flight while
//    its consumers finish the current one.  This is the read-ahead queue of
//    the pages' pipeline(depth); depth 1 is the serial control and the depth
//    never changes a result.  (Reading the activations through L1 instead
//    left every CTA waiting on one load per record: measured 1.6x slower.)
//  * Consumer thread t owns lanes t and t + 128 of a tile: two independent
//    recurrences advanced together by packed f32x2 instructions (each half
//    rounds as the scalar instruction does: the same bits).  When 128 is a
//    multiple of the stream count the two lanes read the same activations, so
//    one float4 serves both.  Per record a thread reads two words and two
//    scales from shared memory (consecutive lanes, consecutive addresses) and
//    its stream's float4 (conflict-free); the bytes become f32 by a byte
//    permute and a packed subtraction, the scalings are packed multiplies and
//    the four ordered fused steps are packed fused multiply-adds.  With one
//    lane per thread the kernel was bound by instruction issue (36.8 us per
//    launch in trains of launches); two lanes per thread issue 12% fewer
//    instructions and, with four-record stages and seven CTAs of four
//    consumer warps per SM, run at the time of a launch that only reads the
//    same bytes (32.5-32.9 us).
//  * Direct path (inputs a TMA copy cannot take: lanes not a multiple of 8,
//    more than 64 streams, unaligned pointers): plain loads, same order and
//    arithmetic, identical bits.
//  * Every wait is bounded; a wait that runs out sets LOOM_DEVERR_TIMEOUT and
//    the affected outputs are NaN.
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace loom {
namespace {

constexpr int PD_LANES = 256;                 // lanes per direct CTA
constexpr int PD_TILE = 256;                  // staged path: lanes per tile, two per consumer thread
constexpr int PD_PAIR = PD_TILE / 2;          // thread t owns lanes t and t + PD_PAIR
constexpr int PD_CONSUMER_WARPS = PD_PAIR / 32;
constexpr int PD_THREADS_STAGED = PD_PAIR + 32;   // + the producer warp

struct PackedDeviceParams {
    const int32_t *fields;
    const uint16_t *scales;
    const float *rhs;
    int32_t problems, records, lanes, streams;
    const int32_t *counts;   // per instance, or NULL: count_scalar for all
    int32_t count_scalar;
    const float *initial;    // [problems][lanes] or NULL (0)
    float *out;              // [problems][lanes]
    int32_t *error;
    int32_t depth;           // stages in the ring
    int32_t rps;             // records per stage
    uint64_t wait_ns;
    int32_t inject_stall;
};

// Shared-memory layout of one stage: fields [rps][256] i32, scales [rps][256]
// u16, activations [rps][streams][4] f32; each part 128-byte aligned.
struct PdStage {
    uint32_t fields_bytes, scales_bytes, rhs_bytes;
    __host__ __device__ PdStage(int rps, int streams)
        : fields_bytes((uint32_t)rps * PD_TILE * 4u), scales_bytes(((uint32_t)rps * PD_TILE * 2u + 127u) & ~127u),
          rhs_bytes(((uint32_t)rps * (uint32_t)streams * 16u + 127u) & ~127u)
    {
    }
    __host__ __device__ uint32_t bytes() const { return fields_bytes + scales_bytes + rhs_bytes; }
};

uint32_t pd_smem_bytes(int depth, int rps, int streams)
{
    return 128u + (uint32_t)depth * PdStage(rps, streams).bytes() + 16u * (uint32_t)depth;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One record of one lane: four signed bytes, scaled exactly, then four fused
// steps in element order.
__device__ __forceinline__ float record_step(float sum, uint32_t word, uint16_t scale_bits, const float4 &a)
{
    const float scale = __half2float(__ushort_as_half(scale_bits));
    const float b0 = (float)(int32_t)(int8_t)(word & 0xFFu);
    const float b1 = (float)(int32_t)(int8_t)((word >> 8) & 0xFFu);
    const float b2 = (float)(int32_t)(int8_t)((word >> 16) & 0xFFu);
    const float b3 = (float)(int32_t)(int8_t)(word >> 24);
    sum = __fmaf_rn(__fmul_rn(b0, scale), a.x, sum);
    sum = __fmaf_rn(__fmul_rn(b1, scale), a.y, sum);
    sum = __fmaf_rn(__fmul_rn(b2, scale), a.z, sum);
    sum = __fmaf_rn(__fmul_rn(b3, scale), a.w, sum);
    return sum;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// One record of two lanes (words w0, w1, f16 scales h0, h1; activations a0 of
// the first lane, a1 of the second), their sums packed in `sum`: the record
// step of both lanes at once, with the same roundings as record_step.
__device__ __forceinline__ uint64_t pair_products(uint32_t w0, uint32_t w1, uint16_t h0, uint16_t h1, uint64_t (&m)[4])
{
    const uint64_t ss = dev::pack2(__half2float(__ushort_as_half(h0)), __half2float(__ushort_as_half(h1)));
    const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
    uint32_t x0, x1, y0, y1, z0, z1, v0, v1;   // byte j of each word as 2^23 + (b + 128)
    asm("prmt.b32 %0, %1, %2, 0x7540;" : "=r"(x0) : "r"(u0), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7540;" : "=r"(x1) : "r"(u1), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7541;" : "=r"(y0) : "r"(u0), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7541;" : "=r"(y1) : "r"(u1), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7542;" : "=r"(z0) : "r"(u0), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7542;" : "=r"(z1) : "r"(u1), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7543;" : "=r"(v0) : "r"(u0), "r"(0x4B000000u));
    asm("prmt.b32 %0, %1, %2, 0x7543;" : "=r"(v1) : "r"(u1), "r"(0x4B000000u));
    const uint64_t bias = dev::pack2(8388736.0f, 8388736.0f);   // 2^23 + 128
    m[0] = mul2(dev::sub2(dev::pack2(__uint_as_float(x0), __uint_as_float(x1)), bias), ss);
    m[1] = mul2(dev::sub2(dev::pack2(__uint_as_float(y0), __uint_as_float(y1)), bias), ss);
    m[2] = mul2(dev::sub2(dev::pack2(__uint_as_float(z0), __uint_as_float(z1)), bias), ss);
    m[3] = mul2(dev::sub2(dev::pack2(__uint_as_float(v0), __uint_as_float(v1)), bias), ss);
    return ss;
}

// Both lanes against the same activations.
__device__ __forceinline__ uint64_t pair_record(uint64_t sum, uint32_t w0, uint32_t w1, uint16_t h0, uint16_t h1,
                                                const float4 &a)
{
    uint64_t m[4];
    pair_products(w0, w1, h0, h1, m);
    sum = fma2(m[0], dev::pack2(a.x, a.x), sum);
    sum = fma2(m[1], dev::pack2(a.y, a.y), sum);
    sum = fma2(m[2], dev::pack2(a.z, a.z), sum);
    sum = fma2(m[3], dev::pack2(a.w, a.w), sum);
    return sum;
}

// Each lane against its own activations.
__device__ __forceinline__ uint64_t pair_record(uint64_t sum, uint32_t w0, uint32_t w1, uint16_t h0, uint16_t h1,
                                                const float4 &a0, const float4 &a1)
{
    uint64_t m[4];
    pair_products(w0, w1, h0, h1, m);
    sum = fma2(m[0], dev::pack2(a0.x, a1.x), sum);
    sum = fma2(m[1], dev::pack2(a0.y, a1.y), sum);
    sum = fma2(m[2], dev::pack2(a0.z, a1.z), sum);
    sum = fma2(m[3], dev::pack2(a0.w, a1.w), sum);
    return sum;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t a)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t a)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ int32_t instance_count(const PackedDeviceParams &p, int32_t inst)
{
    const int32_t raw = p.counts ? __ldg(p.counts + inst) : p.count_scalar;
    const int32_t c = min(max(raw, 0), p.records);
    if (c != raw)
        dev::flag_error(p.error, LOOM_DEVERR_COUNT_RANGE);
    return c;
}

// Staged path: a grid of up to seven CTAs per SM.  The work is a
// list of tiles -- 256 lanes of one instance, instance-major -- and CTA c
// takes tiles c, c + G, c + 2G, ... (1024 tiles of the 128 x 2048-lane
// workload: 6 or 7 per SM).  The producer streams every stage of every tile of the CTA through one
// ring, so the copies of a CTA's next tile are in flight while its consumers
// finish the current one; consumer thread t owns lane t of the tile.
template <bool SAME>
__global__ void __launch_bounds__(PD_THREADS_STAGED, 7) packed_dot_staged_kernel(
    const __grid_constant__ CUtensorMap tm_fields, const __grid_constant__ CUtensorMap tm_scales,
    const __grid_constant__ CUtensorMap tm_rhs, const PackedDeviceParams p)
{
    dev::follow_previous_kernel();
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = (dev::smem_u32(smem_raw) + 127u) & ~127u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.depth, RPS = p.rps;
    const PdStage st(RPS, p.streams);
    const uint32_t bars = base + (uint32_t)D * st.bytes();
    auto full = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bars + 8u * (uint32_t)(D + s); };
    auto stage = [&](int s) { return base + (uint32_t)s * st.bytes(); };
    const int32_t lblocks = (p.lanes + PD_TILE - 1) / PD_TILE;
    const int32_t tiles = p.problems * lblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < D; ++s) {
            dev::mbar_init(full(s), 1);
            dev::mbar_init(empty(s), PD_CONSUMER_WARPS);
        }
        dev::fence_barrier_init();
    }
    __syncthreads();

    if (warp == PD_CONSUMER_WARPS) {
        // ---- producer: three 3-D copies per stage (words, scales, activations)
        if (lane == 0 && !p.inject_stall) {
            const uint64_t once = dev::l2_evict_first_policy();   // words, scales: read once
            const uint64_t shared = dev::l2_evict_last_policy();  // activations: every lane block
            const uint32_t tx = (uint32_t)RPS * PD_TILE * 6u + (uint32_t)RPS * (uint32_t)p.streams * 16u;
            int s = 0, issued = 0;
            uint32_t eph = 0;   // parity of the consumers' release of stage s
            bool ok = true;
            for (int32_t t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int32_t inst = t / lblocks;
                const int32_t l0 = (t - inst * lblocks) * PD_TILE;
                const int32_t count = instance_count(p, inst);
                for (int32_t r0 = 0; r0 < count; r0 += RPS) {
                    if (issued >= D && !dev::mbar_wait_bounded(empty(s), eph, p.wait_ns)) {
                        dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    dev::mbar_arrive_expect_tx(full(s), tx);
                    tma_load_3d(stage(s), &tm_fields, l0, r0, inst, full(s), once);
                    tma_load_3d(stage(s) + st.fields_bytes, &tm_scales, l0, r0, inst, full(s), once);
                    tma_load_3d(stage(s) + st.fields_bytes + st.scales_bytes, &tm_rhs, 0, r0, inst, full(s), shared);
                    ++issued;
                    if (++s == D) {
                        s = 0;
                        if (issued > D)
                            eph ^= 1u;
                    }
                }
            }
            // every copy issued must land before the CTA may leave (bounded)
            for (int j = issued > D ? issued - D : 0; j < issued; ++j)
                dev::mbar_wait_bounded(full(j % D), (j / D) & 1, p.wait_ns);
        }
        return;
    }

    // ---- consumers: thread t owns lanes t and t + PD_PAIR of each tile
    const int t = threadIdx.x;
    const uint32_t astep = 16u * (uint32_t)p.streams;   // activations of one record
    int s = 0;
    uint32_t fph = 0;   // parity of the copies into stage s
    bool ok = true;
    for (int32_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int32_t inst = tile / lblocks;
        const int32_t la = (tile - inst * lblocks) * PD_TILE + t, lb = la + PD_PAIR;
        const bool livea = la < p.lanes, liveb = lb < p.lanes;
        // the lanes' activation streams: offsets within a stage's activations
        const uint32_t xa = 16u * (uint32_t)(la % p.streams), xb = SAME ? xa : 16u * (uint32_t)(lb % p.streams);
        const int32_t count = instance_count(p, inst);
        const float *init = p.initial ? p.initial + (int64_t)inst * p.lanes : nullptr;
        uint64_t sum = dev::pack2(livea && init ? __ldg(init + la) : 0.f, liveb && init ? __ldg(init + lb) : 0.f);
        for (int32_t r0 = 0; r0 < count && ok; r0 += RPS) {
            const bool landed = dev::mbar_wait_bounded(full(s), fph, p.wait_ns);
            if (!__all_sync(dev::FULL_MASK, landed)) {
                ok = false;
                break;
            }
            // this thread's words and scales of record k: fw + k * 1 KiB (+ 512 B for
            // the second lane), sw + k * 512 B (+ 256 B); activations aw + k * astep
            uint32_t fw = stage(s) + 4u * (uint32_t)t;
            uint32_t sw = stage(s) + st.fields_bytes + 2u * (uint32_t)t;
            const uint32_t a0 = stage(s) + st.fields_bytes + st.scales_bytes;
            uint32_t aw = a0 + xa, bw = a0 + xb;
            const int n_here = min(RPS, count - r0);
#pragma unroll 4
            for (int k = 0; k < n_here; ++k) {
                const uint32_t w0 = lds32(fw), w1 = lds32(fw + 4u * PD_PAIR);
                const uint16_t h0 = lds16(sw), h1 = lds16(sw + 2u * PD_PAIR);
                const float4 va = lds128f(aw);
                if (SAME) {
                    sum = pair_record(sum, w0, w1, h0, h1, va);
                } else {
                    sum = pair_record(sum, w0, w1, h0, h1, va, lds128f(bw));
                    bw += astep;
                }
                fw += PD_TILE * 4u;
                sw += PD_TILE * 2u;
                aw += astep;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty(s));
            if (++s == D) {
                s = 0;
                fph ^= 1u;
            }
        }
        if (!ok)
            dev::flag_error(p.error, LOOM_DEVERR_TIMEOUT);
        float ya, yb;
        dev::unpack2(sum, ya, yb);
        if (livea)
            p.out[(int64_t)inst * p.lanes + la] = ok ? ya : __int_as_float(0x7fc00000);
        if (liveb)
            p.out[(int64_t)inst * p.lanes + lb] = ok ? yb : __int_as_float(0x7fc00000);
    }
}

// Direct path: plain loads, one thread per lane, records in order.
__global__ void __launch_bounds__(PD_LANES) packed_dot_direct_kernel(const PackedDeviceParams p)
{
    dev::follow_previous_kernel();
    const int32_t inst = blockIdx.y;
    const int32_t l = blockIdx.x * PD_LANES + threadIdx.x;
    const int32_t count = instance_count(p, inst);
    if (l >= p.lanes)
        return;   // over-dispatched lane: no loads, no stores
    const int32_t sl = l % p.streams;
    float sum = p.initial ? __ldg(p.initial + (int64_t)inst * p.lanes + l) : 0.f;
    for (int32_t r = 0; r < count; ++r) {
        const int64_t at = ((int64_t)inst * p.records + r) * p.lanes + l;
        const float *ap = p.rhs + (((int64_t)inst * p.records + r) * p.streams + sl) * 4;
        const float4 v = make_float4(__ldg(ap), __ldg(ap + 1), __ldg(ap + 2), __ldg(ap + 3));
        sum = record_step(sum, (uint32_t)__ldg(p.fields + at), __ldg(p.scales + at), v);
    }
    p.out[(int64_t)inst * p.lanes + l] = sum;
}

// ---- host: 3-D tensor maps ----------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled pd_encoder()
{
    static EncodeTiled fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// [outer][mid][inner] elements of `esize` bytes, box {box_inner, box_mid, 1}.
bool encode_3d(CUtensorMap *map, CUtensorMapDataType type, uint32_t esize, const void *base, uint64_t inner,
               uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid)
{
    EncodeTiled enc = pd_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {inner * esize, inner * mid * esize};
    const cuuint32_t box[3] = {box_inner, box_mid, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(map, type, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool packed_dot_stageable(const PackedParams &q)
{
    const auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    return q.lanes % 8 == 0 && q.streams >= 1 && q.streams <= PD_MAX_STAGED_STREAMS && al16(q.fields) &&
           al16(q.scales) && al16(q.rhs);
}

uint32_t packed_dot_smem_bytes(bool staged, int depth, int rps, int streams)
{
    return staged ? pd_smem_bytes(depth, rps, streams) : 0u;
}

uint32_t packed_dot_threads(bool staged) { return staged ? PD_THREADS_STAGED : PD_LANES; }

int64_t packed_dot_tiles(int64_t problems, int64_t lanes) { return problems * ((lanes + PD_TILE - 1) / PD_TILE); }

cudaError_t launch_packed_dot(const PackedParams &q, bool staged, const loom_launch &L, cudaStream_t stream)
{
    if (L.grid[0] == 0 || L.grid[1] == 0)
        return cudaSuccess;
    PackedDeviceParams p;
    p.fields = q.fields;
    p.scales = q.scales;
    p.rhs = q.rhs;
    p.problems = q.problems;
    p.records = q.records;
    p.lanes = q.lanes;
    p.streams = q.streams;
    p.counts = q.counts;
    p.count_scalar = q.count;
    p.initial = q.initial;
    p.out = q.out;
    p.error = q.error;
    p.depth = q.depth;
    p.rps = q.rps;
    p.wait_ns = q.wait_ns;
    p.inject_stall = q.inject_stall;
    if (!staged)
        return launch_with(packed_dot_direct_kernel, L, stream, p);
    CUtensorMap tf, ts, tr;
    // a box of 256 lanes x rps records of words, and of scales
    if (!encode_3d(&tf, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, q.fields, (uint64_t)q.lanes, (uint64_t)q.records,
                   (uint64_t)q.problems, PD_TILE, (uint32_t)q.rps) ||
        !encode_3d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, q.scales, (uint64_t)q.lanes, (uint64_t)q.records,
                   (uint64_t)q.problems, PD_TILE, (uint32_t)q.rps) ||
        !encode_3d(&tr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, q.rhs, (uint64_t)q.streams * 4, (uint64_t)q.records,
                   (uint64_t)q.problems, (uint32_t)q.streams * 4, (uint32_t)q.rps))
        return cudaErrorInvalidValue;
    // both lanes of a consumer thread read the same activations when PD_PAIR is a multiple of the streams
    return PD_PAIR % q.streams == 0 ? launch_with(packed_dot_staged_kernel<true>, L, stream, tf, ts, tr, p)
                                    : launch_with(packed_dot_staged_kernel<false>, L, stream, tf, ts, tr, p);
}

}  // namespace loom
