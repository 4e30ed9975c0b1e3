// grouped_gemm.cu -- persistent tcgen05/TMEM grouped GEMM over a tight
// expert-major batch, for sm_103a.
//
// TileOps PR #1738 "Separate dispatched expert compute": Summary (expert
// MLP compute for tight expert-major batches, GPU-resident row counts);
// Review follow-up (one effective grouped-GEMM kernel resolved up front; a
// device-bounded persistent row loop instead of a runtime row-policy branch;
// one fused-gated epilogue). DeepGEMM PR #394 "MegaMoE: add cluster-paired
// FP4 weight packets", Motivation: for sparse small-token work, mark one-use
// routed weight loads EVICT_FIRST.
//
// Three kernels live here:
//  * grouped_gemm_kernel -- one GEMM (gate-up or down) per launch, on a
//    single CTA per tile; the template below, in two operand placements;
//  * fused_small_kernel -- both GEMMs of the M-small path in one persistent
//    launch (16-row token tiles), optionally the whole forward (dispatch and
//    combine inside), and an MXFP8 mode whose converter warps expand E4M3
//    weights to bf16 in TMEM;
//  * grouped_gemm_pair_kernel -- the tiled placement on 2-CTA clusters,
//    tcgen05.mma.cta_group::2 of M=256 x N=256, for the largest batches.
//
// One kernel template, two placements of the operands:
//
//  * tiled (large batches): A = 128 activation rows, B = 256 weight rows
//    (gate-up: 128 gate rows + the 128 matching up rows, so SiLU(gate)*up is
//    formed in the epilogue of the same CTA; down: 256 output columns).
//    One tcgen05.mma of M=128, N=256, K=16 per K step.
//  * M-small (decode, skewed small batches): the weights go on the MMA M
//    side (128 weight rows) and a tile of 16/32/64 activation rows on N, so
//    a handful of routed rows still streams whole 128-row weight tiles at
//    full width. Gate-up issues two MMAs per K step (gate, up) into two TMEM
//    accumulators. Weight loads carry an L2 evict-first policy.
//
// Work unit = (row tile of one expert, output-column tile). Row tiles come
// from the device-resident expert_offsets: every CTA rebuilds the per-expert
// tile prefix in shared memory at start, so no host sync and no extra launch
// is needed and the schedule is identical in every CTA. Units are dealt out
// round-robin over a persistent grid (one CTA per SM).
//
// Warp roles (256 threads): warp 0 = TMA producer, warp 1 = MMA issuer,
// warp 2 = TMEM allocator, warps 4..7 = epilogue (TMEM lanes 0..127).
// Shared-memory ring of kStages stages (full/empty mbarriers); two TMEM
// accumulators so the epilogue of one unit overlaps the main loop of the
// next. Every wait is bounded: on give-up the CTA raises an abort flag,
// drains what it has in flight, frees TMEM and sets MOE_DEVERR_WAIT_TIMEOUT.
// mbarrier waits suspend up to 1 us per test (try_wait with a time hint)
// instead of re-testing in a loop, which leaves shared memory to the TMA
// writes and the MMA operand reads.
//
// Rows of a tile past the end of its expert belong to the next expert (or
// are zero-filled by TMA past the capacity): they are computed and never
// stored.
//
// Outputs: the gate-up GEMM stores h in bf16 (the rounding the MLP defines);
// the down GEMM stores y in fp32, so the only rounding between the fp32
// accumulators and the combine's fp32 sum is the final one to bf16 (on the
// tiled paths moe_forward asks for fp16 y instead, rounded once, saturating).
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kUnitRing = 8;     // persistent single-CTA GEMMs: unit ids in flight between their roles
constexpr int kBK = 64;          // K elements per stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;       // K of one tcgen05.mma kind::f16
constexpr unsigned kFull = 0xffffffffu;

struct GemmArgs {
    const int32_t *expert_offsets;
    const int32_t *perm;    // gathered activations: sorted row -> routed slot (token = slot / k)
    int k;
    void *out;          // gate-up: bf16 h[cap, n_out]; down: fp32 y[cap, n_out]
    int32_t *err;
    uint64_t wait_limit_ns;
    int E, cap, K, n_out;
    int w_rows_per_expert;
    int up_row_offset;
    int w_packed;       // weights in the PACKED layout (see include/moe.h)
    int out_f16;        // tiled down GEMM: y stored as fp16 (saturated at +-65504) instead of fp32
    int32_t *sched;     // grouped_gemm_kernel: {units handed out, CTAs at the tail}, zero at launch and at exit;
                        // null: units dealt round-robin
};

// TMA coordinates {column, row} of the 128-row weight tile starting at
// row-major weight row `wr` (a multiple of 128) for K block `kb`. Row-major:
// the tile itself. PACKED: the pre-swizzled 16 KB image of that tile and block
// (gate-up: packets of 256 lines, gate then up; down: 128 lines).
__device__ __forceinline__ int2 weight_coords(const GemmArgs &a, bool gated, int wr, int kb)
{
    if (!a.w_packed)
        return make_int2(kb * 64, wr);
    const int KB = a.K / 64;
    if (gated) {
        const int two_i = a.w_rows_per_expert, i = a.up_row_offset;
        const int e = wr / two_i, rem = wr - e * two_i;
        const int half = rem >= i ? 1 : 0;
        const int nt = (rem - half * i) >> 7;
        const long long packet = (static_cast<long long>(e) * (i >> 7) + nt) * KB + kb;
        return make_int2(0, static_cast<int>(packet * 256 + half * 128));
    }
    return make_int2(0, static_cast<int>((static_cast<long long>(wr >> 7) * KB + kb) * 128));
}

__host__ __device__ constexpr int pow2_at_least(int v)
{
    int p = 32;
    while (p < v)
        p <<= 1;
    return p;
}

template <bool kSmallM, bool kGated, int kTileRows, int kStages, int kSplitK>
struct Cfg {
    static constexpr int kActRows = kTileRows;
    static constexpr int kWRows = kSmallM ? (kGated ? 256 : 128) : 256;
    static constexpr int kActBytes = kActRows * 128;
    static constexpr int kWBytes = kWRows * 128;
    static constexpr int kStageBytes = kActBytes + kWBytes;
    static constexpr int kOutCols = (kSmallM || kGated) ? 128 : 256;    // output columns per unit
    static constexpr int kAccCols = kSmallM ? (kGated ? 2 * kTileRows : kTileRows) : 256;
    static constexpr int kTmemCols = pow2_at_least(2 * kAccCols);
    static constexpr uint32_t kIdesc = kSmallM ? idesc_bf16_f32(128, kTileRows) : idesc_bf16_f32(128, 256);
    // fp32 output (tiled down GEMM): a 32 x 36-float transpose scratch per epilogue warp
    static constexpr int kEpiScratch = (!kSmallM && !kGated) ? 4 * 32 * 36 * 4 : 0;
    static constexpr int kDynSmem = 1024 + kStages * kStageBytes + kEpiScratch;
    static_assert(kActBytes % 1024 == 0 && kWBytes % 1024 == 0, "tiles must keep 1024-byte alignment");
    static_assert(kTmemCols <= 512, "TMEM has 512 columns");
    static_assert(!kSmallM || (kTileRows % 16 == 0 && kTileRows >= 16 && kTileRows <= 256), "MMA N");
    static_assert(kSplitK == 1 || ((kSplitK == 2 || kSplitK == 4) && kSmallM && !kGated),
                  "split-K: M-small down GEMM only");
};

struct Unit {
    int e, row0, rows, n0;
};

// A CTA's ring of unit ids (kUnitRing shared slots, an mbarrier pair each):
// the TMA producer publishes the units it loads, in order; the roles after it
// (the MMA thread, converter and epilogue warps) take them in the same order.
// Each thread keeps its own cursor; every wait is bounded.
struct UnitRing {
    int *ids;
    uint64_t *full;    // a unit id published (one arrival)
    uint64_t *empty;   // every reader has taken it
    int slot;
    uint32_t phase;

    __device__ __forceinline__ UnitRing(int *i, uint64_t *f, uint64_t *e) : ids(i), full(f), empty(e), slot(0), phase(0)
    {
    }
    __device__ __forceinline__ void advance()
    {
        if (++slot == kUnitRing) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // the producer (one thread)
    __device__ __forceinline__ bool publish(int u, volatile int *abort, uint64_t limit_ns)
    {
        if (!mbar_wait_bounded(smem_u32(&empty[slot]), phase ^ 1u, abort, limit_ns))
            return false;
        ids[slot] = u;
        mbar_arrive(smem_u32(&full[slot]));
        advance();
        return true;
    }
    // a reader of one thread
    __device__ __forceinline__ bool take(int &u, volatile int *abort, uint64_t limit_ns)
    {
        if (!mbar_wait_bounded(smem_u32(&full[slot]), phase, abort, limit_ns))
            return false;
        u = ids[slot];
        mbar_arrive(smem_u32(&empty[slot]));
        advance();
        return true;
    }
    // a reader warp: lane 0 waits and takes, every lane gets the id
    __device__ __forceinline__ bool take_warp(int &u, int lane, volatile int *abort, uint64_t limit_ns)
    {
        int got = 0, v = 0;
        if (lane == 0) {
            got = mbar_wait_bounded(smem_u32(&full[slot]), phase, abort, limit_ns) ? 1 : 0;
            if (got) {
                v = ids[slot];
                mbar_arrive(smem_u32(&empty[slot]));
            }
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        u = __shfl_sync(0xffffffffu, v, 0);
        advance();
        return got != 0;
    }
};

// Largest e in [0, E) with tp[e] * scale <= u (tp non-decreasing, tp[0] = 0).
__device__ __forceinline__ int find_expert(const int *tp, int E, int u, int scale)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tp[mid] * scale <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Unit u of a grouped GEMM. Two orders, both expert-major:
// - kWeightOuter: column tile, then row tile. The row tiles of one weight tile
//   go to neighbouring CTAs, which share it in L2 (the M-small GEMMs, and the
//   CTA-pair gate-up GEMM: `large` gate-up 1079.1 vs 1093.4 us per call
//   against the other order, in one process, outputs bit-identical);
// - otherwise: row tile, then column tile. The column tiles of one row tile go
//   to neighbouring CTAs (the tiled down GEMMs: the other order measured
//   579.6 vs 573.0 us there).
template <bool kSmallM, int kTileRows, int kOutCols, bool kWeightOuter = kSmallM>
__device__ __forceinline__ Unit decode_unit(int u, const int *s_off, const int *s_tp, int E, int NT)
{
    Unit t;
    int rt_local, nt;
    if (!kWeightOuter) {
        const int rt = u / NT;
        nt = u - rt * NT;
        t.e = find_expert(s_tp, E, rt, 1);
        rt_local = rt - s_tp[t.e];
    } else {
        t.e = find_expert(s_tp, E, u, NT);
        const int local = u - s_tp[t.e] * NT;
        const int tiles = s_tp[t.e + 1] - s_tp[t.e];
        nt = local / tiles;
        rt_local = local - nt * tiles;
    }
    t.row0 = s_off[t.e] + rt_local * kTileRows;
    const int left = s_off[t.e + 1] - t.row0;
    t.rows = left < kTileRows ? left : kTileRows;
    t.n0 = nt * kOutCols;
    return t;
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return (g / (1.0f + expf(-g))) * u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// Per-expert row-tile prefix (one warp): s_tp[e] = sum_{e' < e} ceil(rows(e') / tile_rows).
__device__ __forceinline__ void build_tile_prefix(const int *s_off, int *s_tp, int E, int tile_rows, int lane)
{
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int tiles = 0;
        if (e < E) {
            int c = s_off[e + 1] - s_off[e];
            c = c < 0 ? 0 : c;
            tiles = (c + tile_rows - 1) / tile_rows;
        }
        int v = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, v, o);
            if (lane >= o)
                v += n;
        }
        if (e < E)
            s_tp[e] = carry + v - tiles;
        carry += __shfl_sync(kFull, v, 31);
    }
    if (lane == 0)
        s_tp[E] = carry;
}

// The same prefix by the whole block, for the decode kernel whose prologue is
// on the call's critical path: every warp scans its own 32-expert chunks at
// once, one warp scans the chunk totals (s_chunk, ceil(E / 32) entries), and
// every thread adds its chunk's offset. Ends with the block synchronised.
template <int kThreads>
__device__ __forceinline__ void build_tile_prefix_block(const int *s_off, int *s_tp, int *s_chunk, int E,
                                                        int tile_rows)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nchunks = (E + 31) / 32;
    for (int c = warp; c < nchunks; c += kThreads / 32) {
        const int e = c * 32 + lane;
        int tiles = 0;
        if (e < E) {
            int n = s_off[e + 1] - s_off[e];
            n = n < 0 ? 0 : n;
            tiles = (n + tile_rows - 1) / tile_rows;
        }
        int v = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, v, o);
            if (lane >= o)
                v += n;
        }
        if (e < E)
            s_tp[e] = v - tiles;   // exclusive inside the chunk
        if (lane == 31)
            s_chunk[c] = v;        // the chunk's total
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < nchunks; base += 32) {
            const int c = base + lane;
            const int total = c < nchunks ? s_chunk[c] : 0;
            int v = total;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(kFull, v, o);
                if (lane >= o)
                    v += n;
            }
            if (c < nchunks)
                s_chunk[c] = carry + v - total;
            carry += __shfl_sync(kFull, v, 31);
        }
        if (lane == 0)
            s_tp[E] = carry;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads)
        s_tp[e] += s_chunk[e >> 5];
    __syncthreads();
}

// Epilogue of a 128-row tiled unit: this thread owns accumulator row `row`
// (TMEM lane base already in t_row); the warp's 32 rows are consecutive.
// Gate-up: columns [0,128) gate, [128,256) up -> bf16 SiLU(gate)*up into h.
// Down: 256 fp32 columns into y, 32 at a time, turned through the warp's
// 32 x 36-float shared-memory scratch so that each store instruction writes
// four whole 128-byte row segments (a thread-per-row store would write 32
// rows x 16 bytes: 32 partial lines per instruction).
template <bool kGated>
__device__ __forceinline__ void tiled_epilogue(uint32_t t_row, const GemmArgs &args, int row, bool valid, int n0,
                                               float *scratch)
{
    // output columns of this unit inside n_out: a multiple of 64 (n_out and
    // n0 are), so every column chunk below lies wholly inside or outside
    const int cols = args.n_out - n0;
    if (kGated) {
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(args.out) + static_cast<size_t>(row) * args.n_out + n0;
#pragma unroll 1
        for (int c = 0; c < 128 && c < cols; c += 32) {
            uint32_t g[32], v[32];
            tmem_ld_32x32b_x32(t_row + c, g);
            tmem_ld_32x32b_x32(t_row + 128 + c, v);
            tmem_wait_ld();
            if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 o;
                    o.x = pack_bf16x2(silu_mul(__uint_as_float(g[8 * i + 0]), __uint_as_float(v[8 * i + 0])),
                                      silu_mul(__uint_as_float(g[8 * i + 1]), __uint_as_float(v[8 * i + 1])));
                    o.y = pack_bf16x2(silu_mul(__uint_as_float(g[8 * i + 2]), __uint_as_float(v[8 * i + 2])),
                                      silu_mul(__uint_as_float(g[8 * i + 3]), __uint_as_float(v[8 * i + 3])));
                    o.z = pack_bf16x2(silu_mul(__uint_as_float(g[8 * i + 4]), __uint_as_float(v[8 * i + 4])),
                                      silu_mul(__uint_as_float(g[8 * i + 5]), __uint_as_float(v[8 * i + 5])));
                    o.w = pack_bf16x2(silu_mul(__uint_as_float(g[8 * i + 6]), __uint_as_float(v[8 * i + 6])),
                                      silu_mul(__uint_as_float(g[8 * i + 7]), __uint_as_float(v[8 * i + 7])));
                    dst[i] = o;
                }
            }
        }
    } else if (args.out_f16) {
        // fp16 y: 64 columns per pass, so that each row's piece is one 128-byte line
        const int lane = threadIdx.x & 31;
        const int row0 = row - lane;
        const unsigned valid_rows = __ballot_sync(0xffffffffu, valid);
        uint4 *const mine = reinterpret_cast<uint4 *>(scratch + lane * 36);
        __half *const y = static_cast<__half *>(args.out);
        bool clipped = false;
#pragma unroll 1
        for (int c = 0; c < 256 && c < cols; c += 64) {
            uint32_t d[64];
            tmem_ld_32x32b_x32(t_row + c, *reinterpret_cast<uint32_t(*)[32]>(d));
            tmem_ld_32x32b_x32(t_row + c + 32, *reinterpret_cast<uint32_t(*)[32]>(d + 32));
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t h[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float lo = __uint_as_float(d[8 * i + 2 * j]), hi = __uint_as_float(d[8 * i + 2 * j + 1]);
                    clipped |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
                    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(hi), "f"(lo));
                }
                mine[i] = make_uint4(h[0], h[1], h[2], h[3]);
            }
            __syncwarp();
            // lanes 8m..8m+7 take row 4*it + m, 16 bytes each: one whole 128-byte line per row
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int rr = 4 * it + (lane >> 3);
                const uint4 v = *reinterpret_cast<const uint4 *>(scratch + rr * 36 + (lane & 7) * 4);
                if ((valid_rows >> rr) & 1u)
                    *reinterpret_cast<uint4 *>(y + static_cast<size_t>(row0 + rr) * args.n_out + n0 + c +
                                               (lane & 7) * 8) = v;
            }
            __syncwarp();
        }
        if (__any_sync(0xffffffffu, clipped && valid) && lane == 0)
            atomicOr(args.err, MOE_DEVERR_Y_RANGE);
    } else {
        const int lane = threadIdx.x & 31;
        const int row0 = row - lane;                       // the warp's first row
        const unsigned valid_rows = __ballot_sync(0xffffffffu, valid);
        float4 *const mine = reinterpret_cast<float4 *>(scratch + lane * 36);
        float *const y = static_cast<float *>(args.out);
#pragma unroll 1
        for (int c = 0; c < 256 && c < cols; c += 32) {
            uint32_t d[32];
            tmem_ld_32x32b_x32(t_row + c, d);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mine[i] = make_float4(__uint_as_float(d[4 * i]), __uint_as_float(d[4 * i + 1]),
                                      __uint_as_float(d[4 * i + 2]), __uint_as_float(d[4 * i + 3]));
            __syncwarp();
            // lanes 8m..8m+7 take row 4*it + m, 16 bytes each: 128 contiguous bytes per row
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int rr = 4 * it + (lane >> 3);
                const float4 v = *reinterpret_cast<const float4 *>(scratch + rr * 36 + (lane & 7) * 4);
                if ((valid_rows >> rr) & 1u)
                    *reinterpret_cast<float4 *>(y + static_cast<size_t>(row0 + rr) * args.n_out + n0 + c +
                                                (lane & 7) * 4) = v;
            }
            __syncwarp();
        }
    }
}

template <bool kSmallM, bool kGated, int kTileRows, int kStages, int kSplitK, bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                        const GemmArgs args)
{
    using C = Cfg<kSmallM, kGated, kTileRows, kStages, kSplitK>;
    static_assert(!kGather || kGated, "row gather: gate-up GEMM only");
    __shared__ __align__(16) int s_rows[kTileRows];   // gathered: token of each activation row of the unit
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ int s_unit[kUnitRing];                          // the CTA's units, in order (dynamic deal)
    __shared__ __align__(8) uint64_t bar_ufull[kUnitRing];     // a unit id published
    __shared__ __align__(8) uint64_t bar_uempty[kUnitRing];    // the MMA thread and 4 epilogue warps read it
    __shared__ int s_last;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_tp[kMaxExperts + 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = args.E;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 128);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(smem_u32(&bar_ufull[i]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), 5);
        }
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_act);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    // everything above overlaps the previous kernel's tail; its outputs
    // (expert_offsets, the activation rows) are read only after this wait.
    // Dependents are released only when this CTA is done (end of kernel):
    // released early, their CTAs would sit on the SMs next to this
    // persistent grid and take issue slots from it.
    pdl_wait();
    for (int i = threadIdx.x; i <= E; i += kThreads)
        s_off[i] = args.expert_offsets[i];
    __syncthreads();
    if (warp == 3)
        build_tile_prefix(s_off, s_tp, E, kTileRows, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    const int NT = (args.n_out + C::kOutCols - 1) / C::kOutCols;   // the last tile may be partly past n_out
    const int total_units = s_tp[E] * NT * kSplitK;
    const int k_blocks = args.K / kBK / kSplitK;   // K blocks of one unit
    // More units than CTAs (and the counters given): units beyond each CTA's
    // first come from a GPU-wide count, unit = gridDim.x + its old value,
    // asked for one unit ahead; the producer publishes them on a ring of
    // shared slots that the MMA thread and the epilogue warps read in order.
    // CTAs whose units run faster take more of them. Otherwise every role
    // deals itself units blockIdx.x, + gridDim.x, ... and the ring is unused.
    // In one process, against round-robin units (two boxes): the down GEMMs
    // -3.4% (Zipf small batch, M-small) and -0.5 to -0.7% (prefill, tiled),
    // prefill's gate-up -0.6%. The M-small gate-up GEMM keeps round-robin
    // units (+1.2 to 1.4% with the count): there the token tiles of one weight
    // tile, dealt side by side, read it from L2 together.
    const bool dynamic =
        !(kSmallM && kGated) && args.sched != nullptr && total_units > static_cast<int>(gridDim.x);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol_w = kSmallM ? l2_policy_evict_first() : l2_policy_evict_normal();
        const uint64_t pol_a = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;  // per stage: a load in flight, and its phase parity
        bool ok = true;
        UnitRing ring(s_unit, bar_ufull, bar_uempty);
        int u = blockIdx.x;
        while (true) {
            if (dynamic && lane == 0 && !ring.publish(ok ? u : total_units, abort_flag, args.wait_limit_ns))
                ok = false;
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok || u >= total_units)
                break;
            // the unit after this one: asked for after the release above, read after this unit's loads
            int nxt = u + static_cast<int>(gridDim.x);
            if (dynamic && lane == 0)
                nxt = static_cast<int>(gridDim.x) + atomicAdd(args.sched, 1);
            const Unit t = decode_unit<kSmallM, kTileRows, C::kOutCols>(u / kSplitK, s_off, s_tp, E, NT);
            const int kb0 = (u % kSplitK) * k_blocks;
            const int w_row0 = t.e * args.w_rows_per_expert + t.n0;
            const int w_row1 = kGated ? t.e * args.w_rows_per_expert + args.up_row_offset + t.n0 : w_row0 + 128;
            if (kGather) {
                // token of every activation row of the tile; rows past the expert read token 0 and are never stored
                for (int i = lane; i < kTileRows; i += 32)
                    s_rows[i] = i < t.rows ? __ldg(args.perm + t.row0 + i) / args.k : 0;
                __syncwarp();
            }
            if (lane == 0) {
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, abort_flag, args.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&bar_full[stage]);
                    const uint32_t w_dst = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t a_dst = w_dst + C::kWBytes;
                    mbar_arrive_expect_tx(full, C::kStageBytes);
                    const int kc = (kb0 + kb) * kBK;
                    const int2 w0 = weight_coords(args, kGated, w_row0, kb0 + kb);
                    tma_load_2d(w_dst, &tm_w, full, w0.x, w0.y, pol_w);
                    if (C::kWRows == 256) {
                        const int2 w1 = weight_coords(args, kGated, w_row1, kb0 + kb);
                        tma_load_2d(w_dst + 128 * 128, &tm_w, full, w1.x, w1.y, pol_w);
                    }
                    if (kGather) {
#pragma unroll
                        for (int g = 0; g < kTileRows / 4; ++g)
                            tma_gather4(a_dst + g * 512, &tm_act, full, kc, reinterpret_cast<const int4 *>(s_rows)[g],
                                        pol_a);
                    } else {
                        tma_load_2d(a_dst, &tm_act, full, kc, t.row0, pol_a);
                    }
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;   // s_rows is rewritten only after lane 0 issued
            u = __shfl_sync(kFull, nxt, 0);
        }
        if (!ok && lane == 0) {
            // give-up path: let every load still in flight land before the CTA exits
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s)) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(smem_u32(&bar_full[s]), (issued_parity >> s) & 1u) &&
                           global_timer_ns() - t0 < args.wait_limit_ns) {
                    }
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            UnitRing ring(s_unit, bar_ufull, bar_uempty);
            for (int local = 0; ok; ++local) {
                int u = static_cast<int>(blockIdx.x + local * gridDim.x);
                if (dynamic && !ring.take(u, abort_flag, args.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                if (u >= total_units)
                    break;
                const int buf = local & 1;
                const uint32_t use = (local >> 1) & 1;
                if (!mbar_wait_bounded(smem_u32(&bar_tempty[buf]), use ^ 1u, abort_flag, args.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * C::kAccCols;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&bar_full[stage]), phase, abort_flag, args.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t w_addr = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t a_addr = w_addr + C::kWBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        const uint64_t a_desc = smem_desc_kmajor_sw128(a_addr + kk * 32);
                        const uint64_t w_desc = smem_desc_kmajor_sw128(w_addr + kk * 32);
                        if (!kSmallM) {
                            umma_bf16(d_tmem, a_desc, w_desc, C::kIdesc, acc);
                        } else {
                            umma_bf16(d_tmem, w_desc, a_desc, C::kIdesc, acc);
                            if (kGated) {
                                const uint64_t up_desc = smem_desc_kmajor_sw128(w_addr + 128 * 128 + kk * 32);
                                umma_bf16(d_tmem + kTileRows, up_desc, a_desc, C::kIdesc, acc);
                            }
                        }
                    }
                    umma_commit(smem_u32(&bar_empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok)
                    umma_commit(smem_u32(&bar_tfull[buf]));
            }
            // every MMA this thread issued must be complete before TMEM is freed
            umma_commit(smem_u32(&bar_drain));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&bar_drain), 0) && global_timer_ns() - t0 < args.wait_limit_ns) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;  // TMEM lanes [32q, 32q + 32)
        UnitRing ring(s_unit, bar_ufull, bar_uempty);
        for (int local = 0;; ++local) {
            int u = static_cast<int>(blockIdx.x + local * gridDim.x);
            if (dynamic && !ring.take_warp(u, lane, abort_flag, args.wait_limit_ns))
                break;
            if (u >= total_units)
                break;
            const Unit t = decode_unit<kSmallM, kTileRows, C::kOutCols>(u / kSplitK, s_off, s_tp, E, NT);
            const int buf = local & 1;
            const uint32_t use = (local >> 1) & 1;
            int ok = 0;
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&bar_tfull[buf]), use, abort_flag, args.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + buf * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
            if (!kSmallM) {
                const int r = q * 32 + lane;
                const int row = t.row0 + r;
                tiled_epilogue<kGated>(t_row, args, row, r < t.rows && row >= 0 && row < args.cap, t.n0,
                                       reinterpret_cast<float *>(smem + kStages * C::kStageBytes) + q * 32 * 36);
            } else {
                // lane = weight row = output column t.n0 + 32q + lane; TMEM column = token row of the tile
                const int col = t.n0 + q * 32 + lane;
#pragma unroll 1
                for (int c = 0; c < kTileRows; c += 16) {
                    uint32_t g[16], v[16];
                    tmem_ld_32x32b_x16(t_row + c, g);
                    if (kGated)
                        tmem_ld_32x32b_x16(t_row + kTileRows + c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int rr = c + i;
                        const int row = t.row0 + rr;
                        if (rr < t.rows && row >= 0 && row < args.cap && col < args.n_out) {
                            const size_t o = static_cast<size_t>(row) * args.n_out + col;
                            if (kGated)
                                static_cast<__nv_bfloat16 *>(args.out)[o] =
                                    __float2bfloat16_rn(silu_mul(__uint_as_float(g[i]), __uint_as_float(v[i])));
                            else   // K part u % kSplitK to its own buffer (summed in part order later)
                                static_cast<float *>(args.out)[static_cast<size_t>(u % kSplitK) * args.cap *
                                                                   args.n_out + o] = __uint_as_float(g[i]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_tempty[buf]));
        }
    }

    tc_fence_before();
    __syncthreads();
    // the last CTA out returns the count to zero (every CTA's last atomic on
    // it precedes its own add here, in the same thread); a dependent launch
    // reads it only after its wait on this grid
    if (threadIdx.x == 0 && args.sched && dynamic)
        s_last = atom_add_acq_rel_gpu(args.sched + 1, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (threadIdx.x == 0 && args.sched && dynamic && s_last) {
        args.sched[0] = 0;
        args.sched[1] = 0;
    }
    pdl_trigger();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    if (threadIdx.x == 0 && s_abort)
        atomicOr(args.err, MOE_DEVERR_WAIT_TIMEOUT);
}


// ------------------------------------------------------------------ fused M-small expert MLP
//
// Both M-small GEMMs of moe_forward in one persistent launch. Units are the
// gate-up units (rows gathered from x with tile::gather4, SiLU(gate)*up -> h)
// followed by the down units (h -> y), in one list. CTA b takes unit b first;
// every later unit comes from a GPU-wide count (unit = gridDim.x + the
// count's old value), which the producer asks for one unit ahead so that the
// atomic's round trip hides behind the current unit's loads. CTAs whose units
// run faster (an SM nearer its weights' memory, fewer gate-up units) take
// more units, and the CTAs finish within about one unit of each other; dealt
// round-robin, they had finished up to 10 us (one token) and 80 us (eight
// tokens) apart. Units leave the count in list order, so every gate-up unit
// has an owner before any down unit is handed out, and each CTA finishes its
// gate-up units before any of its down units. The producer publishes each unit
// id on a ring of kUnitRing shared slots, which the MMA thread, the converter
// warps and the epilogue warps read in order (one mbarrier pair per slot). A down
// unit of expert e needs every gate-up unit of e: each epilogue warp makes
// its h stores visible (every lane fences, then one lane does a release add
// on ready[e]); the producer of a down unit waits with a bounded acquire loop
// until ready[e] = 4 warps * tiles(e) * I/128, then fences the async proxy
// before its TMA reads of h. No wait can be circular: gate-up units wait on nothing but
// their own pipeline, and the grid is one CTA per SM, all resident once the
// (independent) previous kernel leaves. The count and ready[] are zero when
// the kernel starts and again when it ends. The GPU-wide tail between the two
// GEMMs disappears: an SM moves on to down units of finished experts while
// others still stream gate-up weights. The last CTA to leave clears ready[]
// and the count.
// A stage holds 32 KB of weights either way: the gate and up tiles of one K
// block, or two K blocks of a down tile (with two token-tile slots), so the
// down units keep as many weight bytes in flight as the gate-up units.
//
// Whole-forward form (kMega): the same kernel is all of moe_forward. Every
// CTA first runs the local dispatch of the call's few routed slots itself
// (histogram, scan, stable scatter into shared memory; CTA 0 also writes
// expert_offsets and perm for the caller), so no other kernel precedes the
// GEMMs. Each CTA, once through with its GEMM units, counts itself on a
// GPU-wide count (one add per CTA, not one per unit: the polls and adds on
// that one address stay few); when every CTA has, each combines its share of
// tokens x 1024 columns. The last CTA
// to leave returns every counter to zero (FlashInfer moe_ep page, launch-path
// notes: workspaces are allocated zeroed and the kernel cleans its
// counters and flags at its tail), also after a timed-out wait, so repeated
// calls need no memset. A down GEMM that splits K (2 or 4 parts, in both
// forms) writes each part to its own fp32 buffer and the combine adds them
// in part order, so y needs no zeroing and the sum is deterministic.
//
// MXFP8 weights (kFp8): a weight block is 128 K elements (one 128-byte row of
// E4M3 codes) plus its 4 scale bytes per row; a stage holds two such 16 KB
// tiles (gate and up, or two K blocks of a down tile), their two 512-byte
// scale blocks and the matching bf16 token tiles (64-wide K blocks). Eight
// converter warps (two per TMEM lane quarter, one per weight tile) expand
// each row's 128 codes times its scales to bf16, exactly, into a ring of TMEM
// slots (sixteen warps, splitting K, measured 9-13% slower); the MMAs read their A operand (the weights) from there and the token
// tile from shared memory as before. Weight bytes in flight per SM stay at
// 32 KB per stage, which now hold twice the K of the bf16 stages.
template <int kTileRows, int kStages, bool kFp8 = false>
struct FusedCfg {
    static constexpr int kConvWarps = kFp8 ? 8 : 0;          // fp8: converter warps (8 or 16)
    static constexpr int kThreadsCta = 256 + 32 * kConvWarps;
    static constexpr int kWK = kFp8 ? 128 : 64;               // K elements of one weight block
    static constexpr int kActSlot = kTileRows * 128;          // one 64-wide K block of the token tile
    static constexpr int kActSlots = kFp8 ? 4 : 2;
    static constexpr int kWBytes = 256 * 128;                 // gate + up tile, or two K blocks of a down tile
    static constexpr int kScaleOffset = kWBytes + kActSlots * kActSlot;
    static constexpr int kStageBytes = kScaleOffset + (kFp8 ? 1024 : 0);
    static constexpr int kAccCols = 2 * kTileRows;           // gate-up: two accumulators; down: one
    static constexpr int kASlotCols = 128;                    // fp8: the two bf16 weight tiles of one stage
    static constexpr int kASlots = kFp8 ? (512 - 2 * kAccCols) / kASlotCols : 0;
    static constexpr int kTmemCols = kFp8 ? 512 : pow2_at_least(2 * kAccCols);
    static constexpr uint32_t kIdesc = idesc_bf16_f32(128, kTileRows);
    static constexpr int kDynSmem = 1024 + kStages * kStageBytes;
    static_assert(kTileRows % 16 == 0 && kTileRows >= 16 && kTileRows <= 64, "token tile");
    static_assert(kActSlot % 1024 == 0 && kStageBytes % 1024 == 0, "1024-byte aligned tiles");
    static_assert(!kFp8 || kASlots >= 2, "fp8: at least two TMEM weight slots");
};

struct FusedArgs {
    GemmArgs up;       // gate-up: act = x (gathered), out = h, K = H, n_out = I
    GemmArgs down;     // down: act = h, out = y, K = I, n_out = H
    int32_t *ready;    // [E] finished gate-up units per expert, zero at launch and at exit
    int32_t *exits;    // CTAs at the tail, zero at launch and at exit
    int32_t *next_unit;   // units handed out beyond each CTA's first, zero at launch and at exit
    const uint8_t *sc13;   // MXFP8: scale blocks of W13 and W2 (512 B per 128-row tile and 128-wide K block)
    const uint8_t *sc2;
    // whole-forward form only
    const int32_t *ids;            // [T_max, k] routed expert of each slot, -1 = dropped
    const float *topk_w;           // [T_max, k]
    const int32_t *d_num_tokens;   // device T, or null for T_max
    int T_max;
    int slots_max;                 // T_max * k: size of the shared-memory perm / inv tables
    int32_t *expert_offsets_out;   // [E + 1] for the caller
    int32_t *perm_out;             // [cap] for the caller
    __nv_bfloat16 *out;            // [T_max, H]
    int32_t *done;                 // CTAs through with their GEMM units, zero at launch and at exit
    // 1: the call's dispatch kernel runs beside this kernel (it writes
    // expert_offsets, perm and inv for the caller and the combine) and the
    // combine kernel after it: no in-kernel combine, and no wait for the
    // dispatch before the GEMM units (this kernel's own local dispatch of the
    // same slots gives the same tables)
    int combine_apart;
    // MXFP8, separate form: the gate-up activation rows come from a sorted
    // copy (x_sorted, one 2-D TMA box of kTileRows rows per 64-wide K block)
    // instead of tile::gather4 from x through perm
    int act_sorted;
};

// Local dispatch of all routed slots inside one CTA (every CTA of the
// whole-forward kernel runs it on the same input and gets the same tables):
// s_off[E+1] = exclusive prefix of the per-expert slot counts, s_perm[row] =
// slot in ascending slot order inside each expert (stable scatter), s_inv[slot]
// = row or -1. s_cur[E] is scratch. The ids of all T_max tokens are fetched
// together with T (those past T are never used), so the prologue pays one
// global round trip. Returns T.
template <int kThreads>
__device__ int cta_dispatch(const FusedArgs &fa, int E, int *s_off, int *s_cur, int *s_perm, int *s_inv)
{
    const bool write_outputs = !fa.combine_apart;   // else the dispatch kernel beside writes them
    static_assert(4 * kThreads >= kMaxExperts, "the scan covers four experts per thread");
    __shared__ int s_warp_sum[kThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = fa.up.k;
    int T = fa.d_num_tokens ? *fa.d_num_tokens : fa.T_max;
    for (int s = tid; s < fa.slots_max; s += kThreads)
        s_inv[s] = __ldg(fa.ids + s);                  // ids staged in s_inv, replaced by rows below
    for (int e = tid; e < E; e += kThreads)
        s_cur[e] = 0;
    T = T < 0 ? 0 : (T > fa.T_max ? fa.T_max : T);
    const int R = T * k;
    __syncthreads();
    bool bad = false;
    for (int s = tid; s < R; s += kThreads) {
        const int e = s_inv[s];
        if (e >= 0 && e < E)
            atomicAdd(&s_cur[e], 1);
        else if (e != -1)
            bad = true;
    }
    if (bad && blockIdx.x == 0 && write_outputs)
        atomicOr(fa.up.err, MOE_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    // exclusive scan over experts, four consecutive experts per thread (E <= 1024)
    int c[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = 4 * tid + i;
        c[i] = e < E ? s_cur[e] : 0;
        sum += c[i];
    }
    int v = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += n;
    }
    if (lane == 31)
        s_warp_sum[warp] = v;
    __syncthreads();
    int before = v - sum;
    for (int w = 0; w < warp; ++w)
        before += s_warp_sum[w];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = 4 * tid + i;
        if (e < E) {
            s_off[e] = before;
            s_cur[e] = before;
        }
        before += c[i];
    }
    if (tid == kThreads - 1)
        s_off[E] = before;
    __syncthreads();
    if (warp == 0) {
        // 32 slots at a time in ascending order: a slot's row is its expert's
        // cursor plus the same-expert slots on lower lanes
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < R; base += 32) {
            const int s = base + lane;
            const int e = s < R ? s_inv[s] : -1;
            const bool valid = e >= 0 && e < E;
            const unsigned peers = __match_any_sync(kFull, valid ? e : -1 - lane);
            const int rank = __popc(peers & lt);
            if (valid) {
                const int row = s_cur[e] + rank;
                s_perm[row] = s;
                s_inv[s] = row;
            } else if (s < R) {
                s_inv[s] = -1;
            }
            __syncwarp();
            if (valid && rank == 0)
                s_cur[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && write_outputs) {
        for (int i = tid; i <= E; i += kThreads)
            fa.expert_offsets_out[i] = s_off[i];
        for (int r = tid; r < s_off[E]; r += kThreads)
            fa.perm_out[r] = s_perm[r];
    }
    return T;
}

// This CTA's share of the combine: work items of one token x 1024 columns,
// out[t, m] = bf16( sum_j w[t, j] * y[inv[t*k + j], m] ), fp32, j ascending,
// no fused multiply-add (the arithmetic of combine_kernel). y was written by
// other CTAs during this launch: read through L2 (ld.global.cg), never the
// read-only path. With a split down GEMM the row is y0 + y1.
template <int kSplitDown, int kThreads>
__device__ void cta_combine(const FusedArgs &fa, const int *s_inv, int T)
{
    const int k = fa.up.k;
    const int H = fa.down.n_out;
    const int vec = H / 4;
    const int groups = (vec + kThreads - 1) / kThreads;
    const float4 *y0 = static_cast<const float4 *>(fa.down.out);
    const size_t part = static_cast<size_t>(fa.down.cap) * vec;   // float4s between K parts
    const long long items = static_cast<long long>(T) * groups;
    for (long long item = blockIdx.x; item < items; item += gridDim.x) {
        const int t = static_cast<int>(item / groups);
        const int c = static_cast<int>(item % groups) * kThreads + threadIdx.x;
        if (c >= vec)
            continue;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < k; j0 += 4) {
            float4 a[4];
            int row[4];
            float wj[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                row[q] = (j0 + q < k) ? s_inv[t * k + j0 + q] : -1;
                wj[q] = (j0 + q < k) ? __ldg(fa.topk_w + static_cast<size_t>(t) * k + j0 + q) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (row[q] >= 0) {
                    // the row is the sum of its K parts in part order, as moe_expert_compute reduces them
                    const size_t i = static_cast<size_t>(row[q]) * vec + c;
                    a[q] = __ldcg(y0 + i);
#pragma unroll
                    for (int pp = 1; pp < kSplitDown; ++pp) {
                        const float4 b = __ldcg(y0 + pp * part + i);
                        a[q].x = __fadd_rn(a[q].x, b.x);
                        a[q].y = __fadd_rn(a[q].y, b.y);
                        a[q].z = __fadd_rn(a[q].z, b.z);
                        a[q].w = __fadd_rn(a[q].w, b.w);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (row[q] < 0)
                    continue;
                acc[0] = __fadd_rn(acc[0], __fmul_rn(wj[q], a[q].x));
                acc[1] = __fadd_rn(acc[1], __fmul_rn(wj[q], a[q].y));
                acc[2] = __fadd_rn(acc[2], __fmul_rn(wj[q], a[q].z));
                acc[3] = __fadd_rn(acc[3], __fmul_rn(wj[q], a[q].w));
            }
        }
        uint2 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        reinterpret_cast<uint2 *>(fa.out)[static_cast<size_t>(t) * vec + c] = o;
    }
}

template <int kTileRows, int kStages, int kSplitDown, bool kMega, bool kFp8>
__global__ void __launch_bounds__(FusedCfg<kTileRows, kStages, kFp8>::kThreadsCta, 1)
    fused_small_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w13,
                       const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w2,
                       const FusedArgs fa)
{
    using C = FusedCfg<kTileRows, kStages, kFp8>;
    constexpr int kThreads = C::kThreadsCta;
    constexpr int kASlotsRing = kFp8 ? C::kASlots : 1;
    // the whole-forward form keeps its expert tables (sized by E and T_max * k)
    // in dynamic shared memory after the stages
    constexpr int kStaticTable = kMega ? 1 : kMaxExperts + 1;
    __shared__ __align__(16) int s_rows[kTileRows];
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(8) uint64_t bar_conv_full[kASlotsRing];    // fp8: weights expanded into a TMEM slot
    __shared__ __align__(8) uint64_t bar_conv_empty[kASlotsRing];   // fp8: the MMAs reading a slot are done
    __shared__ int s_unit[kUnitRing];                                 // the CTA's units, in order
    __shared__ __align__(8) uint64_t bar_ufull[kUnitRing];           // a unit id published
    __shared__ __align__(8) uint64_t bar_uempty[kUnitRing];          // every role has read it
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_T;
    __shared__ int s_last;
    __shared__ int s_off_static[kStaticTable];
    __shared__ int s_tp_static[kStaticTable];
    __shared__ int s_chunk[(kMaxExperts + 31) / 32];   // tile prefix: the 32-expert chunks' offsets

    const GemmArgs &A1 = fa.up;
    const GemmArgs &A2 = fa.down;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = A1.E;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int *const tables = reinterpret_cast<int *>(smem + kStages * C::kStageBytes);
    int *const s_off = kMega ? tables : s_off_static;
    int *const s_tp = kMega ? tables + (E + 1) : s_tp_static;
    int *const s_perm = tables + 2 * (E + 1);
    int *const s_inv = s_perm + fa.slots_max;
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 128);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(smem_u32(&bar_ufull[i]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), 5 + C::kConvWarps);   // MMA thread, 4 epilogue warps, converters
        }
        if (kFp8)
            for (int i = 0; i < kASlotsRing; ++i) {
                mbar_init(smem_u32(&bar_conv_full[i]), C::kConvWarps);
                mbar_init(smem_u32(&bar_conv_empty[i]), 1);
            }
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w13);
        tma_prefetch_desc(&tm_h);
        tma_prefetch_desc(&tm_w2);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&s_tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    // With the dispatch kernel beside it, the kernel needs nothing the
    // dispatch writes: it waits for it only before releasing its dependents.
    if (!(kMega && fa.combine_apart))
        pdl_wait();
    if (kMega) {
        const int T = cta_dispatch<kThreads>(fa, E, s_off, s_tp, s_perm, s_inv);
        if (threadIdx.x == 0)
            s_T = T;
    } else {
        for (int i = threadIdx.x; i <= E; i += kThreads)
            s_off[i] = A1.expert_offsets[i];
    }
    __syncthreads();
    // bf16: the block-wide prefix. MXFP8: one warp's, as before (measured with
    // the block-wide one: decode T=8 749.4 vs 680.5 us, T=1 127.4 vs 118.4 us;
    // the converter warps' schedule, which sets that kernel's pace, came out
    // slower)
    if constexpr (kFp8) {
        if (warp == 3)
            build_tile_prefix(s_off, s_tp, E, kTileRows, lane);
    } else {
        build_tile_prefix_block<kThreads>(s_off, s_tp, s_chunk, E, kTileRows);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    const int NT1 = (A1.n_out + 127) / 128;         // gate-up column tiles (ceil(I / 128))
    const int NT2 = (A2.n_out + 127) / 128;         // down column tiles (ceil(H / 128))
    const int units1 = s_tp[E] * NT1;
    const int total_units = units1 + s_tp[E] * NT2 * kSplitDown;
    const int kb1 = A1.K / C::kWK;
    const int kb2 = A2.K / C::kWK / kSplitDown;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol_w = l2_policy_evict_first();
        const uint64_t pol_a = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        bool ok = true;
        UnitRing ring(s_unit, bar_ufull, bar_uempty);
        int u = blockIdx.x;
        const bool dynamic = units1 > static_cast<int>(gridDim.x);
        while (true) {
            if (lane == 0 && !ring.publish(ok ? u : total_units, abort_flag, A1.wait_limit_ns))
                ok = false;
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok || u >= total_units)
                break;
            // the unit after this one: asked for after the release above, read after this unit's loads
            int nxt = u + static_cast<int>(gridDim.x);
            if (dynamic && lane == 0)
                nxt = static_cast<int>(gridDim.x) + atomicAdd(fa.next_unit, 1);
            const bool up = u < units1;
            const int v = up ? u : u - units1;
            const Unit t = up ? decode_unit<true, kTileRows, 128>(v, s_off, s_tp, E, NT1)
                              : decode_unit<true, kTileRows, 128>(v / kSplitDown, s_off, s_tp, E, NT2);
            const int kb0 = up ? 0 : (v % kSplitDown) * kb2;
            const int steps = up ? kb1 : (kb2 + 1) / 2;   // down: two K blocks per stage
            // bf16 gate-up units gathering from x: the first stage's weights do not
            // depend on the tile's rows, so lane 0 requests them while the lanes
            // read the rows' slots (the stage completes on the same count)
            bool pre = false;
            if (!kFp8 && up && !fa.act_sorted) {
                static_assert(kFp8 || kTileRows <= 32, "one row per lane");
                const int slot = lane < t.rows && lane < kTileRows
                                     ? (kMega ? s_perm[t.row0 + lane] : __ldg(A1.perm + t.row0 + lane))
                                     : 0;
                if (lane == 0 && ok && steps > 0) {
                    if (mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, abort_flag, A1.wait_limit_ns)) {
                        const uint32_t full = smem_u32(&bar_full[stage]);
                        const uint32_t w_dst = smem_u32(smem + stage * C::kStageBytes);
                        mbar_arrive_expect_tx(full, C::kWBytes + C::kActSlot);
                        const int wr = t.e * A1.w_rows_per_expert + t.n0;
                        const int2 g = weight_coords(A1, true, wr, 0);
                        const int2 w = weight_coords(A1, true, wr + A1.up_row_offset, 0);
                        tma_load_2d(w_dst, &tm_w13, full, g.x, g.y, pol_w);
                        tma_load_2d(w_dst + 128 * 128, &tm_w13, full, w.x, w.y, pol_w);
                        pre = true;
                    } else {
                        ok = false;
                    }
                }
                if (lane < kTileRows)
                    s_rows[lane] = slot / A1.k;
                __syncwarp();
            } else if (up && !fa.act_sorted) {
                for (int i = lane; i < kTileRows; i += 32)
                    s_rows[i] = i < t.rows ? (kMega ? s_perm[t.row0 + i] : __ldg(A1.perm + t.row0 + i)) / A1.k : 0;
                __syncwarp();
            }
            if (lane == 0) {
                if (!up) {
                    // every gate-up unit of this expert (4 epilogue warps each) must have stored its h rows
                    const int need = (s_tp[t.e + 1] - s_tp[t.e]) * NT1 * 4;
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_gpu(fa.ready + t.e) < need) {
                        if (*abort_flag || global_timer_ns() - t0 > A1.wait_limit_ns) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                    }
                    fence_proxy_async_global();
                }
                for (int st = 0; ok && st < steps; ++st) {
                    const bool pre_st = pre && st == 0;   // this stage's slot and weights already taken
                    if (!pre_st &&
                        !mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, abort_flag, A1.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&bar_full[stage]);
                    const uint32_t w_dst = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t a_dst = w_dst + C::kWBytes;
                    const uint32_t sc_dst = w_dst + C::kScaleOffset;
                    if (kFp8 && up) {
                        // gate and up code tiles of K block st, their scales, two token K blocks
                        mbar_arrive_expect_tx(full, C::kWBytes + 1024 + 2 * C::kActSlot);
                        const int wr = t.e * A1.w_rows_per_expert + t.n0;
                        const long long kbt = A1.K / 128;
                        tma_load_2d(w_dst, &tm_w13, full, st * 128, wr, pol_w);
                        tma_load_2d(w_dst + 128 * 128, &tm_w13, full, st * 128, wr + A1.up_row_offset, pol_w);
                        bulk_load(sc_dst, fa.sc13 + ((wr / 128) * kbt + st) * 512, 512, full, pol_w);
                        bulk_load(sc_dst + 512, fa.sc13 + (((wr + A1.up_row_offset) / 128) * kbt + st) * 512, 512,
                                  full, pol_w);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (fa.act_sorted) {   // the tile's rows of x_sorted, one box (the same bytes)
                                tma_load_2d(a_dst + j * C::kActSlot, &tm_x, full, st * 128 + 64 * j, t.row0, pol_a);
                            } else {
#pragma unroll
                                for (int q = 0; q < kTileRows / 4; ++q)
                                    tma_gather4(a_dst + j * C::kActSlot + q * 512, &tm_x, full, st * 128 + 64 * j,
                                                reinterpret_cast<const int4 *>(s_rows)[q], pol_a);
                            }
                        }
                    } else if (kFp8) {
                        const int nkb = (2 * st + 1 < kb2) ? 2 : 1;
                        mbar_arrive_expect_tx(full, nkb * (C::kWBytes / 2 + 512 + 2 * C::kActSlot));
                        const int wr = t.e * A2.w_rows_per_expert + t.n0;
                        const long long kbt = A2.K / 128;
                        for (int j = 0; j < nkb; ++j) {
                            const int kb = kb0 + 2 * st + j;
                            tma_load_2d(w_dst + j * 128 * 128, &tm_w2, full, kb * 128, wr, pol_w);
                            bulk_load(sc_dst + j * 512, fa.sc2 + ((wr / 128) * kbt + kb) * 512, 512, full, pol_w);
                            tma_load_2d(a_dst + (2 * j) * C::kActSlot, &tm_h, full, kb * 128, t.row0, pol_a);
                            tma_load_2d(a_dst + (2 * j + 1) * C::kActSlot, &tm_h, full, kb * 128 + 64, t.row0,
                                        pol_a);
                        }
                    } else if (up) {
                        if (!pre_st) {
                            mbar_arrive_expect_tx(full, C::kWBytes + C::kActSlot);
                            const int wr = t.e * A1.w_rows_per_expert + t.n0;
                            const int2 g = weight_coords(A1, true, wr, st);
                            const int2 w = weight_coords(A1, true, wr + A1.up_row_offset, st);
                            tma_load_2d(w_dst, &tm_w13, full, g.x, g.y, pol_w);
                            tma_load_2d(w_dst + 128 * 128, &tm_w13, full, w.x, w.y, pol_w);
                        }
#pragma unroll
                        for (int q = 0; q < kTileRows / 4; ++q)
                            tma_gather4(a_dst + q * 512, &tm_x, full, st * kBK,
                                        reinterpret_cast<const int4 *>(s_rows)[q], pol_a);
                    } else {
                        const int nkb = (2 * st + 1 < kb2) ? 2 : 1;
                        mbar_arrive_expect_tx(full, nkb * (C::kWBytes / 2 + C::kActSlot));
                        for (int j = 0; j < nkb; ++j) {
                            const int kb = kb0 + 2 * st + j;
                            const int2 d = weight_coords(A2, false, t.e * A2.w_rows_per_expert + t.n0, kb);
                            tma_load_2d(w_dst + j * 128 * 128, &tm_w2, full, d.x, d.y, pol_w);
                            tma_load_2d(a_dst + j * C::kActSlot, &tm_h, full, kb * kBK, t.row0, pol_a);
                        }
                    }
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            u = __shfl_sync(kFull, nxt, 0);
        }
        if (!ok && lane == 0) {
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s)) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(smem_u32(&bar_full[s]), (issued_parity >> s) & 1u) &&
                           global_timer_ns() - t0 < A1.wait_limit_ns) {
                    }
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int slot = 0;
            uint32_t slot_phase = 0;
            bool ok = true;
            UnitRing ring(s_unit, bar_ufull, bar_uempty);
            for (int local = 0; ok; ++local) {
                int u = total_units;
                if (!ring.take(u, abort_flag, A1.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                if (u >= total_units)
                    break;
                const bool up = u < units1;
                const int steps = up ? kb1 : (kb2 + 1) / 2;
                const int buf = local & 1;
                const uint32_t use = (local >> 1) & 1;
                if (!mbar_wait_bounded(smem_u32(&bar_tempty[buf]), use ^ 1u, abort_flag, A1.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * C::kAccCols;
                for (int st = 0; st < steps; ++st) {
                    if (!mbar_wait_bounded(smem_u32(&bar_full[stage]), phase, abort_flag, A1.wait_limit_ns) ||
                        (kFp8 && !mbar_wait_bounded(smem_u32(&bar_conv_full[slot]), slot_phase, abort_flag,
                                                    A1.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t w_addr = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t a_addr = w_addr + C::kWBytes;
                    if (kFp8) {
                        // weights (A) from the TMEM slot the converters filled, 8 K steps of 16 per block
                        const uint32_t a_tm = tmem_base + 2 * C::kAccCols + slot * C::kASlotCols;
                        const int nkb = up ? 1 : ((2 * st + 1 < kb2) ? 2 : 1);
                        for (int j = 0; j < nkb; ++j) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t acc = (st > 0 || j > 0 || kk > 0) ? 1u : 0u;
                                const uint64_t b_desc =
                                    smem_desc_kmajor_sw128(a_addr + (2 * j + (kk >> 2)) * C::kActSlot + (kk & 3) * 32);
                                umma_bf16_tmem_a(d_tmem, a_tm + 64 * j + 8 * kk, b_desc, C::kIdesc, acc);
                                if (up)
                                    umma_bf16_tmem_a(d_tmem + kTileRows, a_tm + 64 + 8 * kk, b_desc, C::kIdesc, acc);
                            }
                        }
                        umma_commit(smem_u32(&bar_conv_empty[slot]));
                        if (++slot == kASlotsRing) {
                            slot = 0;
                            slot_phase ^= 1u;
                        }
                    } else if (up) {
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                            const uint32_t acc = (st > 0 || kk > 0) ? 1u : 0u;
                            const uint64_t a_desc = smem_desc_kmajor_sw128(a_addr + kk * 32);
                            umma_bf16(d_tmem, smem_desc_kmajor_sw128(w_addr + kk * 32), a_desc, C::kIdesc, acc);
                            umma_bf16(d_tmem + kTileRows, smem_desc_kmajor_sw128(w_addr + 128 * 128 + kk * 32),
                                      a_desc, C::kIdesc, acc);
                        }
                    } else {
                        const int nkb = (2 * st + 1 < kb2) ? 2 : 1;
                        for (int j = 0; j < nkb; ++j) {
#pragma unroll
                            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                                const uint32_t acc = (st > 0 || j > 0 || kk > 0) ? 1u : 0u;
                                umma_bf16(d_tmem, smem_desc_kmajor_sw128(w_addr + j * 128 * 128 + kk * 32),
                                          smem_desc_kmajor_sw128(a_addr + j * C::kActSlot + kk * 32), C::kIdesc, acc);
                            }
                        }
                    }
                    umma_commit(smem_u32(&bar_empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok)
                    umma_commit(smem_u32(&bar_tfull[buf]));
            }
            umma_commit(smem_u32(&bar_drain));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&bar_drain), 0) && global_timer_ns() - t0 < A1.wait_limit_ns) {
            }
        }
        __syncwarp();
    } else if (kFp8 && warp >= 8) {
        // ------------------------------------------------------------ converters (MXFP8 weights)
        // warp 8 + 8p + 4h + q expands rows 32q..32q+31 of weight tile h of
        // each stage (gate / up, or the stage's first / second K block), K
        // part p of 128 / parts codes, into TMEM lanes 32q.. of the slot:
        // lane i owns row 32q + i; each TMEM store takes 64 codes as 32
        // columns of bf16 pairs.
        constexpr int kParts = C::kConvWarps >= 8 ? C::kConvWarps / 8 : 1;   // 1 in the bf16 instances (no converters)
        const int quarter = warp & 3;
        const int half = ((warp - 8) >> 2) & 1;
        const int kpart = (warp - 8) >> 3;
        const int row = quarter * 32 + lane;
        int stage = 0;
        uint32_t phase = 0;
        int slot = 0;
        uint32_t slot_phase = 0;
        bool ok = true;
        UnitRing ring(s_unit, bar_ufull, bar_uempty);
        while (ok) {
            int u = total_units;
            if (!ring.take_warp(u, lane, abort_flag, A1.wait_limit_ns) || u >= total_units)
                break;
            const bool up = u < units1;
            const int steps = up ? kb1 : (kb2 + 1) / 2;
            for (int st = 0; st < steps; ++st) {
                const bool good = mbar_wait_bounded(smem_u32(&bar_full[stage]), phase, abort_flag, A1.wait_limit_ns) &&
                                  mbar_wait_bounded(smem_u32(&bar_conv_empty[slot]), slot_phase ^ 1u, abort_flag,
                                                    A1.wait_limit_ns);
                if (!__all_sync(kFull, good)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nkb = up ? 2 : ((2 * st + 1 < kb2) ? 2 : 1);
                if (half < nkb) {
                    const uint8_t *tile = smem + stage * C::kStageBytes + half * 128 * 128 + row * 128;
                    const uint32_t codes4 =
                        *reinterpret_cast<const uint32_t *>(smem + stage * C::kStageBytes + C::kScaleOffset +
                                                             half * 512 + row * 4);
                    const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                            2 * C::kAccCols + slot * C::kASlotCols + half * 64;
#pragma unroll
                    for (int q4 = 0; q4 < 2 / kParts; ++q4) {
                        const int c0 = 4 * (kpart + q4);
                        uint32_t out[32];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            // 16 codes of K [16c, 16c + 16), at the 128-byte swizzled position of chunk c
                            const int c = c0 + i;
                            const uint4 raw = *reinterpret_cast<const uint4 *>(tile + ((c ^ (row & 7)) << 4));
                            const int o = i * 8;
                            // E8M0 code sc: 2^(sc - 127). One bf16 multiply by 2^(sc - 7) when that is
                            // a normal bf16 (sc <= 134), else by 2^127 and then by 2^(sc - 134)
                            const uint32_t sc = (codes4 >> (8 * (c >> 1))) & 0xffu;
                            const bool big = sc > 134u;
                            const uint32_t s1 = ((big ? 254u : sc + 120u) << 7) * 0x00010001u;
                            e4m3x4_to_bf16x4(raw.x, s1, out[o + 0], out[o + 1]);
                            e4m3x4_to_bf16x4(raw.y, s1, out[o + 2], out[o + 3]);
                            e4m3x4_to_bf16x4(raw.z, s1, out[o + 4], out[o + 5]);
                            e4m3x4_to_bf16x4(raw.w, s1, out[o + 6], out[o + 7]);
                            if (big) {
                                const uint32_t s2 = ((sc - 7u) << 7) * 0x00010001u;
#pragma unroll
                                for (int z = 0; z < 8; ++z)
                                    asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(out[o + z]) : "r"(s2));
                            }
                        }
                        tmem_st_32x32b_x32(t_addr + c0 * 8, out);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_conv_full[slot]));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++slot == kASlotsRing) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;
        UnitRing ring(s_unit, bar_ufull, bar_uempty);
        for (int local = 0;; ++local) {
            int u = total_units;
            if (!ring.take_warp(u, lane, abort_flag, A1.wait_limit_ns) || u >= total_units)
                break;
            const bool up = u < units1;
            const int v = up ? u : u - units1;
            const Unit t = up ? decode_unit<true, kTileRows, 128>(v, s_off, s_tp, E, NT1)
                              : decode_unit<true, kTileRows, 128>(v / kSplitDown, s_off, s_tp, E, NT2);
            const int buf = local & 1;
            const uint32_t use = (local >> 1) & 1;
            int ok = 0;
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&bar_tfull[buf]), use, abort_flag, A1.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + buf * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
            const int col = t.n0 + q * 32 + lane;
            // a down unit's K part goes to its own buffer (summed in part order by the combine)
            float *const y_out = static_cast<float *>(A2.out) +
                                 (!up ? static_cast<size_t>(v % kSplitDown) * A2.cap * A2.n_out : 0);
#pragma unroll 1
            for (int c = 0; c < kTileRows; c += 16) {
                uint32_t g[16], w[16];
                tmem_ld_32x32b_x16(t_row + c, g);
                if (up)
                    tmem_ld_32x32b_x16(t_row + kTileRows + c, w);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int rr = c + i;
                    const int row = t.row0 + rr;
                    if (rr < t.rows && row >= 0 && row < A1.cap && col < (up ? A1.n_out : A2.n_out)) {
                        if (up) {
                            static_cast<__nv_bfloat16 *>(A1.out)[static_cast<size_t>(row) * A1.n_out + col] =
                                __float2bfloat16_rn(silu_mul(__uint_as_float(g[i]), __uint_as_float(w[i])));
                        } else {
                            y_out[static_cast<size_t>(row) * A2.n_out + col] = __uint_as_float(g[i]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_tempty[buf]));
            if (up) {
                // publish this warp's h rows: every storing lane fences, then
                // one lane releases the expert's count (4 warps per unit; no
                // cross-warp wait)
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    red_release_gpu_add(fa.ready + t.e, 1);
            }
        }
        // whole-forward form: this thread's y stores before the CTA's one count
        // on `done` (after the CTA barrier below)
        if (kMega)
            __threadfence();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    if (kMega && !fa.combine_apart) {
        // every CTA counts itself once on `done`, after all its units (its
        // epilogue threads fenced their y stores before the barrier above;
        // also after giving up, so that the others need not wait the limit);
        // the combine starts once every CTA has counted itself
        if (threadIdx.x == 0)
            red_release_gpu_add(fa.done, 1);
        const int need = static_cast<int>(gridDim.x);
        if (threadIdx.x == 0 && !s_abort) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(fa.done) < need) {
                if (global_timer_ns() - t0 > A1.wait_limit_ns) {
                    s_abort = 1;
                    break;
                }
            }
        }
        __syncthreads();
        if (!s_abort)
            cta_combine<kSplitDown, kThreads>(fa, s_inv, s_T);
        __syncthreads();
    }
    // tail clean-up: the last CTA out (every other CTA has passed all its
    // waits on the counters) returns them to zero for the next launch
    if (threadIdx.x == 0)
        s_last = atom_add_acq_rel_gpu(fa.exits, 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (s_last) {
        for (int e = threadIdx.x; e < E; e += kThreads)
            fa.ready[e] = 0;
        if (threadIdx.x == 0) {
            if (kMega)
                *fa.done = 0;
            *fa.next_unit = 0;
            *fa.exits = 0;
        }
    }
    if (kMega && fa.combine_apart)
        pdl_wait();   // the dispatch kernel beside is complete before any dependent starts
    pdl_trigger();
    if (threadIdx.x == 0 && s_abort)
        atomicOr(A1.err, MOE_DEVERR_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ CTA-pair tiled kernel
//
// Same work decomposition as the tiled path, on a 2-CTA cluster sharing one
// tcgen05.mma.cta_group::2 of M=256, N=256: a unit is 256 activation rows of
// one expert x 256 weight rows; each CTA of the pair loads its own 128
// activation rows and half of the weight tile (gate-up: CTA 0 the 128 gate
// rows, CTA 1 the 128 matching up rows; down: 128 output columns each), so a
// stage is 32 KB per CTA instead of 48 KB and the ring is 6 deep. CTA 0 issues
// the MMAs; each CTA's TMEM receives its 128 rows x 256 columns, so the
// epilogue is the single-CTA one. Every TMA load of both CTAs completes on
// CTA 0's full barrier (2 arrivals + both CTAs' bytes); CTA 0's commits are
// multicast to both CTAs' empty / TMEM-full barriers; both epilogues release
// the accumulator on CTA 0's TMEM-empty barrier.
//
// Swapped last tiles. The last row tile of an expert holds count % 256 rows;
// on a 256-row tile those past the count are padding the tensor cores still
// multiply (11% of the MMAs of the large-batch shape, where a quarter of the
// experts hold just over 512 rows). A last tile of at most 128 rows runs
// swapped instead: the weights go on the MMA's M side (128 weight rows per
// CTA) and the tile's rows on N, rounded up to 64 (N/2 per CTA, loaded with a
// 32-row box), so the MMAs and the activation loads shrink with the rows.
// Each CTA's TMEM then holds its 128 weight rows x N rows; the epilogue
// stores it transposed (lane = output column). Down: the CTA's 128 W2 rows
// are its 128 output columns. Gate-up: the CTA's 128 weight rows are 64 gate
// rows and the matching 64 up rows (two 64-row boxes), so SiLU(gate)*up pairs
// TMEM lane i with lane i + 64: epilogue warps 6 and 7 hand their up values to
// warps 4 and 5 through shared memory, 16 rows at a time, on a pair of
// mbarriers (bounded waits). Row-major weights only (the PACKED images are
// whole 128-row tiles).
template <bool kGated, int kStages>
struct PairCfg {
    static constexpr int kHalfBytes = 128 * 128;                 // 128 rows x 64 bf16
    static constexpr int kStageBytes = 2 * kHalfBytes;           // A half + B half
    static constexpr int kPairRows = 256;
    static constexpr int kOutCols = kGated ? 128 : 256;
    static constexpr int kAccCols = 256;
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kIdesc = idesc_bf16_f32(256, 256);
    static constexpr int kSwapRows = 128;     // last tiles with at most this many rows run swapped
    static constexpr int kSwapBox = 32;       // activation rows of one TMA box of a swapped unit
    static constexpr int kXchStride = 17;     // gate-up exchange: floats per lane (16 rows + 1 against bank conflicts)
    // down: fp32 transpose scratch; gate-up: the up values of two warps, 32 lanes x 16 rows each
    static constexpr int kEpiScratch = kGated ? 2 * 32 * kXchStride * 4 : 4 * 32 * 36 * 4;
    static constexpr int kDynSmem = 1024 + kStages * kStageBytes + kEpiScratch;
};

// Rows on the MMA's N side of a swapped unit (a multiple of 64: each CTA
// loads whole 32-row boxes), or 0 for a unit that runs as usual.
template <int kSwapRows>
__device__ __forceinline__ int swap_tokens(const Unit &t, bool swap_ok)
{
    return (swap_ok && t.rows <= kSwapRows) ? ((t.rows + 63) & ~63) : 0;
}

template <bool kGated, int kStages>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                             const __grid_constant__ CUtensorMap tm_act_swap,
                             const __grid_constant__ CUtensorMap tm_w_swap, const GemmArgs args)
{
    using C = PairCfg<kGated, kStages>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];   // used in CTA 0
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];       // used in CTA 0
    __shared__ __align__(8) uint64_t bar_drain;           // used in CTA 0
    __shared__ __align__(8) uint64_t bar_xfull[2];        // gate-up, swapped units: up values handed over
    __shared__ __align__(8) uint64_t bar_xempty[2];       // ... and taken
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_tp[kMaxExperts + 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = args.E;
    const uint32_t rank = cluster_ctarank();
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 2);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 8);   // 4 epilogue warps x 2 CTAs
            mbar_init(smem_u32(&bar_xfull[b]), 1);
            mbar_init(smem_u32(&bar_xempty[b]), 1);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_act);
        tma_prefetch_desc(&tm_w);
        if (!args.w_packed) {
            tma_prefetch_desc(&tm_act_swap);
            tma_prefetch_desc(&tm_w_swap);
        }
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(&s_tmem_base), C::kTmemCols);
        tmem_relinquish_pair();
    }
    for (int i = threadIdx.x; i <= E; i += kThreads)
        s_off[i] = args.expert_offsets[i];
    __syncthreads();
    if (warp == 3)
        build_tile_prefix(s_off, s_tp, E, C::kPairRows, lane);
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers initialised before any remote arrive
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    const int NT = (args.n_out + C::kOutCols - 1) / C::kOutCols;
    const int cluster_id = blockIdx.x >> 1;
    const int n_clusters = gridDim.x >> 1;
    const int total_units = s_tp[E] * NT;
    const int k_blocks = args.K / kBK;
    const bool swap_ok = !args.w_packed;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        const uint64_t pol_w = l2_policy_evict_normal();
        const uint64_t pol_a = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = cluster_id; ok && u < total_units; u += n_clusters) {
            const Unit t = decode_unit<false, C::kPairRows, C::kOutCols, kGated>(u, s_off, s_tp, E, NT);
            const int n_swap = swap_tokens<C::kSwapRows>(t, swap_ok);
            const int a_row = t.row0 + 128 * static_cast<int>(rank);
            const int w_row = kGated ? t.e * args.w_rows_per_expert + (rank ? args.up_row_offset : 0) + t.n0
                                     : t.e * args.w_rows_per_expert + t.n0 + 128 * static_cast<int>(rank);
            // swapped: this CTA's 128 weight rows (gate-up: 64 gate + the 64 matching up rows) in the A half,
            // its n_swap / 2 activation rows in the B half
            const int half = n_swap >> 1;
            const int sw_row = kGated ? t.e * args.w_rows_per_expert + t.n0 + 64 * static_cast<int>(rank)
                                      : w_row;
            const int sa_row = t.row0 + half * static_cast<int>(rank);
            if (lane == 0) {
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, abort_flag, args.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full0 = map_to_cta(smem_u32(&bar_full[stage]), 0);
                    const uint32_t a_dst = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t b_dst = a_dst + C::kHalfBytes;
                    const int kc = kb * kBK;
                    if (n_swap == 0) {
                        mbar_arrive_expect_tx_cluster(full0, C::kStageBytes);
                        tma_load_2d_pair(a_dst, &tm_act, full0, kc, a_row, pol_a);
                        const int2 wc = weight_coords(args, kGated, w_row, kb);
                        tma_load_2d_pair(b_dst, &tm_w, full0, wc.x, wc.y, pol_w);
                    } else {
                        mbar_arrive_expect_tx_cluster(full0, C::kHalfBytes + half * 128);
                        if (kGated) {
                            tma_load_2d_pair(a_dst, &tm_w_swap, full0, kc, sw_row, pol_w);
                            tma_load_2d_pair(a_dst + 64 * 128, &tm_w_swap, full0, kc, sw_row + args.up_row_offset,
                                             pol_w);
                        } else {
                            tma_load_2d_pair(a_dst, &tm_w, full0, kc, sw_row, pol_w);
                        }
                        for (int j = 0; j < half; j += C::kSwapBox)
                            tma_load_2d_pair(b_dst + j * 128, &tm_act_swap, full0, kc, sa_row + j, pol_a);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (CTA 0 only)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int u = cluster_id; ok && u < total_units; u += n_clusters, ++local) {
                const int buf = local & 1;
                const uint32_t use = (local >> 1) & 1;
                const int n_swap =
                    swap_tokens<C::kSwapRows>(decode_unit<false, C::kPairRows, C::kOutCols, kGated>(u, s_off, s_tp, E, NT),
                                              swap_ok);
                const uint32_t idesc = n_swap ? idesc_bf16_f32(256, n_swap) : C::kIdesc;
                if (!mbar_wait_bounded(smem_u32(&bar_tempty[buf]), use ^ 1u, abort_flag, args.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * C::kAccCols;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&bar_full[stage]), phase, abort_flag, args.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t b_addr = a_addr + C::kHalfBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        umma_bf16_pair(d_tmem, smem_desc_kmajor_sw128(a_addr + kk * 32),
                                       smem_desc_kmajor_sw128(b_addr + kk * 32), idesc, acc);
                    }
                    umma_commit_pair(smem_u32(&bar_empty[stage]), 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok)
                    umma_commit_pair(smem_u32(&bar_tfull[buf]), 0x3);
            }
            umma_commit_pair(smem_u32(&bar_drain), 0x1);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&bar_drain), 0) && global_timer_ns() - t0 < args.wait_limit_ns) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp - 4;
        float *const scratch = reinterpret_cast<float *>(smem + kStages * C::kStageBytes);
        uint32_t xk = 0;   // gate-up exchanges of this warp so far (their mbarrier phases)
        int local = 0;
        for (int u = cluster_id; u < total_units; u += n_clusters, ++local) {
            const Unit t = decode_unit<false, C::kPairRows, C::kOutCols, kGated>(u, s_off, s_tp, E, NT);
            const int n_swap = swap_tokens<C::kSwapRows>(t, swap_ok);
            const int buf = local & 1;
            const uint32_t use = (local >> 1) & 1;
            int ok = 0;
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&bar_tfull[buf]), use, abort_flag, args.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok)
                break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + buf * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
            if (n_swap == 0) {
                const int r = 128 * static_cast<int>(rank) + q * 32 + lane;   // row within the 256-row pair tile
                const int row = t.row0 + r;
                tiled_epilogue<kGated>(t_row, args, row, r < t.rows && row >= 0 && row < args.cap, t.n0,
                                       scratch + q * 32 * 36);
            } else if (!kGated) {
                // lane = W2 row = output column; TMEM columns = the unit's rows
                const int col = t.n0 + 128 * static_cast<int>(rank) + q * 32 + lane;
                const bool col_ok = col < args.n_out;
                bool clipped = false;
#pragma unroll 1
                for (int c = 0; c < n_swap && c < t.rows; c += 16) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(t_row + c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (!col_ok || c + i >= t.rows)
                            continue;
                        const size_t o = static_cast<size_t>(t.row0 + c + i) * args.n_out + col;
                        const float y = __uint_as_float(v[i]);
                        if (args.out_f16) {
                            // the rounding of the unswapped epilogue: to nearest, saturating at +-65504
                            clipped |= fabsf(y) > 65504.f;
                            uint32_t h2;
                            asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h2) : "f"(0.f), "f"(y));
                            static_cast<uint16_t *>(args.out)[o] = static_cast<uint16_t>(h2 & 0xffffu);
                        } else {
                            static_cast<float *>(args.out)[o] = y;
                        }
                    }
                }
                if (__any_sync(kFull, clipped) && lane == 0)
                    atomicOr(args.err, MOE_DEVERR_Y_RANGE);
            } else {
                // lanes 0..63: gate rows, lanes 64..127: the matching up rows, of this CTA's 64 output
                // columns; warp q + 2 hands its up values to warp q, 16 rows at a time
                const int pair = q & 1;
                float *const xch = scratch + pair * 32 * C::kXchStride;
                const uint32_t xfull = smem_u32(&bar_xfull[pair]);
                const uint32_t xempty = smem_u32(&bar_xempty[pair]);
                const int col = t.n0 + 64 * static_cast<int>(rank) + pair * 32 + lane;
                const bool col_ok = col < args.n_out;
                bool good = true;
#pragma unroll 1
                for (int c = 0; c < n_swap && c < t.rows; c += 16, ++xk) {
                    uint32_t v[16];
                    tmem_ld_32x32b_x16(t_row + c, v);
                    tmem_wait_ld();
                    int w_ok = 0;
                    if (lane == 0)
                        w_ok = mbar_wait_bounded(q >= 2 ? xempty : xfull, q >= 2 ? ((xk & 1u) ^ 1u) : (xk & 1u),
                                                 abort_flag, args.wait_limit_ns)
                                   ? 1
                                   : 0;
                    if (!__shfl_sync(kFull, w_ok, 0)) {
                        good = false;
                        break;
                    }
                    if (q >= 2) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            xch[lane * C::kXchStride + i] = __uint_as_float(v[i]);
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(xfull);
                    } else {
                        float up[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            up[i] = xch[lane * C::kXchStride + i];
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(xempty);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (col_ok && c + i < t.rows)
                                static_cast<__nv_bfloat16 *>(args.out)[static_cast<size_t>(t.row0 + c + i) *
                                                                           args.n_out + col] =
                                    __float2bfloat16_rn(silu_mul(__uint_as_float(v[i]), up[i]));
                    }
                }
                if (!good)
                    break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(map_to_cta(smem_u32(&bar_tempty[buf]), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (s_abort) {
        // give-up path: let loads and remote arrivals still in flight land first
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    cluster_sync();   // neither CTA leaves while its peer may still touch its shared memory
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
    if (threadIdx.x == 0 && s_abort)
        atomicOr(args.err, MOE_DEVERR_WAIT_TIMEOUT);
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box of 64 columns x box_rows rows, 128-byte swizzle
// (none for data that is already stored as swizzled shared-memory images).
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool swizzle = true)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Weight tensor map: row-major [E * rows_per_expert, K] with swizzle, or the
// packed buffer as [bytes / 128, 64] lines of pre-swizzled images, no swizzle.
bool make_weight_map(CUtensorMap *m, const GemmProblem &p)
{
    const uint64_t rows = static_cast<uint64_t>(p.E) * p.w_rows_per_expert;
    if (!p.w_packed)
        return make_map(m, p.w, rows, static_cast<uint64_t>(p.K), 128);
    return make_map(m, p.w, rows * static_cast<uint64_t>(p.K) / 64, 64, 128, false);
}

template <bool kSmallM, bool kGated, int kTileRows, int kStages, int kSplitK = 1, bool kGather = false>
cudaError_t run(const GemmProblem &p, int num_sms, cudaStream_t stream)
{
    using C = Cfg<kSmallM, kGated, kTileRows, kStages, kSplitK>;
    auto kern = grouped_gemm_kernel<kSmallM, kGated, kTileRows, kStages, kSplitK, kGather>;
    static thread_local int attr_done_for_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (attr_done_for_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
        if (e != cudaSuccess)
            return e;
        attr_done_for_device = dev;
    }
    CUtensorMap tm_act, tm_w;
    if (!make_map(&tm_act, p.act, static_cast<uint64_t>(p.act_rows), static_cast<uint64_t>(p.K), kGather ? 1 : kTileRows) ||
        !make_weight_map(&tm_w, p))
        return cudaErrorInvalidValue;
    GemmArgs a;
    a.expert_offsets = p.expert_offsets;
    a.perm = p.perm;
    a.k = p.k;
    a.out = p.out;
    a.err = p.err;
    a.wait_limit_ns = kWaitLimitNs;
    a.E = p.E;
    a.cap = p.cap;
    a.K = p.K;
    a.n_out = p.n_out;
    a.w_rows_per_expert = p.w_rows_per_expert;
    a.up_row_offset = p.up_row_offset;
    a.w_packed = p.w_packed ? 1 : 0;
    a.out_f16 = p.out_f16 ? 1 : 0;
    a.sched = p.sched;
    // Upper bound of the units any routing can produce; no more CTAs than that.
    const long long max_row_tiles = (static_cast<long long>(p.cap) + kTileRows - 1) / kTileRows + p.E;
    const long long max_units = max_row_tiles * ((p.n_out + C::kOutCols - 1) / C::kOutCols) * kSplitK;
    const int grid = static_cast<int>(max_units < num_sms ? (max_units < 1 ? 1 : max_units) : num_sms);
    return launch_k(kern, dim3(grid), dim3(kThreads), C::kDynSmem, stream, p.pdl, tm_act, tm_w, a);
}


template <bool kGated, int kStages>
cudaError_t run_pair(const GemmProblem &p, int num_sms, cudaStream_t stream)
{
    using C = PairCfg<kGated, kStages>;
    auto kern = grouped_gemm_pair_kernel<kGated, kStages>;
    static thread_local int attr_done_for_device = -1;
    static thread_local int max_clusters = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kDynSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (attr_done_for_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
        if (e != cudaSuccess)
            return e;
        cfg.gridDim = dim3(2 * (num_sms / 2));
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess)
            return e;
        max_clusters = n > 0 ? n : 1;
        attr_done_for_device = dev;
    }
    CUtensorMap tm_act, tm_w, tm_act_swap, tm_w_swap;
    if (!make_map(&tm_act, p.act, static_cast<uint64_t>(p.act_rows), static_cast<uint64_t>(p.K), 128) ||
        !make_weight_map(&tm_w, p))
        return cudaErrorInvalidValue;
    // swapped last tiles (row-major weights): activation rows in 32-row boxes;
    // gate-up weights in 64-row boxes (64 gate + 64 up rows per CTA)
    tm_act_swap = tm_act;
    tm_w_swap = tm_w;
    if (!p.w_packed &&
        (!make_map(&tm_act_swap, p.act, static_cast<uint64_t>(p.act_rows), static_cast<uint64_t>(p.K),
                   C::kSwapBox) ||
         (kGated && !make_map(&tm_w_swap, p.w, static_cast<uint64_t>(p.E) * p.w_rows_per_expert,
                              static_cast<uint64_t>(p.K), 64))))
        return cudaErrorInvalidValue;
    GemmArgs a;
    a.expert_offsets = p.expert_offsets;
    a.perm = p.perm;
    a.k = p.k;
    a.out = p.out;
    a.err = p.err;
    a.wait_limit_ns = kWaitLimitNs;
    a.E = p.E;
    a.cap = p.cap;
    a.K = p.K;
    a.n_out = p.n_out;
    a.w_rows_per_expert = p.w_rows_per_expert;
    a.up_row_offset = p.up_row_offset;
    a.w_packed = p.w_packed ? 1 : 0;
    a.out_f16 = p.out_f16 ? 1 : 0;
    a.sched = nullptr;
    const long long max_units =
        ((static_cast<long long>(p.cap) + 255) / 256 + p.E) * ((p.n_out + C::kOutCols - 1) / C::kOutCols);
    long long clusters = max_units < max_clusters ? max_units : max_clusters;
    if (clusters < 1)
        clusters = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    return cudaLaunchKernelEx(&cfg, kern, tm_act, tm_w, tm_act_swap, tm_w_swap, a);
}


GemmArgs make_args(const GemmProblem &p)
{
    GemmArgs a;
    a.expert_offsets = p.expert_offsets;
    a.perm = p.perm;
    a.k = p.k;
    a.out = p.out;
    a.err = p.err;
    a.wait_limit_ns = kWaitLimitNs;
    a.E = p.E;
    a.cap = p.cap;
    a.K = p.K;
    a.n_out = p.n_out;
    a.w_rows_per_expert = p.w_rows_per_expert;
    a.up_row_offset = p.up_row_offset;
    a.w_packed = p.w_packed ? 1 : 0;
    a.out_f16 = 0;
    a.sched = nullptr;
    return a;
}

// Shared memory the whole-forward form needs for its expert tables:
// offsets and tile prefix [E + 1] each, perm and inv [T_max * k] each.
long long mega_table_bytes(int E, long long slots) { return 4LL * (2LL * (E + 1) + 2LL * slots); }

// Per-block shared memory the device grants (opt-in) minus the static shared
// memory of the whole-forward kernel and its stages: what is left for the
// tables. Cached per host thread and device; -1 if a query fails.
template <int kTileRows, int kStages, bool kFp8>
long long mega_table_budget()
{
    static thread_local int cached_dev = -1;
    static thread_local long long cached = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    if (dev != cached_dev) {
        int optin = 0;
        cudaFuncAttributes fa1 = {}, fa2 = {}, fa4 = {};
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa1, fused_small_kernel<kTileRows, kStages, 1, true, kFp8>) != cudaSuccess ||
            cudaFuncGetAttributes(&fa2, fused_small_kernel<kTileRows, kStages, 2, true, kFp8>) != cudaSuccess ||
            cudaFuncGetAttributes(&fa4, fused_small_kernel<kTileRows, kStages, 4, true, kFp8>) != cudaSuccess)
            return -1;
        size_t st = fa1.sharedSizeBytes > fa2.sharedSizeBytes ? fa1.sharedSizeBytes : fa2.sharedSizeBytes;
        st = st > fa4.sharedSizeBytes ? st : fa4.sharedSizeBytes;
        cached = static_cast<long long>(optin) - static_cast<long long>(st) -
                 FusedCfg<kTileRows, kStages, kFp8>::kDynSmem;
        cached_dev = dev;
    }
    return cached;
}

// E4M3 codes [rows, K] as a 2-D byte tensor: 128-byte x 128-row boxes, 128-byte swizzle.
bool make_map_codes(CUtensorMap *m, const void *base, uint64_t rows, uint64_t K)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kTileRows, int kStages, int kSplitDown, bool kMega, bool kFp8>
cudaError_t run_fused(const GemmProblem &up, const GemmProblem &down, int32_t *ready, int32_t *counters,
                      int num_sms, cudaStream_t stream, const MegaParams *mega)
{
    using C = FusedCfg<kTileRows, kStages, kFp8>;
    auto kern = fused_small_kernel<kTileRows, kStages, kSplitDown, kMega, kFp8>;
    const long long slots = mega ? static_cast<long long>(mega->T_max) * up.k : 0;
    const long long tables = kMega ? mega_table_bytes(up.E, slots) : 0;
    long long budget = 0;
    if constexpr (kMega) {
        budget = mega_table_budget<kTileRows, kStages, kFp8>();
        if (tables > budget)
            return cudaErrorInvalidValue;
    }
    const int dyn_smem = C::kDynSmem + static_cast<int>(tables);
    static thread_local int attr_done_for_device = -1;
    static thread_local int attr_bytes = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (attr_done_for_device != dev || attr_bytes < dyn_smem) {
        const int want = C::kDynSmem + static_cast<int>(budget);
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
        if (e != cudaSuccess)
            return e;
        attr_done_for_device = dev;
        attr_bytes = want;
    }
    CUtensorMap tm_x, tm_w13, tm_h, tm_w2;
    const uint64_t rows13 = static_cast<uint64_t>(up.E) * up.w_rows_per_expert;
    const uint64_t rows2 = static_cast<uint64_t>(down.E) * down.w_rows_per_expert;
    const bool maps = kFp8 ? make_map_codes(&tm_w13, up.w, rows13, static_cast<uint64_t>(up.K)) &&
                                 make_map_codes(&tm_w2, down.w, rows2, static_cast<uint64_t>(down.K))
                           : make_weight_map(&tm_w13, up) && make_weight_map(&tm_w2, down);
    // gathered rows: a one-row box for tile::gather4; sorted rows (MXFP8,
    // separate form): a box of the tile's rows
    const uint32_t x_box = up.gather ? 1u : static_cast<uint32_t>(kTileRows);
    if (!maps || !make_map(&tm_x, up.act, static_cast<uint64_t>(up.act_rows), static_cast<uint64_t>(up.K), x_box) ||
        !make_map(&tm_h, down.act, static_cast<uint64_t>(down.cap), static_cast<uint64_t>(down.K), kTileRows))
        return cudaErrorInvalidValue;
    FusedArgs fa = {};
    fa.act_sorted = up.gather ? 0 : 1;
    fa.up = make_args(up);
    fa.down = make_args(down);
    fa.ready = ready;
    if (kFp8) {   // scale blocks follow the codes
        fa.sc13 = static_cast<const uint8_t *>(up.w) + rows13 * static_cast<uint64_t>(up.K);
        fa.sc2 = static_cast<const uint8_t *>(down.w) + rows2 * static_cast<uint64_t>(down.K);
    }
    fa.exits = counters + 1;
    fa.next_unit = counters + 2;
    if (kMega) {
        fa.ids = mega->ids;
        fa.topk_w = mega->topk_w;
        fa.d_num_tokens = mega->d_num_tokens;
        fa.T_max = mega->T_max;
        fa.slots_max = static_cast<int>(slots);
        fa.expert_offsets_out = mega->expert_offsets_out;
        fa.perm_out = mega->perm_out;
        fa.out = static_cast<__nv_bfloat16 *>(mega->out);
        fa.done = counters;
        fa.combine_apart = mega->combine_apart ? 1 : 0;
    }
    // one CTA per SM, all resident at once (the down units and the combine
    // wait on counts other CTAs publish): a cooperative launch, sized against
    // the device's occupancy for this kernel
    const long long tiles = (static_cast<long long>(up.cap) + kTileRows - 1) / kTileRows + up.E;
    const long long max_units = tiles * ((up.n_out + 127) / 128 + ((down.n_out + 127) / 128) * kSplitDown);
    const bool whole_forward = kMega && !(mega && mega->combine_apart);
    const int grid_sms = fused_grid_sms(whole_forward, kFp8, up.cap, up.E, up.n_out, kTileRows, num_sms);
    const long long want = max_units < grid_sms ? (max_units < 1 ? 1 : max_units) : grid_sms;
    return launch_k_coresident(kern, want, dim3(C::kThreadsCta), dyn_smem, stream, up.pdl, num_sms, tm_x, tm_w13,
                               tm_h, tm_w2, fa);
}

}  // namespace

cudaError_t launch_grouped_gemm(const GemmProblem &p, int num_sms, cudaStream_t stream)
{
    if (p.w_mxfp8)   // MXFP8 weights run through the fused M-small kernel only
        return cudaErrorInvalidValue;
    if (p.out_f16 && (p.small_m || p.gated))   // fp16 y: tiled down GEMM only
        return cudaErrorInvalidValue;
    if (p.split_k != 1 && ((p.split_k != 2 && p.split_k != 4) || !p.small_m || p.gated || p.tile_rows != 16 ||
                           (p.K / kBK) % p.split_k != 0))
        return cudaErrorInvalidValue;
    if (p.gather && (!p.gated || !p.perm || p.k < 1))
        return cudaErrorInvalidValue;
    if (!p.small_m) {
        if (p.tile_rows != 128)
            return cudaErrorInvalidValue;
        if (p.gather)   // tiled tiles would need 32 gather4 per stage: not built (see moe_forward)
            return cudaErrorInvalidValue;
        if (p.cta_pair)
            return p.gated ? run_pair<true, 6>(p, num_sms, stream) : run_pair<false, 6>(p, num_sms, stream);
        return p.gated ? run<false, true, 128, 4>(p, num_sms, stream) : run<false, false, 128, 4>(p, num_sms, stream);
    }
    switch (p.tile_rows) {
    case 16:
        if (!p.gated && p.split_k == 2)
            return run<true, false, 16, 10, 2>(p, num_sms, stream);
        if (!p.gated && p.split_k == 4)
            return run<true, false, 16, 10, 4>(p, num_sms, stream);
        if (p.gated)
            return p.gather ? run<true, true, 16, 6, 1, true>(p, num_sms, stream) : run<true, true, 16, 6>(p, num_sms, stream);
        return run<true, false, 16, 10>(p, num_sms, stream);
    case 32:
        if (p.gated)
            return p.gather ? run<true, true, 32, 5, 1, true>(p, num_sms, stream) : run<true, true, 32, 5>(p, num_sms, stream);
        return run<true, false, 32, 9>(p, num_sms, stream);
    case 64:
        if (p.gated)
            return p.gather ? run<true, true, 64, 5, 1, true>(p, num_sms, stream) : run<true, true, 64, 5>(p, num_sms, stream);
        return run<true, false, 64, 8>(p, num_sms, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fused_small(const GemmProblem &up, const GemmProblem &down, int32_t *ready, int32_t *counters,
                               int num_sms, cudaStream_t stream, const MegaParams *mega)
{
    // rows gathered from x through perm, or (MXFP8 weights, separate form) a sorted copy
    if (!up.small_m || !down.small_m || !up.gated || down.gated || up.tile_rows != down.tile_rows || !ready ||
        !counters || (down.split_k != 1 && down.split_k != 2 && down.split_k != 4) ||
        (!up.gather && (mega || !up.w_mxfp8)))
        return cudaErrorInvalidValue;
    if (mega ? (!mega->ids || !mega->topk_w || !mega->expert_offsets_out || !mega->perm_out || !mega->out ||
                mega->T_max < 1)
             : (up.gather && !up.perm))
        return cudaErrorInvalidValue;
    if (up.w_mxfp8 != down.w_mxfp8)
        return cudaErrorInvalidValue;
    if (up.w_mxfp8) {
        // MXFP8 weights: every M-small tile height (this kernel is their only GEMM)
        if (up.K % 128 != 0 || down.K % 128 != 0 || (down.K / 128) % down.split_k != 0)
            return cudaErrorInvalidValue;
        if (mega && (up.tile_rows != 16))
            return cudaErrorInvalidValue;
        switch (up.tile_rows) {
        case 16:
            if (mega)
                return down.split_k == 4   ? run_fused<16, 5, 4, true, true>(up, down, ready, counters, num_sms, stream, mega)
                       : down.split_k == 2 ? run_fused<16, 5, 2, true, true>(up, down, ready, counters, num_sms, stream, mega)
                                           : run_fused<16, 5, 1, true, true>(up, down, ready, counters, num_sms, stream, mega);
            return down.split_k == 4   ? run_fused<16, 5, 4, false, true>(up, down, ready, counters, num_sms, stream, nullptr)
                   : down.split_k == 2 ? run_fused<16, 5, 2, false, true>(up, down, ready, counters, num_sms, stream, nullptr)
                                       : run_fused<16, 5, 1, false, true>(up, down, ready, counters, num_sms, stream, nullptr);
        case 32:
            return down.split_k == 1
                       ? run_fused<32, 4, 1, false, true>(up, down, ready, counters, num_sms, stream, nullptr)
                       : cudaErrorInvalidValue;
        case 64:
            return down.split_k == 1
                       ? run_fused<64, 3, 1, false, true>(up, down, ready, counters, num_sms, stream, nullptr)
                       : cudaErrorInvalidValue;
        default:
            return cudaErrorInvalidValue;
        }
    }
    // bf16 weights: built for decode-size batches only (16-row token tiles):
    // with 32-row tiles (the Zipf small batch) two launches measured 2% faster
    if (up.tile_rows != 16)
        return cudaErrorInvalidValue;
    if ((down.K / kBK) % down.split_k != 0)
        return cudaErrorInvalidValue;
    if (mega)
        return down.split_k == 4   ? run_fused<16, 6, 4, true, false>(up, down, ready, counters, num_sms, stream, mega)
               : down.split_k == 2 ? run_fused<16, 6, 2, true, false>(up, down, ready, counters, num_sms, stream, mega)
                                   : run_fused<16, 6, 1, true, false>(up, down, ready, counters, num_sms, stream, mega);
    return down.split_k == 4   ? run_fused<16, 6, 4, false, false>(up, down, ready, counters, num_sms, stream, nullptr)
           : down.split_k == 2 ? run_fused<16, 6, 2, false, false>(up, down, ready, counters, num_sms, stream, nullptr)
                               : run_fused<16, 6, 1, false, false>(up, down, ready, counters, num_sms, stream, nullptr);
}

bool fused_mega_fits(int E, long long slots, bool mxfp8)
{
    const long long budget = mxfp8 ? mega_table_budget<16, 5, true>() : mega_table_budget<16, 6, false>();
    return budget >= 0 && mega_table_bytes(E, slots) <= budget;
}

}  // namespace moe
