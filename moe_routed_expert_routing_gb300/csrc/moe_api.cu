// moe_api.cu -- the C ABI of libmoe.so (declared and documented in include/moe.h).
//
// Host side only: validation (fails closed before any launch), workspace
// layout, the static choice of the expert-GEMM path, and the launches.
// TileOps PR #1738 "Separate dispatched expert compute", Review follow-up:
// resolve one effective grouped-GEMM kernel up front, before building the
// gate-up and down steps, so nothing later can undo that choice.
#include <cstring>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t err, ready, counters, block_counts, block_base, h, x_sorted, y_sorted, inv, total;
};

// Workspace header, at fixed offsets so that moe_clear_device_error can clear
// it without the problem: the error word, then the fused decode kernel's
// per-expert readiness counts and its three GPU-wide counters (CTAs through
// their GEMM units, CTAs at the tail, units handed out), then the separate
// grouped GEMMs' two (units handed out, CTAs at the tail). The kernels leave
// the counters at zero after every launch.
constexpr size_t kReadyOffset = kAlign;
constexpr size_t kCountersOffset = kReadyOffset + sizeof(int32_t) * kMaxExperts;
constexpr size_t kHeaderBytes = (kCountersOffset + 5 * sizeof(int32_t) + kAlign - 1) / kAlign * kAlign;

void resolve(const moe_problem_t &p, int *path, int *tile_rows);

// 128-wide K blocks of the down GEMM, the unit its K parts are made of (for
// every weight layout alike, so that MXFP8 and bf16 weights split the same
// way and stay bit-identical); 1 when I is not a multiple of 128 (no split).
int down_k_blocks(const moe_problem_t &p) { return p.I % 128 == 0 ? p.I / 128 : 1; }

// The most K parts the down GEMM may split into for this problem (the SM
// count decides how many it does): its fp32 y then takes that many buffers.
int split_parts_max(const moe_problem_t &p)
{
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    if (path != MOE_PATH_SMALL_M || tile_rows != 16)
        return 1;
    const int kb = down_k_blocks(p);
    return kb % 4 == 0 ? 4 : (kb % 2 == 0 ? 2 : 1);
}

Layout layout_of(const moe_problem_t &p)
{
    const size_t cap = static_cast<size_t>(capacity_of(p));
    const size_t R = static_cast<size_t>(p.T_max) * p.k;
    const size_t n_blocks = static_cast<size_t>(dispatch_blocks(p));
    Layout L;
    L.err = 0;
    L.ready = kReadyOffset;
    L.counters = kCountersOffset;
    size_t o = kHeaderBytes;
    L.block_counts = o;
    o = align_up(o + sizeof(int32_t) * n_blocks * p.E);
    L.block_base = o;
    o = align_up(o + sizeof(int32_t) * n_blocks * p.E);
    L.h = o;
    o = align_up(o + 2 * cap * p.I);
    L.x_sorted = o;
    o = align_up(o + 2 * cap * p.H);
    L.y_sorted = o;
    o = align_up(o + 4 * cap * p.H * static_cast<size_t>(split_parts_max(p)));
    L.inv = o;
    o = align_up(o + sizeof(int32_t) * R);
    L.total = o;
    return L;
}

// H and I are whole 128-row weight tiles (and 128-wide K blocks)
bool tiles_of_128(const moe_problem_t &p) { return p.H % 128 == 0 && p.I % 128 == 0; }

moe_status_t check_problem(const moe_problem_t *p)
{
    if (!p)
        return MOE_ERR_NULL;
    if (p->T_max < 1 || p->E < 1 || p->E > kMaxExperts || p->k < 1 || p->k > p->E || p->k > kMaxTopK ||
        p->H < 1 || p->I < 1)
        return MOE_ERR_SHAPE;
    if (p->path < MOE_PATH_AUTO || p->path > MOE_PATH_TILED_1CTA)
        return MOE_ERR_SHAPE;
    if (p->weight_layout != MOE_WEIGHTS_ROW_MAJOR && p->weight_layout != MOE_WEIGHTS_PACKED &&
        p->weight_layout != MOE_WEIGHTS_MXFP8)
        return MOE_ERR_SHAPE;
    if (p->forward_form < MOE_FORWARD_AUTO || p->forward_form > MOE_FORWARD_ONE_KERNEL)
        return MOE_ERR_SHAPE;
    const long long R = static_cast<long long>(p->T_max) * p->k;
    if (R > (1LL << 28))
        return MOE_ERR_SHAPE;
    if (p->capacity != 0 && p->capacity < R)
        return MOE_ERR_SHAPE;
    if (static_cast<long long>(p->E) * 2 * p->I > (1LL << 31) || static_cast<long long>(p->E) * p->H > (1LL << 31))
        return MOE_ERR_SHAPE;
    // 64-element K blocks (one 128-byte swizzle row) and 64-column output
    // granularity; the PACKED and MXFP8 layouts are built of 128-row weight
    // tiles (and, for MXFP8, 128-wide K blocks), so they need multiples of 128
    if (p->H % 64 != 0 || p->I % 64 != 0)
        return MOE_ERR_ALIGN;
    if (p->weight_layout != MOE_WEIGHTS_ROW_MAJOR && !tiles_of_128(*p))
        return MOE_ERR_ALIGN;
    return MOE_OK;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

bool aligned256(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 255u) == 0; }

void resolve(const moe_problem_t &p, int *path, int *tile_rows)
{
    const double avg_rows = static_cast<double>(p.T_max) * p.k / p.E;
    int chosen = p.path;
    // M-small up to 8 routed rows per expert on average (16- and 32-row token
    // tiles; with 64-row tiles the gate-up GEMM's 16 tile::gather4 per stage
    // set the pace: at E=384, k=6, H=7168, I=3072, M-small vs single-CTA per
    // call, 8 rows 7065 vs 7062 us, 12 rows 9575 vs 7389, 16 rows 9578 vs
    // 7427, 24 rows 9644 vs 7498); single-CTA 128-row tiles from there to
    // 128 rows; CTA pairs from 128 rows, where experts start to
    // need a second 128-row tile (and stream their weights twice) while a
    // pair tile covers 256 rows and runs an expert's last tile of at most 128
    // rows swapped. Measured at E=384, k=6, H=7168, I=3072, pair vs single-CTA
    // per call: 64 rows 8163 vs 7717 us, 96 rows 8407 vs 7884, 128 rows 8662
    // vs 9170, 160 rows 9176 vs 10954.
    // MXFP8 weights: the M-small path at every batch size (its fused kernel
    // is the one that expands them).
    if (chosen == MOE_PATH_AUTO)
        chosen = (avg_rows <= 8.0 || p.weight_layout == MOE_WEIGHTS_MXFP8)
                     ? MOE_PATH_SMALL_M
                     : (avg_rows < 128.0 ? MOE_PATH_TILED_1CTA : MOE_PATH_TILED);
    *path = chosen;
    if (chosen == MOE_PATH_TILED || chosen == MOE_PATH_TILED_1CTA)
        *tile_rows = 128;
    else
        *tile_rows = avg_rows <= 2.0 ? 16 : (avg_rows <= 8.0 ? 32 : 64);
}

// The binary carries sm_103a code only: refuse any other device up front.
moe_status_t check_device()
{
    static thread_local int checked_device = -1;
    static thread_local bool ok = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (checked_device != dev) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        ok = (major == 10 && minor == 3);
        checked_device = dev;
    }
    return ok ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

template <typename T>
T *at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_ws(const moe_problem_t &p, const void *ws, size_t ws_bytes)
{
    if (!ws)
        return MOE_ERR_NULL;
    if (!aligned256(ws))
        return MOE_ERR_ALIGN;
    if (ws_bytes < layout_of(p).total)
        return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t record_stage(void *const *stage_events, int i, cudaStream_t s)
{
    if (!stage_events)
        return MOE_OK;
    return cuda_status(
        cudaEventRecordWithFlags(static_cast<cudaEvent_t>(stage_events[i]), s, cudaEventRecordExternal));
}

// K parts of the M-small down GEMM (1, 2 or 4), from static shapes only.
// Decode batches touch a handful of experts, so the down GEMM has few units
// (experts x H/128 weight tiles) for the SMs, and the last wave of units runs
// on a fraction of them: splitting K gives more, smaller units. The choice
// is the one with the fewest waves of full-K work, ceil(units * S / sms) / S,
// ties going to fewer parts. Each part goes to its own fp32 y buffer; the
// combine (or moe_expert_compute's reduction) adds them in part order, so
// the result is deterministic whatever the split. More parts must save at
// least 5% of the waves: each unit costs its readiness wait and epilogue.
// At one token, E=384, H=7168, I=3072 (336 units of full K): 2 parts give
// 672 units, 5 on 64 SMs and 4 on 88; 4 parts give 1344, 9 and 8.
int down_split_k(const moe_problem_t &p, int path, int tile_rows, int sms)
{
    if (path != MOE_PATH_SMALL_M || tile_rows != 16 || sms <= 0)
        return 1;
    const int kb = down_k_blocks(p);
    const long long R_max = static_cast<long long>(p.T_max) * p.k;
    const long long units = (R_max < p.E ? R_max : p.E) * ((p.H + 127) / 128);
    int best = 1;
    double best_waves = static_cast<double>((units + sms - 1) / sms);
    for (int parts = 2; parts <= 4; parts *= 2) {
        if (kb % parts != 0)
            continue;
        const double waves = static_cast<double>((units * parts + sms - 1) / sms) / parts;
        if (waves < 0.95 * best_waves) {
            best = parts;
            best_waves = waves;
        }
    }
    return best;
}

// Enqueue both GEMMs. With gather_perm set, `act` is x[T_max, H] itself and
// the gate-up GEMM fetches each sorted row x[perm[row] / k] straight into
// shared memory (no x_sorted round trip). A down GEMM that splits K writes
// its parts to the workspace's y buffers; with reduce_into set (the caller's
// y of moe_expert_compute) they are then summed into it in part order,
// otherwise (moe_forward) y_sorted is those buffers and the combine sums them.
moe_status_t enqueue_expert_compute(const moe_problem_t &p, const void *act, const int32_t *expert_offsets,
                                    const void *W13, const void *W2, float *y_sorted, void *ws, cudaStream_t s,
                                    void *const *stage_events = nullptr, float *reduce_into = nullptr,
                                    const int32_t *gather_perm = nullptr, bool fused = false,
                                    const MegaParams *mega = nullptr, bool y_f16 = false)
{
    const Layout L = layout_of(p);
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    const int sms = device_sm_count();
    if (sms <= 0)
        return MOE_ERR_CUDA;
    const int parts = down_split_k(p, path, tile_rows, sms);
    GemmProblem g;
    g.expert_offsets = expert_offsets;
    g.err = at<int32_t>(ws, L.err);
    g.E = p.E;
    g.cap = capacity_of(p);
    g.small_m = path == MOE_PATH_SMALL_M;
    g.cta_pair = path == MOE_PATH_TILED;
    g.w_packed = p.weight_layout == MOE_WEIGHTS_PACKED;
    g.w_mxfp8 = p.weight_layout == MOE_WEIGHTS_MXFP8;
    g.out_f16 = false;
    g.tile_rows = tile_rows;
    g.split_k = 1;
    g.pdl = path == MOE_PATH_SMALL_M;
    g.sched = at<int32_t>(ws, L.counters) + 3;
    // gate-up with the fused SiLU(gate) * up epilogue: x_sorted[cap, H] x W13[E, 2I, H] -> h[cap, I]
    g.act = act;
    g.gather = gather_perm != nullptr || mega != nullptr;
    g.perm = gather_perm;
    g.k = p.k;
    g.act_rows = g.gather ? p.T_max : g.cap;
    g.w = W13;
    g.out = at<void>(ws, L.h);
    g.K = p.H;
    g.n_out = p.I;
    g.w_rows_per_expert = 2 * p.I;
    g.up_row_offset = p.I;
    g.gated = true;
    GemmProblem up = g;
    moe_status_t st = MOE_OK;
    if (!fused) {
        st = cuda_status(launch_grouped_gemm(g, sms, s));
        if (st != MOE_OK)
            return st;
        if ((st = record_stage(stage_events, 3, s)) != MOE_OK)
            return st;
    }
    // down: h[cap, I] x W2[E, H, I] -> y_sorted[cap, H] (fp32, or fp16 for moe_forward's tiled paths)
    g.out_f16 = y_f16;
    g.act = at<void>(ws, L.h);
    g.gather = false;
    g.perm = nullptr;
    g.act_rows = g.cap;
    g.w = W2;
    g.out = y_sorted;
    g.K = p.I;
    g.n_out = p.H;
    g.w_rows_per_expert = p.H;
    g.up_row_offset = 0;
    g.gated = false;
    g.split_k = parts;
    if (!fused) {
        if (parts == 1 || !reduce_into)
            return cuda_status(launch_grouped_gemm(g, sms, s));
        g.out = at<float>(ws, L.y_sorted);   // the parts, then their sum into the caller's y
        st = cuda_status(launch_grouped_gemm(g, sms, s));
        if (st != MOE_OK)
            return st;
        return cuda_status(launch_reduce_parts(at<float>(ws, L.y_sorted), parts, expert_offsets, p.E, p.H, g.cap,
                                               reduce_into, sms, s, g.pdl));
    }
    // both GEMMs in one persistent launch; its stage marks share one instant
    st = cuda_status(launch_fused_small(up, g, at<int32_t>(ws, L.ready), at<int32_t>(ws, L.counters), sms, s, mega));
    if (st != MOE_OK)
        return st;
    return record_stage(stage_events, 3, s);
}

// moe_forward can run as one kernel: decode-size batches whose dispatch
// tables fit in the fused kernel's shared memory.
bool megakernel_possible(const moe_problem_t &p)
{
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    return path == MOE_PATH_SMALL_M && tile_rows == 16 &&
           fused_mega_fits(p.E, static_cast<long long>(p.T_max) * p.k, p.weight_layout == MOE_WEIGHTS_MXFP8);
}

// Both GEMMs in one persistent kernel: 16-row token tiles, or any M-small
// tile with MXFP8 weights (that kernel is their only GEMM).
bool fused_mlp_of(const moe_problem_t &p, int path, int tile_rows)
{
    return path == MOE_PATH_SMALL_M && (tile_rows == 16 || p.weight_layout == MOE_WEIGHTS_MXFP8);
}

bool use_megakernel(const moe_problem_t &p);

// moe_forward's gate-up GEMM gathers its activation rows from x itself
// (tile::gather4 through perm), with no x_sorted and no gather kernel: the
// M-small path, except MXFP8 weights in the three-kernel form. Their stages
// hold two 64-wide K blocks of the token tile (8, 16 or 32 gather4), which
// the TMA issues beside the code tiles and scale blocks; a sorted copy read
// with one box per K block measured faster at every tile height (in one
// process, bit-identical: decode T=8 679.4 vs 718.6 us, T=1 118.2 vs 119.3;
// Zipf small batch 1859.5 vs 2191.0; prefill 6267.3 vs 9831.6). The tiled
// paths read a materialised x_sorted for the same reason. The one-kernel
// form dispatches inside its CTAs and keeps the gather. bf16 weights (4
// gather4 per stage) keep it too: the sorted copy measured T=1 129.6 vs
// 127.7 us, T=8 813.7 vs 810.8.
bool gemm_gathers_rows(const moe_problem_t &p, int path, int tile_rows)
{
    (void)tile_rows;
    return path == MOE_PATH_SMALL_M && !(p.weight_layout == MOE_WEIGHTS_MXFP8 && !use_megakernel(p));
}

// MXFP8 weights are read by the M-small path only.
moe_status_t check_layout_path(const moe_problem_t &p)
{
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    return (p.weight_layout == MOE_WEIGHTS_MXFP8 && path != MOE_PATH_SMALL_M) ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

// moe_forward runs as one kernel (decode-size batches whose tables fit).
bool use_megakernel(const moe_problem_t &p)
{
    // On request only. AUTO keeps three kernels chained by programmatic
    // dependent launch: measured in one process at T=1, E=384, H=7168,
    // I=3072 with the down GEMM in 4 K parts, bf16 129.6 vs 131.5 us for one
    // kernel, MXFP8 117.3 vs 121.8 us (with 2 parts bf16 had been 133.0 vs
    // 132.5 us, and AUTO took one kernel there).
    return p.forward_form == MOE_FORWARD_ONE_KERNEL && megakernel_possible(p);
}

moe_status_t check_form(const moe_problem_t &p)
{
    return (p.forward_form == MOE_FORWARD_ONE_KERNEL && !megakernel_possible(p)) ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

// Kernel launches one moe_forward call enqueues (memsets not counted).
int forward_launches(const moe_problem_t &p)
{
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    if (use_megakernel(p))
        return 1;
    const long long R = static_cast<long long>(p.T_max) * p.k;
    int n = R <= kDispatchSlotsPerBlock ? 1 : 3;            // dispatch
    n += gemm_gathers_rows(p, path, tile_rows) ? 0 : 1;     // row gather (or fused into the gate-up GEMM)
    n += fused_mlp_of(p, path, tile_rows) ? 1 : 2;
    return n + 1;                                           // combine
}

}  // namespace

int device_sm_count()
{
    static thread_local int cached_dev = -1;
    static thread_local int cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (dev != cached_dev) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cached = n;
        cached_dev = dev;
    }
    return cached;
}

moe_status_t validate_problem(const moe_problem_t *problem) { return check_problem(problem); }

int capacity_of(const moe_problem_t &p) { return p.capacity ? p.capacity : p.T_max * p.k; }

long long dispatch_blocks(const moe_problem_t &p)
{
    const long long R = static_cast<long long>(p.T_max) * p.k;
    return (R + kDispatchSlotsPerBlock - 1) / kDispatchSlotsPerBlock;
}

moe_status_t validate_device() { return check_device(); }

bool use_pdl(const moe_problem_t &problem)
{
    int path = 0, tile_rows = 0;
    resolve(problem, &path, &tile_rows);
    return path == MOE_PATH_SMALL_M;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_workspace_size(const moe_problem_t *problem, size_t *bytes)
{
    if (!bytes)
        return MOE_ERR_NULL;
    const moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    *bytes = layout_of(*problem).total;
    return MOE_OK;
}

moe_status_t moe_resolve_path(const moe_problem_t *problem, int32_t *path, int32_t *tile_rows)
{
    if (!path || !tile_rows)
        return MOE_ERR_NULL;
    const moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    int p = 0, t = 0;
    resolve(*problem, &p, &t);
    *path = p;
    *tile_rows = t;
    return MOE_OK;
}

moe_status_t moe_resolve_profile(const moe_problem_t *problem, moe_profile_t *profile)
{
    if (!profile)
        return MOE_ERR_NULL;
    const moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const int sms = device_sm_count();
    if (sms <= 0)
        return MOE_ERR_CUDA;
    if (check_form(*problem) != MOE_OK || check_layout_path(*problem) != MOE_OK)
        return MOE_ERR_UNSUPPORTED;
    int path = 0, tile_rows = 0;
    resolve(*problem, &path, &tile_rows);
    std::memset(profile, 0, sizeof *profile);
    profile->path = path;
    profile->tile_rows = tile_rows;
    profile->down_split_k = down_split_k(*problem, path, tile_rows, sms);
    profile->pdl = use_pdl(*problem) ? 1 : 0;
    profile->fused_gather = gemm_gathers_rows(*problem, path, tile_rows) ? 1 : 0;
    profile->cta_pair = path == MOE_PATH_TILED ? 1 : 0;
    profile->fused_mlp = fused_mlp_of(*problem, path, tile_rows) ? 1 : 0;
    profile->megakernel = use_megakernel(*problem) ? 1 : 0;
    profile->kernel_launches = forward_launches(*problem);
    return MOE_OK;
}

moe_status_t moe_dispatch(const moe_problem_t *problem, const int32_t *topk_ids, const int32_t *d_num_tokens,
                          int32_t *expert_offsets, int32_t *perm, int32_t *inv, const void *x, void *x_sorted,
                          void *ws, size_t ws_bytes, void *stream)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!topk_ids || !expert_offsets || !perm || !inv)
        return MOE_ERR_NULL;
    if ((x == nullptr) != (x_sorted == nullptr))
        return MOE_ERR_NULL;
    if (x && (!aligned16(x) || !aligned16(x_sorted)))
        return MOE_ERR_ALIGN;
    if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK)
        return st;
    if ((st = check_device()) != MOE_OK)
        return st;
    const Layout L = layout_of(p);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = cuda_status(launch_dispatch(topk_ids, d_num_tokens, p.T_max, p.k, p.E, at<int32_t>(ws, L.block_counts),
                                     at<int32_t>(ws, L.block_base), expert_offsets, perm, inv,
                                     at<int32_t>(ws, L.err), s, use_pdl(p)));
    if (st != MOE_OK || !x)
        return st;
    return cuda_status(launch_gather_rows(x, perm, expert_offsets, p.E, p.k, p.H, capacity_of(p), x_sorted,
                                          device_sm_count(), s, use_pdl(p)));
}

moe_status_t moe_expert_compute(const moe_problem_t *problem, const void *x_sorted, const int32_t *expert_offsets,
                                const void *W13, const void *W2, float *y_sorted, void *ws, size_t ws_bytes,
                                void *stream)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!x_sorted || !expert_offsets || !W13 || !W2 || !y_sorted)
        return MOE_ERR_NULL;
    if (!aligned16(x_sorted) || !aligned16(W13) || !aligned16(W2) || !aligned16(y_sorted))
        return MOE_ERR_ALIGN;
    if (p.weight_layout == MOE_WEIGHTS_MXFP8)   // read by moe_forward's fused M-small kernel only
        return MOE_ERR_UNSUPPORTED;
    if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK)
        return st;
    if ((st = check_device()) != MOE_OK)
        return st;
    return enqueue_expert_compute(p, x_sorted, expert_offsets, W13, W2, y_sorted, ws,
                                  static_cast<cudaStream_t>(stream), nullptr, y_sorted);
}

moe_status_t moe_combine(const moe_problem_t *problem, const float *y_sorted, const int32_t *inv,
                         const float *topk_weights, const int32_t *d_num_tokens, void *out, void *stream)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!y_sorted || !inv || !topk_weights || !out)
        return MOE_ERR_NULL;
    if (!aligned16(y_sorted) || !aligned16(out))
        return MOE_ERR_ALIGN;
    if ((st = check_device()) != MOE_OK)
        return st;
    return cuda_status(launch_combine(y_sorted, false, inv, topk_weights, d_num_tokens, p.T_max, p.k, p.H, out,
                                      device_sm_count(), static_cast<cudaStream_t>(stream), use_pdl(p)));
}

static moe_status_t forward_impl(const moe_problem_t *problem, const void *x, const int32_t *topk_ids,
                                 const float *topk_weights, const int32_t *d_num_tokens, const void *W13,
                                 const void *W2, int32_t *expert_offsets, int32_t *perm, void *out, void *ws,
                                 size_t ws_bytes, void *stream, void *const *stage_events)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!x || !topk_ids || !topk_weights || !W13 || !W2 || !expert_offsets || !perm || !out)
        return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(W13) || !aligned16(W2) || !aligned16(out))
        return MOE_ERR_ALIGN;
    if ((st = check_ws(p, ws, ws_bytes)) != MOE_OK)
        return st;
    if ((st = check_device()) != MOE_OK)
        return st;
    if ((st = check_form(p)) != MOE_OK || (st = check_layout_path(p)) != MOE_OK)
        return st;
    const Layout L = layout_of(p);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = device_sm_count();
    int32_t *inv = at<int32_t>(ws, L.inv);
    void *x_sorted = at<void>(ws, L.x_sorted);
    float *y_sorted = at<float>(ws, L.y_sorted);
    auto mark = [&](int i) { return record_stage(stage_events, i, s); };
    int path = 0, tile_rows = 0;
    resolve(p, &path, &tile_rows);
    // decode-size batches (M-small, 16-row token tiles) whose dispatch tables
    // fit in shared memory: the whole call is one persistent kernel (local
    // dispatch in every CTA, both GEMMs, combine); its stage marks all fall
    // after it.
    if (use_megakernel(p)) {
        MegaParams mp;
        mp.ids = topk_ids;
        mp.topk_w = topk_weights;
        mp.d_num_tokens = d_num_tokens;
        mp.T_max = p.T_max;
        mp.expert_offsets_out = expert_offsets;
        mp.perm_out = perm;
        mp.out = out;
        if ((st = mark(0)) != MOE_OK)
            return st;
        st = enqueue_expert_compute(p, x, nullptr, W13, W2, y_sorted, ws, s, nullptr, nullptr, nullptr, true, &mp);
        for (int i = 1; st == MOE_OK && i < 6; ++i)
            st = mark(i);
        return st;
    }
    // a down GEMM that splits K leaves its parts in the workspace's y buffers;
    // the combine sums them in part order
    const int parts = down_split_k(p, path, tile_rows, sms);
    // decode-size batches (M-small, 16-row token tiles): both GEMMs run as one
    // persistent kernel whose down units wait on per-expert counts (zero at
    // every launch: the kernel clears them at its tail). Measured in one
    // process against two launches: -1.3% per decode step; +2% on 32-row
    // tiles, which keep two launches.
    const bool fused_mlp = fused_mlp_of(p, path, tile_rows);
    if ((st = mark(0)) != MOE_OK)
        return st;
    st = cuda_status(launch_dispatch(topk_ids, d_num_tokens, p.T_max, p.k, p.E, at<int32_t>(ws, L.block_counts),
                                     at<int32_t>(ws, L.block_base), expert_offsets, perm, inv,
                                     at<int32_t>(ws, L.err), s, use_pdl(p)));
    if (st != MOE_OK || (st = mark(1)) != MOE_OK)
        return st;
    // On the M-small path the gate-up GEMM gathers its few rows per tile from x
    // itself (tile::gather4, at most 16 per stage). The tiled paths read a
    // materialised x_sorted: at 32 gather4 per 128-row stage the TMA issue rate,
    // not the data, limited the gate-up GEMM (4.5x slower on the large shape).
    const bool fused_gather = gemm_gathers_rows(p, path, tile_rows);
    if (!fused_gather)
        st = cuda_status(launch_gather_rows(x, perm, expert_offsets, p.E, p.k, p.H, capacity_of(p), x_sorted, sms, s,
                                            use_pdl(p)));
    if (st != MOE_OK || (st = mark(2)) != MOE_OK)
        return st;
    // tiled paths: y between the down GEMM and the combine in fp16 (half the
    // bytes of the largest intermediate; within the output tolerance). The
    // M-small path keeps fp32 (its y is small).
    const bool y_f16 = path != MOE_PATH_SMALL_M;
    // A few tokens with bf16 weights, whose dispatch tables fit the fused
    // kernel's shared memory and whose gate-up units fit one wave on one SM
    // fewer (so the fused kernel starts beside the dispatch block): the fused
    // kernel dispatches the call's slots itself (the stable dispatch, the
    // same tables) and starts its GEMM units without waiting for the dispatch
    // kernel, which runs beside it for the caller's expert_offsets and perm
    // and the combine's inv. Measured at one token, E=384, H=7168, I=3072, in
    // one process, outputs bit-identical: 126.6 vs 127.5 us per call; at
    // eight tokens (full grid) +1.9 us, so those keep the plain form.
    const bool dispatch_beside = fused_mlp && megakernel_possible(p) && p.weight_layout != MOE_WEIGHTS_MXFP8 &&
                                 fused_grid_sms(false, false, capacity_of(p), p.E, p.I, tile_rows, sms) < sms;
    if (dispatch_beside) {
        MegaParams mp;
        mp.ids = topk_ids;
        mp.topk_w = topk_weights;
        mp.d_num_tokens = d_num_tokens;
        mp.T_max = p.T_max;
        mp.expert_offsets_out = expert_offsets;
        mp.perm_out = perm;
        mp.out = out;
        mp.combine_apart = true;
        st = enqueue_expert_compute(p, x, nullptr, W13, W2, y_sorted, ws, s, stage_events, nullptr, nullptr, true,
                                    &mp);
    } else {
        st = enqueue_expert_compute(p, fused_gather ? x : x_sorted, expert_offsets, W13, W2, y_sorted, ws, s,
                                    stage_events, nullptr, fused_gather ? perm : nullptr, fused_mlp, nullptr,
                                    y_f16);
    }
    if (st != MOE_OK || (st = mark(4)) != MOE_OK)
        return st;
    st = cuda_status(launch_combine(y_sorted, y_f16, inv, topk_weights, d_num_tokens, p.T_max, p.k, p.H, out, sms,
                                    s, use_pdl(p), parts, static_cast<size_t>(capacity_of(p)) * p.H, true));
    if (st != MOE_OK)
        return st;
    return mark(5);
}

moe_status_t moe_forward(const moe_problem_t *problem, const void *x, const int32_t *topk_ids,
                         const float *topk_weights, const int32_t *d_num_tokens, const void *W13, const void *W2,
                         int32_t *expert_offsets, int32_t *perm, void *out, void *ws, size_t ws_bytes, void *stream)
{
    return forward_impl(problem, x, topk_ids, topk_weights, d_num_tokens, W13, W2, expert_offsets, perm, out, ws,
                        ws_bytes, stream, nullptr);
}

moe_status_t moe_forward_profiled(const moe_problem_t *problem, const void *x, const int32_t *topk_ids,
                                  const float *topk_weights, const int32_t *d_num_tokens, const void *W13,
                                  const void *W2, int32_t *expert_offsets, int32_t *perm, void *out, void *ws,
                                  size_t ws_bytes, void *stream, void *const *stage_events)
{
    if (!stage_events)
        return MOE_ERR_NULL;
    for (int i = 0; i < 6; ++i)
        if (!stage_events[i])
            return MOE_ERR_NULL;
    return forward_impl(problem, x, topk_ids, topk_weights, d_num_tokens, W13, W2, expert_offsets, perm, out, ws,
                        ws_bytes, stream, stage_events);
}

moe_status_t moe_pack_weights(const moe_problem_t *problem, const void *W13, const void *W2, void *W13_packed,
                              void *W2_packed, void *stream)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!W13 || !W2 || !W13_packed || !W2_packed)
        return MOE_ERR_NULL;
    if (!tiles_of_128(p) || !aligned16(W13) || !aligned16(W2) || !aligned16(W13_packed) || !aligned16(W2_packed))
        return MOE_ERR_ALIGN;
    if ((st = check_device()) != MOE_OK)
        return st;
    return cuda_status(launch_pack_weights(W13, W2, W13_packed, W2_packed, p.E, p.H, p.I, device_sm_count(),
                                           static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_weight_bytes(const moe_problem_t *problem, int32_t layout, size_t *w13_bytes, size_t *w2_bytes)
{
    if (!w13_bytes || !w2_bytes)
        return MOE_ERR_NULL;
    const moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    if (layout != MOE_WEIGHTS_ROW_MAJOR && layout != MOE_WEIGHTS_PACKED && layout != MOE_WEIGHTS_MXFP8)
        return MOE_ERR_SHAPE;
    const size_t n13 = static_cast<size_t>(problem->E) * 2 * problem->I * problem->H;
    const size_t n2 = static_cast<size_t>(problem->E) * problem->H * problem->I;
    if (layout == MOE_WEIGHTS_MXFP8) {
        *w13_bytes = n13 + n13 / 32;
        *w2_bytes = n2 + n2 / 32;
    } else {
        *w13_bytes = 2 * n13;
        *w2_bytes = 2 * n2;
    }
    return MOE_OK;
}

moe_status_t moe_quantize_weights(const moe_problem_t *problem, const void *W13, const void *W2, void *W13_mx,
                                  void *W2_mx, void *stream)
{
    moe_status_t st = check_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!W13 || !W2 || !W13_mx || !W2_mx)
        return MOE_ERR_NULL;
    if (!tiles_of_128(p) || !aligned16(W13) || !aligned16(W2) || !aligned16(W13_mx) || !aligned16(W2_mx))
        return MOE_ERR_ALIGN;
    if ((st = check_device()) != MOE_OK)
        return st;
    return cuda_status(launch_quantize_weights_mxfp8(W13, W2, W13_mx, W2_mx, p.E, p.H, p.I, device_sm_count(),
                                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_last_device_error(const void *ws, void *stream, int32_t *host_code)
{
    if (!ws || !host_code)
        return MOE_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    *host_code = v;
    return MOE_OK;
}

moe_status_t moe_clear_device_error(void *ws, void *stream)
{
    if (!ws)
        return MOE_ERR_NULL;
    // the error word and the fused decode kernel's counters: afterwards a
    // workspace of any former contents is ready for moe_forward
    return cudaMemsetAsync(ws, 0, kHeaderBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK
                                                                                                 : MOE_ERR_CUDA;
}

const char *moe_status_string(moe_status_t status)
{
    switch (status) {
    case MOE_OK:
        return "MOE_OK";
    case MOE_ERR_NULL:
        return "MOE_ERR_NULL: a required pointer is NULL";
    case MOE_ERR_SHAPE:
        return "MOE_ERR_SHAPE: a size is out of range or inconsistent";
    case MOE_ERR_ALIGN:
        return "MOE_ERR_ALIGN: H or I not a multiple of 64 (of 128 for the PACKED and MXFP8 weight layouts), "
               "or a misaligned buffer";
    case MOE_ERR_WORKSPACE:
        return "MOE_ERR_WORKSPACE: workspace smaller than moe_workspace_size()";
    case MOE_ERR_UNSUPPORTED:
        return "MOE_ERR_UNSUPPORTED: the device is not sm_103 (GB300), or the weight layout or forward form "
               "asked for is not available for this shape";
    case MOE_ERR_CUDA:
        return "MOE_ERR_CUDA: a CUDA call failed";
    }
    return "unknown moe_status_t";
}

}  // extern "C"
