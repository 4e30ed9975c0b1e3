// moe_internal.h -- declarations shared by the translation units of libmoe.so
// (kernels + launchers). Not part of the public ABI (include/moe.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

// ---- limits of this build (checked by host validation) ----
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 64;
constexpr int kDispatchThreads = 256;
constexpr int kDispatchSlotsPerBlock = 1024;  // routed slots counted/scattered by one block

// Pipeline waits inside the GEMM kernels give up after this long (the device
// error word then carries MOE_DEVERR_WAIT_TIMEOUT).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---- programmatic dependent launch ----
// With `pdl` set, a kernel of the library may start while the kernel before
// it on the stream is still finishing (cudaLaunchAttributeProgrammaticStream-
// Serialization): it runs its prologue, then waits (griddepcontrol.wait) for
// the previous grid's completion and memory before touching any global data,
// and releases its own dependents (griddepcontrol.launch_dependents), only
// after that wait. Every kernel waits before it finishes, so completion stays
// transitive along the stream, and when a kernel starts, every kernel two or
// more launches back has completed; without the attribute both instructions
// are no-ops. The host turns
// it on for the M-small (decode) path only: measured in one process, it saves
// ~8 us per decode step and costs ~90 us per large-batch step, where the early
// dependents share the SMs with the persistent GEMM.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l1(const void *p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                     Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- kernels whose CTAs wait on one another ----
// Such a kernel is correct only if every CTA of its grid is resident at
// once. The launch asks for that guarantee (cudaLaunchAttributeCooperative:
// the grid starts only when all of its CTAs fit, and a grid that could never
// fit is refused), and the host first sizes the grid against the occupancy
// the device reports for the kernel. Pure host arithmetic: the grid to
// launch for `want` CTAs when `per_sm` CTAs fit on one of `sms` SMs, or 0
// when none fits (the launch is then refused before it is made).
inline int coresident_grid(long long want, int per_sm, int sms)
{
    if (want < 1 || per_sm < 1 || sms < 1)
        return 0;
    const long long most = static_cast<long long>(per_sm) * sms;
    return static_cast<int>(want < most ? want : most);
}

// SMs the fused decode kernel's grid may use. The dispatch block launched
// before it and one of its CTAs cannot share an SM (shared memory), and the
// cooperative launch waits until the whole grid fits. Where its gate-up
// units (at most (min(cap, E) + cap / tile_rows) row tiles x ceil(I / 128))
// fit one wave on one SM fewer (a few tokens; bf16, three-kernel form) the
// grid leaves that SM to the dispatch, so the kernel starts, and runs its
// prologue, under it. Measured at one token, E=384, H=7168, I=3072, in one
// process, outputs bit-identical: 127.4 vs 128.3 us per call; at eight
// tokens the SM is worth more.
inline int fused_grid_sms(bool whole_forward, bool mxfp8, long long cap, int E, int I, int tile_rows, int sms)
{
    const long long tiles_bound = (cap < E ? cap : E) + cap / tile_rows;
    const long long units1_bound = tiles_bound * ((I + 127) / 128);
    return (!whole_forward && !mxfp8 && sms > 1 && units1_bound <= sms - 1) ? sms - 1 : sms;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k_coresident(void (*kernel)(KArgs...), long long want_ctas, dim3 block, size_t smem,
                                cudaStream_t stream, bool pdl, int sms, Args &&...args)
{
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, static_cast<int>(block.x),
                                                                  smem);
    if (e != cudaSuccess)
        return e;
    const int grid = coresident_grid(want_ctas, per_sm, sms);
    if (grid < 1)
        return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- dispatch (dispatch.cu) ----
cudaError_t launch_dispatch(const int32_t *topk_ids, const int32_t *d_num_tokens, int T_max, int k, int E,
                            int32_t *block_counts, int32_t *block_base, int32_t *expert_offsets,
                            int32_t *perm, int32_t *inv, int32_t *err, cudaStream_t stream, bool pdl);

cudaError_t launch_gather_rows(const void *x, const int32_t *perm, const int32_t *expert_offsets, int E, int k,
                               int H, int cap, void *x_sorted, int num_sms, cudaStream_t stream, bool pdl);

// ---- combine (combine.cu) ----
// y_sorted is fp32, or fp16 when y_f16 is set (moe_forward's tiled paths).
// fp32 y may be `parts` partial buffers of a down GEMM that split K,
// part_stride elements apart: each row is their sum in part order.
// routing_early: inv was written at least two launches back on this stream
// (moe_forward) and the token count and weights are inputs, so the kernel
// may pull a block's routing into L1 before its dependency wait.
cudaError_t launch_combine(const void *y_sorted, bool y_f16, const int32_t *inv, const float *topk_weights,
                           const int32_t *d_num_tokens, int T_max, int k, int H, void *out, int num_sms,
                           cudaStream_t stream, bool pdl, int parts = 1, size_t part_stride = 0,
                           bool routing_early = false);

// y_sorted[r] = ((p0 + p1) + p2) + p3 over the `parts` fp32 partial buffers of
// [cap, H] starting at parts_base, for r < expert_offsets[E].
cudaError_t launch_reduce_parts(const float *parts_base, int parts, const int32_t *expert_offsets, int E, int H,
                                int cap, float *y_sorted, int num_sms, cudaStream_t stream, bool pdl);

// ---- packed weights (weights_pack.cu) ----
cudaError_t launch_pack_weights(const void *W13, const void *W2, void *W13_packed, void *W2_packed, int E, int H,
                                int I, int num_sms, cudaStream_t stream);

// ---- MXFP8 weights (weights_mx.cu) ----
// W13[E, 2I, H] and W2[E, H, I] bf16 -> the MOE_WEIGHTS_MXFP8 buffers: E4M3
// codes (row-major), then the E8M0 scale codes in (128-row tile, 128-wide K
// block, row, sub-block) order.
cudaError_t launch_quantize_weights_mxfp8(const void *W13, const void *W2, void *W13_mx, void *W2_mx, int E, int H,
                                          int I, int num_sms, cudaStream_t stream);

// ---- expert GEMMs (grouped_gemm.cu) ----
struct GemmProblem {
    const void *act;          // [act_rows, K] bf16: sorted rows, or x itself when gather is set
    int act_rows;             // rows of `act` (cap, or T_max for x)
    bool gather;              // A rows fetched from x through perm (tile::gather4), gate-up only
    const int32_t *perm;      // gather: sorted row -> routed slot
    int k;                    // gather: token = slot / k
    const void *w;            // [E, w_rows_per_expert, K] bf16
    void *out;                // [cap, n_out]: bf16 h (gated) or fp32 y (down)
    const int32_t *expert_offsets;
    int32_t *err;
    int E, cap, K, n_out;
    int w_rows_per_expert;
    int up_row_offset;        // gated: row offset of the up half inside one expert
    bool gated;               // fused SiLU(gate) * up epilogue
    bool small_m;             // weights on the MMA M side (M-small path)
    int tile_rows;            // activation rows per tile: 128 (tiled) or 16/32/64 (M-small)
    int split_k;              // 1, 2 or 4 (M-small down GEMM only): K parts, part p of fp32 out at out + p * cap * n_out
    bool pdl;                 // programmatic dependent launch
    bool cta_pair;            // tiled path on 2-CTA clusters (tcgen05 cta_group::2)
    bool w_packed;            // `w` is in the access-ordered PACKED layout
    bool w_mxfp8;             // `w` is in the MXFP8 layout (codes, then scale blocks): fused kernel only
    bool out_f16;             // tiled down GEMM: y as fp16 (saturated; MOE_DEVERR_Y_RANGE if clipped)
    int32_t *sched = nullptr; // single-CTA grouped GEMM (M-small and tiled): two workspace counters (units
                              // handed out, CTAs at the tail), zero before the launch and left zero by it;
                              // null: units dealt round-robin
};

cudaError_t launch_grouped_gemm(const GemmProblem &p, int num_sms, cudaStream_t stream);

// The rest of moe_forward for the whole-forward form of the fused kernel:
// the dispatch inputs and outputs and the combine's weights and output.
struct MegaParams {
    const int32_t *ids;            // [T_max, k]
    const float *topk_w;           // [T_max, k]
    const int32_t *d_num_tokens;   // nullable
    int T_max;
    int32_t *expert_offsets_out;   // [E + 1]
    int32_t *perm_out;             // [cap]
    void *out;                     // [T_max, H] bf16
    // the dispatch kernel runs beside the fused kernel (and writes the tables
    // above and inv) and the combine kernel after it: the fused kernel only
    // dispatches locally for its own units
    bool combine_apart = false;
};

// Both M-small GEMMs in one persistent launch (gate-up with gathered rows, then
// down). ready[E] and counters[2] must be zero when the kernel starts; the
// kernel leaves them at zero (the last CTA out clears them), so a workspace
// that starts zeroed needs no clearing between calls. With `mega`, the launch
// is the whole forward (dispatch, both GEMMs, combine); up.perm and the
// expert_offsets of both problems are then not read, and a split down GEMM
// writes its halves to down.out and down.out + cap * H (no zeroing needed).
cudaError_t launch_fused_small(const GemmProblem &up, const GemmProblem &down, int32_t *ready, int32_t *counters,
                               int num_sms, cudaStream_t stream, const MegaParams *mega = nullptr);

// Whether the whole-forward kernel's shared-memory expert tables for E experts
// and `slots` = T_max * k routed slots fit next to its pipeline on this device.
bool fused_mega_fits(int E, long long slots, bool mxfp8);

// number of SMs of the current device (cached)
int device_sm_count();

// host validation shared by the entry points (moe_api.cu)
moe_status_t validate_problem(const moe_problem_t *problem);
// rows of the sorted batch: the problem's capacity, or T_max * k when it is 0
int capacity_of(const moe_problem_t &problem);
// blocks of the multi-block dispatch: one per kDispatchSlotsPerBlock routed slots
long long dispatch_blocks(const moe_problem_t &problem);
moe_status_t validate_device();
// whether launches for this problem use programmatic dependent launch (M-small path)
bool use_pdl(const moe_problem_t &problem);

}  // namespace moe
