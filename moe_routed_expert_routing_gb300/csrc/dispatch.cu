// dispatch.cu -- local dispatch of routed slots into a tight expert-major batch.
//
// TileOps PR #1738 "Separate dispatched expert compute", Summary: routed
// expert execution starts with a local dispatch into tight expert-major
// batches, with GPU-resident row counts behind a static capacity; Scope:
// no padding, the valid-row count is expert_offsets[E].
//
// Sized from static shapes only; the token count is read on the device, so a
// captured graph can replay with another T.
//
// Up to 1024 routed slots (decode-size batches) one block does everything in
// one launch: histogram, exclusive scan over experts, stable scatter.
// Larger batches take three launches:
//   1. count:   each block histograms its 1024 consecutive slots (shared-
//               memory atomics; order does not matter for counts).
//   2. scan:    one block turns the per-block counts into expert_offsets
//               (exclusive prefix over experts) and, per expert, the first
//               row owned by each block (exclusive prefix over blocks).
//   3. scatter: each block walks its slots again in ascending order, 256 at
//               a time.
// In both forms a slot's row = the first row its block owns for the expert +
// the same-expert slots before it in earlier rounds, earlier warps and lower
// lanes: exactly the stable order (ascending slot index inside each expert),
// bit-exact and independent of scheduling.
// A separate, optional launch gathers x rows into the sorted batch.
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kDispatchThreads / 32;

__device__ __forceinline__ int dynamic_slots(const int32_t *d_num_tokens, int T_max, int k)
{
    int T = T_max;
    if (d_num_tokens) {
        T = *d_num_tokens;
        T = T < 0 ? 0 : (T > T_max ? T_max : T);
    }
    return T * k;
}

// Histogram of slots [s0, s1) into hist[E] (shared memory, zeroed by the caller).
__device__ __forceinline__ void count_slots(const int32_t *__restrict__ ids, int s0, int s1, int E, int *hist,
                                            int32_t *err)
{
    bool bad = false;
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
        const int e = ids[s];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else if (e != -1)
            bad = true;
    }
    if (bad)
        atomicOr(err, MOE_DEVERR_BAD_EXPERT_ID);
}

// Stable scatter of slots [s0, s1): cursor[E] holds the next free row of each
// expert for this block (advanced here); wcnt[kWarps * E] is zeroed scratch.
__device__ __forceinline__ void scatter_slots(const int32_t *__restrict__ ids, int s0, int s1, int E, int *cursor,
                                              int *wcnt, int32_t *__restrict__ perm, int32_t *__restrict__ inv)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = s0; base < s1; base += kDispatchThreads) {
        const int s = base + threadIdx.x;
        const int e = s < s1 ? ids[s] : -1;
        const bool valid = e >= 0 && e < E;
        // lanes routed to the same expert; invalid lanes get a key of their own
        const unsigned peers = __match_any_sync(kFull, valid ? e : -1 - lane);
        const int rank = __popc(peers & lt_mask);
        const int cnt = __popc(peers);
        if (valid && rank == 0)
            wcnt[warp * E + e] = cnt;
        __syncthreads();
        if (valid) {
            int before = 0;
            for (int w = 0; w < warp; ++w)
                before += wcnt[w * E + e];
            const int row = cursor[e] + before + rank;
            perm[row] = s;
            inv[s] = row;
        } else if (s < s1) {
            inv[s] = -1;
        }
        __syncthreads();
        if (valid && rank == 0) {
            atomicAdd(&cursor[e], cnt);
            wcnt[warp * E + e] = 0;
        }
        __syncthreads();
    }
}

// Exclusive scan of v over the 256 threads of the block; returns the prefix
// before this thread and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, x, o);
        if (lane >= o)
            x += n;
    }
    if (lane == 31)
        warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, w, o);
            if (lane >= o)
                w += n;
        }
        if (lane < kWarps)
            warp_tot[lane] = w;
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
    *total = warp_tot[kWarps - 1];
    __syncthreads();
    return excl;
}

// All slots (<= 1024) in one block: histogram, scan, stable scatter.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_single_block_kernel(
    const int32_t *__restrict__ ids, const int32_t *d_num_tokens, int T_max, int k, int E,
    int32_t *__restrict__ expert_offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv, int32_t *err)
{
    extern __shared__ int sm[];
    int *cursor = sm;                 // [E]: counts, then first rows
    int *wcnt = sm + E;               // [kWarps][E]
    __shared__ int warp_tot[kWarps];
    pdl_wait();
    pdl_trigger();
    const int R = dynamic_slots(d_num_tokens, T_max, k);
    for (int i = threadIdx.x; i < E * (1 + kWarps); i += blockDim.x)
        sm[i] = 0;
    __syncthreads();
    count_slots(ids, 0, R, E, cursor, err);
    __syncthreads();
    // exclusive scan over experts: thread i owns experts [i*per, (i+1)*per)
    const int per = (E + kDispatchThreads - 1) / kDispatchThreads;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e)
        local += cursor[e];
    int total = 0;
    int run = block_exclusive_scan(local, warp_tot, &total);
    for (int e = e0; e < e0 + per && e < E; ++e) {
        const int c = cursor[e];
        cursor[e] = run;
        expert_offsets[e] = run;
        run += c;
    }
    if (threadIdx.x == 0)
        expert_offsets[E] = total;
    __syncthreads();
    scatter_slots(ids, 0, R, E, cursor, wcnt, perm, inv);
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_count_kernel(const int32_t *__restrict__ ids,
                                                                          const int32_t *d_num_tokens, int T_max,
                                                                          int k, int E,
                                                                          int32_t *__restrict__ block_counts,
                                                                          int32_t *err)
{
    extern __shared__ int hist[];
    pdl_wait();
    pdl_trigger();
    const int R = dynamic_slots(d_num_tokens, T_max, k);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        hist[e] = 0;
    __syncthreads();
    const int s0 = blockIdx.x * kDispatchSlotsPerBlock;
    const int s1 = min(s0 + kDispatchSlotsPerBlock, R);
    count_slots(ids, s0, s1, E, hist, err);
    __syncthreads();
    int32_t *dst = block_counts + static_cast<size_t>(blockIdx.x) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        dst[e] = hist[e];
}

// One block of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(const int32_t *__restrict__ block_counts,
                                                             int n_blocks, int E,
                                                             int32_t *__restrict__ block_base,
                                                             int32_t *__restrict__ expert_offsets)
{
    __shared__ int warp_tot[32];
    pdl_wait();
    pdl_trigger();
    const int e = threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int total = 0;
    if (e < E) {
        for (int b = 0; b < n_blocks; ++b) {
            const size_t i = static_cast<size_t>(b) * E + e;
            const int c = block_counts[i];
            block_base[i] = total;
            total += c;
        }
    }
    // exclusive scan of `total` over experts
    int v = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += n;
    }
    if (lane == 31)
        warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFull, w, o);
            if (lane >= o)
                w += n;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = v - total + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < E) {
        expert_offsets[e] = excl;
        if (e == E - 1)
            expert_offsets[E] = excl + total;
        for (int b = 0; b < n_blocks; ++b)
            block_base[static_cast<size_t>(b) * E + e] += excl;
    }
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_scatter_kernel(
    const int32_t *__restrict__ ids, const int32_t *d_num_tokens, int T_max, int k, int E,
    const int32_t *__restrict__ block_base, int32_t *__restrict__ perm, int32_t *__restrict__ inv)
{
    extern __shared__ int sm[];
    int *cursor = sm;          // [E]   next free row of each expert for this block
    int *wcnt = sm + E;        // [kWarps][E] slots per expert in each warp, this pass of 256 slots
    pdl_wait();
    pdl_trigger();
    const int R = dynamic_slots(d_num_tokens, T_max, k);
    const int s0 = blockIdx.x * kDispatchSlotsPerBlock;
    const int s1 = min(s0 + kDispatchSlotsPerBlock, R);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        cursor[e] = block_base[static_cast<size_t>(blockIdx.x) * E + e];
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x)
        wcnt[i] = 0;
    __syncthreads();
    scatter_slots(ids, s0, s1, E, cursor, wcnt, perm, inv);
}

// x_sorted[row] = x[perm[row] / k] for row < expert_offsets[E]. One warp per
// row (grid-stride over rows); each lane moves 16-byte vectors lane, lane+32,
// ..., with eight loads in flight before their stores.
constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 8;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint4 *__restrict__ x,
                                                                     const int32_t *__restrict__ perm,
                                                                     const int32_t *__restrict__ expert_offsets,
                                                                     int E, int k, int vec_per_row, int cap,
                                                                     uint4 *__restrict__ x_sorted)
{
    pdl_wait();
    pdl_trigger();
    const int n_rows = min(expert_offsets[E], cap);
    const int lane = threadIdx.x & 31;
    const int warps = kGatherThreads / 32;
    for (int r = blockIdx.x * warps + (threadIdx.x >> 5); r < n_rows; r += gridDim.x * warps) {
        const int t = perm[r] / k;
        const uint4 *src = x + static_cast<size_t>(t) * vec_per_row;
        uint4 *dst = x_sorted + static_cast<size_t>(r) * vec_per_row;
        for (int c0 = lane; c0 < vec_per_row; c0 += 32 * kGatherUnroll) {
            uint4 v[kGatherUnroll];
#pragma unroll
            for (int q = 0; q < kGatherUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < vec_per_row)
                    v[q] = __ldg(src + c);
            }
#pragma unroll
            for (int q = 0; q < kGatherUnroll; ++q) {
                const int c = c0 + 32 * q;
                if (c < vec_per_row)
                    dst[c] = v[q];
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const int32_t *topk_ids, const int32_t *d_num_tokens, int T_max, int k, int E,
                            int32_t *block_counts, int32_t *block_base, int32_t *expert_offsets, int32_t *perm,
                            int32_t *inv, int32_t *err, cudaStream_t stream, bool pdl)
{
    const int R_max = T_max * k;
    const int n_blocks = (R_max + kDispatchSlotsPerBlock - 1) / kDispatchSlotsPerBlock;
    const size_t scatter_smem = sizeof(int) * E * (1 + kWarps);
    if (n_blocks <= 1)
        return launch_k(dispatch_single_block_kernel, dim3(1), dim3(kDispatchThreads), scatter_smem, stream, pdl,
                        topk_ids, d_num_tokens, T_max, k, E, expert_offsets, perm, inv, err);
    const size_t count_smem = sizeof(int) * E;
    cudaError_t e = launch_k(dispatch_count_kernel, dim3(n_blocks), dim3(kDispatchThreads), count_smem, stream, pdl,
                             topk_ids, d_num_tokens, T_max, k, E, block_counts, err);
    if (e != cudaSuccess)
        return e;
    e = launch_k(dispatch_scan_kernel, dim3(1), dim3(1024), 0, stream, pdl, block_counts, n_blocks, E, block_base,
                 expert_offsets);
    if (e != cudaSuccess)
        return e;
    return launch_k(dispatch_scatter_kernel, dim3(n_blocks), dim3(kDispatchThreads), scatter_smem, stream, pdl,
                    topk_ids, d_num_tokens, T_max, k, E, block_base, perm, inv);
}

cudaError_t launch_gather_rows(const void *x, const int32_t *perm, const int32_t *expert_offsets, int E, int k, int H,
                               int cap, void *x_sorted, int num_sms, cudaStream_t stream, bool pdl)
{
    const int warps = kGatherThreads / 32;
    int blocks = (cap + warps - 1) / warps;
    blocks = blocks < num_sms * 8 ? blocks : num_sms * 8;
    if (blocks < 1)
        blocks = 1;
    return launch_k(gather_rows_kernel, dim3(blocks), dim3(kGatherThreads), 0, stream, pdl,
                    static_cast<const uint4 *>(x), perm, expert_offsets, E, k, H / 8, cap,
                    static_cast<uint4 *>(x_sorted));
}

}  // namespace moe
