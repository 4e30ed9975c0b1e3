// combine.cu -- routing-weighted top-k sum back into token order.
//
// TileOps PR #1738 "Separate dispatched expert compute", Summary: routed
// expert execution ends with a combine, and the routing weights stay outside
// expert compute. The FlashInfer moe_ep page (kernel API migration) likewise
// reduces the top-k contributions into one (T, hidden) output.
//
//   out[t, m] = bf16( sum_{j = 0..k-1} w[t, j] * y_sorted[inv[t*k + j], m] )
//
// y_sorted is the down GEMM's output: fp32, or fp16 on moe_forward's tiled
// paths (widened exactly before use). fp32 products and sums in
// ascending j (no fused multiply-add), one rounding at the end: the result
// is deterministic (no atomics) and identical to a plain sequential loop.
// Work item = one token x 1024 columns, so even a single token spreads over
// several SMs; each thread owns 8 consecutive columns, read as two 16-byte
// loads per routed row and written as one 16-byte store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

constexpr int kCombineThreads = 128;
constexpr int kColsPerItem = kCombineThreads * 8;   // one work item = one token x 1024 columns

// Eight consecutive columns of one fp32 y row: two 16-byte loads. (fp16 y is
// read as raw 16-byte vectors and widened exactly where it is summed; a down
// GEMM that split K leaves fp32 y as `parts` partial rows, `part_stride`
// elements apart, summed in part order (((p0 + p1) + p2) + p3), the order in
// which moe_expert_compute reduces its parts, so every route gives the same
// bits.)
__device__ __forceinline__ void load8(const float *y, size_t i, float (&f)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4 *>(y + i));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(y + i) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <typename Y, int kParts>
__global__ void __launch_bounds__(kCombineThreads, sizeof(Y) == 2 ? 8 : 1) combine_kernel(const Y *__restrict__ y_sorted,
                                                                  const int32_t *__restrict__ inv,
                                                                  const float *__restrict__ w,
                                                                  const int32_t *d_num_tokens, int T_max, int k,
                                                                  int vec_per_row, uint4 *__restrict__ out,
                                                                  size_t part_stride, bool routing_early)
{
    const int groups = (vec_per_row * 8 + kColsPerItem - 1) / kColsPerItem;
    if (routing_early && threadIdx.x < k && blockIdx.x < static_cast<long long>(T_max) * groups) {
        // the routing of this block's first item, pulled into L1 ahead of the
        // wait for y (a token past the device count only costs a prefetch)
        const size_t slot = static_cast<size_t>(blockIdx.x / groups) * k + threadIdx.x;
        prefetch_l1(inv + slot);
        prefetch_l1(w + slot);
    }
    pdl_wait();
    pdl_trigger();
    int T = T_max;
    if (d_num_tokens) {
        T = *d_num_tokens;
        T = T < 0 ? 0 : (T > T_max ? T_max : T);
    }
    const long long items = static_cast<long long>(T) * groups;
    if constexpr (sizeof(Y) == 2) {
        if (k <= 8) {
            // fp16 y, k <= 8 (the tiled paths): the next item's routing is read
            // while this item's rows are in flight, so no round trip for the
            // routing separates one item's row loads from the next item's. The
            // fp16 instance is compiled for 8 resident blocks per SM (64
            // registers, a few spilled): with 88 registers and 5 blocks it ran
            // slower than without the pipelining; with 8, in one process,
            // outputs bit-identical, `large` 99.8 vs 104.0 us, prefill 37.1 vs
            // 41.2 us.
            int nrow[8];
            float nw[8];
            auto routing = [&](long long it) {
                const size_t base = static_cast<size_t>(it / groups) * k;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const bool on = it < items && q < k;
                    nrow[q] = on ? __ldg(inv + base + q) : -1;
                    nw[q] = on ? __ldg(w + base + q) : 0.f;
                }
            };
            routing(blockIdx.x);
            for (long long item = blockIdx.x; item < items; item += gridDim.x) {
                int row[8];
                float wj[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    row[q] = nrow[q];
                    wj[q] = nw[q];
                }
                const int t = static_cast<int>(item / groups);
                const int c = static_cast<int>(item % groups) * kCombineThreads + threadIdx.x;
                const bool mine = c < vec_per_row;
                uint4 raw[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (mine && row[q] >= 0)
                        raw[q] = __ldg(reinterpret_cast<const uint4 *>(y_sorted + (static_cast<size_t>(row[q]) *
                                                                                    vec_per_row + c) * 8));
                routing(item + gridDim.x);
                if (!mine)
                    continue;
                // widened and summed in ascending j, as the loop below does
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (row[q] < 0)
                        continue;
                    const uint32_t u[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
                        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wj[q], f.x));
                        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wj[q], f.y));
                    }
                }
                uint4 o;
                o.x = pack_bf16x2(acc[0], acc[1]);
                o.y = pack_bf16x2(acc[2], acc[3]);
                o.z = pack_bf16x2(acc[4], acc[5]);
                o.w = pack_bf16x2(acc[6], acc[7]);
                out[static_cast<size_t>(t) * vec_per_row + c] = o;
            }
            return;
        }
    }
    for (long long item = blockIdx.x; item < items; item += gridDim.x) {
        const int t = static_cast<int>(item / groups);
        const int c = static_cast<int>(item % groups) * kCombineThreads + threadIdx.x;   // 8-column chunk
        if (c >= vec_per_row)
            continue;
        const int32_t *inv_t = inv + static_cast<size_t>(t) * k;
        const float *w_t = w + static_cast<size_t>(t) * k;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if constexpr (sizeof(Y) == 2) {
            // fp16 y: the loads of up to eight routed rows are issued together
            // and kept as raw 16-byte vectors (4 registers a row, where widened
            // rows would take 8), so twice the bytes are in flight for the same
            // registers; then widened and summed in ascending j as below
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 raw[8];
                int row[8];
                float wj[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    row[q] = (j0 + q < k) ? __ldg(inv_t + j0 + q) : -1;
                    wj[q] = (j0 + q < k) ? __ldg(w_t + j0 + q) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (row[q] >= 0)
                        raw[q] = __ldg(reinterpret_cast<const uint4 *>(y_sorted + (static_cast<size_t>(row[q]) *
                                                                                    vec_per_row + c) * 8));
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (row[q] < 0)
                        continue;
                    const uint32_t u[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
                        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wj[q], f.x));
                        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wj[q], f.y));
                    }
                }
            }
        } else if (kParts > 1) {
            // fp32 y in K parts (decode-size batches, where the combine's
            // latency is on the call's critical path): with k <= 8 the token's
            // routing is read once, before any row; then the K parts of four
            // routed rows are loaded together. Each row is the sum of its parts
            // in part order, then weighted and summed in ascending j.
            int rows8[8];
            float w8[8];
            const bool k8 = k <= 8;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                rows8[q] = (k8 && q < k) ? __ldg(inv_t + q) : -1;
                w8[q] = (k8 && q < k) ? __ldg(w_t + q) : 0.f;
            }
            for (int j0 = 0; j0 < k; j0 += 4) {
                float4 lo[4][kParts], hi[4][kParts];
                int row[4];
                float wj[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (k8) {
                        row[q] = j0 == 0 ? rows8[q] : rows8[4 + q];
                        wj[q] = j0 == 0 ? w8[q] : w8[4 + q];
                    } else {
                        row[q] = (j0 + q < k) ? __ldg(inv_t + j0 + q) : -1;
                        wj[q] = (j0 + q < k) ? __ldg(w_t + j0 + q) : 0.f;
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int pp = 0; pp < kParts; ++pp)
                        if (row[q] >= 0) {
                            const float4 *src = reinterpret_cast<const float4 *>(
                                y_sorted + pp * part_stride + (static_cast<size_t>(row[q]) * vec_per_row + c) * 8);
                            lo[q][pp] = __ldg(src);
                            hi[q][pp] = __ldg(src + 1);
                        }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (row[q] < 0)
                        continue;
                    float f[8] = {lo[q][0].x, lo[q][0].y, lo[q][0].z, lo[q][0].w,
                                  hi[q][0].x, hi[q][0].y, hi[q][0].z, hi[q][0].w};
#pragma unroll
                    for (int pp = 1; pp < kParts; ++pp) {
                        f[0] = __fadd_rn(f[0], lo[q][pp].x); f[1] = __fadd_rn(f[1], lo[q][pp].y);
                        f[2] = __fadd_rn(f[2], lo[q][pp].z); f[3] = __fadd_rn(f[3], lo[q][pp].w);
                        f[4] = __fadd_rn(f[4], hi[q][pp].x); f[5] = __fadd_rn(f[5], hi[q][pp].y);
                        f[6] = __fadd_rn(f[6], hi[q][pp].z); f[7] = __fadd_rn(f[7], hi[q][pp].w);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[i] = __fadd_rn(acc[i], __fmul_rn(wj[q], f[i]));
                }
            }
        } else {
            // loads of up to four routed rows are issued together, then summed in
            // ascending j, so the sum is the same sequence of roundings as a plain loop
            for (int j0 = 0; j0 < k; j0 += 4) {
                float f[4][8];
                int row[4];
                float wj[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    row[q] = (j0 + q < k) ? __ldg(inv_t + j0 + q) : -1;
                    wj[q] = (j0 + q < k) ? __ldg(w_t + j0 + q) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (row[q] >= 0)
                        load8(y_sorted, (static_cast<size_t>(row[q]) * vec_per_row + c) * 8, f[q]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (row[q] < 0)
                        continue;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[i] = __fadd_rn(acc[i], __fmul_rn(wj[q], f[q][i]));
                }
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        out[static_cast<size_t>(t) * vec_per_row + c] = o;
    }
}

// y[r, :] = ((p0 + p1) + p2) + p3 over the `parts` partial rows of a down
// GEMM that split K, for r < expert_offsets[E] (rows past it are not
// written): four columns per thread, grid-stride over rows x H/4.
__global__ void __launch_bounds__(256) reduce_parts_kernel(const float4 *__restrict__ part0, int parts,
                                                           size_t part_stride4, const int32_t *__restrict__ offsets,
                                                           int E, int vec4_per_row, int cap, float4 *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    const int n_rows = min(offsets[E], cap);
    const size_t n = static_cast<size_t>(n_rows) * vec4_per_row;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float4 a = __ldg(part0 + i);
        for (int q = 1; q < parts; ++q) {
            const float4 b = __ldg(part0 + q * part_stride4 + i);
            a.x = __fadd_rn(a.x, b.x);
            a.y = __fadd_rn(a.y, b.y);
            a.z = __fadd_rn(a.z, b.z);
            a.w = __fadd_rn(a.w, b.w);
        }
        y[i] = a;
    }
}

}  // namespace

cudaError_t launch_reduce_parts(const float *parts_base, int parts, const int32_t *expert_offsets, int E, int H,
                                int cap, float *y_sorted, int num_sms, cudaStream_t stream, bool pdl)
{
    const size_t rows_vec4 = static_cast<size_t>(cap) * (H / 4);
    long long blocks = static_cast<long long>((rows_vec4 + 255) / 256);
    blocks = blocks < num_sms * 8LL ? blocks : num_sms * 8LL;
    if (blocks < 1)
        blocks = 1;
    return launch_k(reduce_parts_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl,
                    reinterpret_cast<const float4 *>(parts_base), parts, rows_vec4, expert_offsets, E, H / 4, cap,
                    reinterpret_cast<float4 *>(y_sorted));
}

cudaError_t launch_combine(const void *y_sorted, bool y_f16, const int32_t *inv, const float *topk_weights,
                           const int32_t *d_num_tokens, int T_max, int k, int H, void *out, int num_sms,
                           cudaStream_t stream, bool pdl, int parts, size_t part_stride, bool routing_early)
{
    if (y_f16 && parts != 1)   // fp16 y comes from the tiled paths, whose down GEMM never splits K
        return cudaErrorInvalidValue;
    const long long groups = (static_cast<long long>(H) + kColsPerItem - 1) / kColsPerItem;
    const long long items = static_cast<long long>(T_max) * groups;
    int blocks = static_cast<int>(items < num_sms * 16LL ? items : num_sms * 16LL);
    if (blocks < 1)
        blocks = 1;
    if (y_f16)
        return launch_k(combine_kernel<__half, 1>, dim3(blocks), dim3(kCombineThreads), 0, stream, pdl,
                        static_cast<const __half *>(y_sorted), inv, topk_weights, d_num_tokens, T_max, k, H / 8,
                        static_cast<uint4 *>(out), size_t(0), routing_early);
    auto kern = parts == 4 ? combine_kernel<float, 4> : parts == 2 ? combine_kernel<float, 2> : combine_kernel<float, 1>;
    if (parts != 1 && parts != 2 && parts != 4)
        return cudaErrorInvalidValue;
    return launch_k(kern, dim3(blocks), dim3(kCombineThreads), 0, stream, pdl, static_cast<const float *>(y_sorted),
                    inv, topk_weights, d_num_tokens, T_max, k, H / 8, static_cast<uint4 *>(out), part_stride,
                    routing_early);
}

}  // namespace moe
