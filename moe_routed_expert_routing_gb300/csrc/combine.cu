// combine.cu -- routing-weighted top-k sum back into token order.
//
// TileOps PR #1738 "Separate dispatched expert compute", Summary: routed
// expert execution ends with a combine, and the routing weights stay outside
// expert compute. The FlashInfer moe_ep page (kernel API migration) likewise
// reduces the top-k contributions into one (T, hidden) output.
//
//   out[t, m] = bf16( sum_{j = 0..k-1} w[t, j] * y_sorted[inv[t*k + j], m] )
//
// y_sorted is the fp32 output of the down GEMM. fp32 products and sums in
// ascending j (no fused multiply-add), one rounding at the end: the result
// is deterministic (no atomics) and identical to a plain sequential loop.
// Work item = one token x 1024 columns, so even a single token spreads over
// several SMs; each thread owns 8 consecutive columns, read as two 16-byte
// loads per routed row and written as one 16-byte store.
#include <cuda_bf16.h>

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

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float4 *__restrict__ y_sorted,
                                                                  const int32_t *__restrict__ inv,
                                                                  const float *__restrict__ w,
                                                                  const int32_t *d_num_tokens, int T_max, int k,
                                                                  int vec_per_row, uint4 *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    int T = T_max;
    if (d_num_tokens) {
        T = *d_num_tokens;
        T = T < 0 ? 0 : (T > T_max ? T_max : T);
    }
    const int groups = (vec_per_row * 8 + kColsPerItem - 1) / kColsPerItem;
    const long long items = static_cast<long long>(T) * groups;
    for (long long item = blockIdx.x; item < items; item += gridDim.x) {
        const int t = static_cast<int>(item / groups);
        const int c = static_cast<int>(item % groups) * kCombineThreads + threadIdx.x;   // 8-column chunk
        if (c >= vec_per_row)
            continue;
        const int32_t *inv_t = inv + static_cast<size_t>(t) * k;
        const float *w_t = w + static_cast<size_t>(t) * k;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // loads of up to four routed rows are issued together, then summed in
        // ascending j, so the sum is the same sequence of roundings as a plain loop
        for (int j0 = 0; j0 < k; j0 += 4) {
            float4 a[4], b[4];
            int row[4];
            float wj[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                row[q] = (j0 + q < k) ? __ldg(inv_t + j0 + q) : -1;
                wj[q] = (j0 + q < k) ? __ldg(w_t + j0 + q) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (row[q] >= 0) {
                    const float4 *src = y_sorted + (static_cast<size_t>(row[q]) * vec_per_row + c) * 2;
                    a[q] = __ldg(src);
                    b[q] = __ldg(src + 1);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (row[q] < 0)
                    continue;
                const float f[8] = {a[q].x, a[q].y, a[q].z, a[q].w, b[q].x, b[q].y, b[q].z, b[q].w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = __fadd_rn(acc[i], __fmul_rn(wj[q], f[i]));
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

}  // namespace

cudaError_t launch_combine(const float *y_sorted, const int32_t *inv, const float *topk_weights,
                           const int32_t *d_num_tokens, int T_max, int k, int H, void *out, int num_sms,
                           cudaStream_t stream, bool pdl)
{
    const long long groups = (static_cast<long long>(H) + kColsPerItem - 1) / kColsPerItem;
    const long long items = static_cast<long long>(T_max) * groups;
    int blocks = static_cast<int>(items < num_sms * 16LL ? items : num_sms * 16LL);
    if (blocks < 1)
        blocks = 1;
    return launch_k(combine_kernel, dim3(blocks), dim3(kCombineThreads), 0, stream, pdl,
                    reinterpret_cast<const float4 *>(y_sorted), inv, topk_weights, d_num_tokens, T_max, k, H / 8,
                    static_cast<uint4 *>(out));
}

}  // namespace moe
