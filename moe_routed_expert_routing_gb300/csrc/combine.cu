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
// One block per token (grid-stride); each thread owns 8 consecutive columns,
// read as two 16-byte loads per routed row and written as one 16-byte store;
// the k row indices and weights of the token sit in shared memory.
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {

namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

__global__ void __launch_bounds__(128) combine_kernel(const float4 *__restrict__ y_sorted,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ w, const int32_t *d_num_tokens,
                                                      int T_max, int k, int vec_per_row, uint4 *__restrict__ out)
{
    __shared__ int s_row[kMaxTopK];
    __shared__ float s_w[kMaxTopK];
    int T = T_max;
    if (d_num_tokens) {
        T = *d_num_tokens;
        T = T < 0 ? 0 : (T > T_max ? T_max : T);
    }
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();
        for (int j = threadIdx.x; j < k; j += blockDim.x) {
            s_row[j] = inv[static_cast<size_t>(t) * k + j];
            s_w[j] = w[static_cast<size_t>(t) * k + j];
        }
        __syncthreads();
        for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < k; ++j) {
                const int row = s_row[j];
                if (row < 0)
                    continue;
                const float4 *src = y_sorted + (static_cast<size_t>(row) * vec_per_row + c) * 2;
                const float4 a = __ldg(src), b = __ldg(src + 1);
                const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                const float wj = s_w[j];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i] = __fadd_rn(acc[i], __fmul_rn(wj, f[i]));
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            out[static_cast<size_t>(t) * vec_per_row + c] = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const float *y_sorted, const int32_t *inv, const float *topk_weights,
                           const int32_t *d_num_tokens, int T_max, int k, int H, void *out, int num_sms,
                           cudaStream_t stream)
{
    int blocks = T_max < num_sms * 16 ? T_max : num_sms * 16;
    if (blocks < 1)
        blocks = 1;
    combine_kernel<<<blocks, 128, 0, stream>>>(reinterpret_cast<const float4 *>(y_sorted), inv, topk_weights,
                                               d_num_tokens, T_max, k, H / 8, static_cast<uint4 *>(out));
    return cudaGetLastError();
}

}  // namespace moe
