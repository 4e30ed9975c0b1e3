// weights_mx.cu -- MXFP8 quantization of the expert weights, once, at model load.
//
// The pages' MXFP8 path keeps its routed expert weights prequantized
// (FlashInfer moe_ep page, PR #3980: MXFP8 mega MoE, prequantized weight
// packs; its quantized combine wire names the format: 32 e4m3 x e8m0). The
// format is OCP Microscaling (MX) v1.0: every 32 consecutive elements of a
// row along K share one E8M0 scale X = 2^e, each element an FP8 E4M3 code.
// Per block: e = floor(log2(max |V|)) - 8 (8: exponent of E4M3's largest
// normal, 448), clamped to [-127, 127]; P = E4M3(V * 2^-e), rounded to
// nearest even and saturated at 448 (cvt.rn.satfinite). A block of zeros gets
// e = -127.
//
// Output layout (MOE_WEIGHTS_MXFP8 in include/moe.h): the E4M3 codes,
// row-major like the bf16 source, then the scale codes in the order the
// decode GEMMs read them: for each 128-row tile and 128-wide K block, 512
// bytes, 4 per row (the scales of its four 32-element sub-blocks).
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kQuantThreads = 256;

// floor(log2(a)) - 8 for the block maximum a (fp32 bits), clamped to E8M0's range.
__device__ __forceinline__ int block_exponent(float amax)
{
    const int field = (__float_as_int(amax) >> 23) & 0xff;
    if (field == 0)   // zero or an fp32 subnormal: below 2^-126, so e < -127
        return -127;
    const int e = field - 127 - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two fp32 -> two E4M3 codes, round to nearest even, saturated to +-448;
// lo lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// One thread per 32-element block of one row. rows = all rows of the matrix
// (E * rows per expert, a multiple of 128), K a multiple of 128.
__global__ void __launch_bounds__(kQuantThreads) mx_quantize_kernel(const uint4 *__restrict__ w, long long rows, int K,
                                                                    uint4 *__restrict__ q, uint8_t *__restrict__ sc)
{
    const int nb = K / 32;
    const long long blocks = rows * nb;
    for (long long i = blockIdx.x * static_cast<long long>(kQuantThreads) + threadIdx.x; i < blocks;
         i += static_cast<long long>(gridDim.x) * kQuantThreads) {
        const long long r = i / nb;
        const int b = static_cast<int>(i - r * nb);
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = __ldg(w + i * 4 + j);
        float f[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                f[8 * j + 2 * h] = __uint_as_float(u[h] << 16);
                f[8 * j + 2 * h + 1] = __uint_as_float(u[h] & 0xffff0000u);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            amax = fmaxf(amax, fabsf(f[j]));
        const int e = block_exponent(amax);
        const float inv = __int_as_float((127 - e) << 23);   // 2^-e, a normal float for e in [-127, 119]
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t lo = e4m3x2(f[4 * j] * inv, f[4 * j + 1] * inv);
            const uint32_t hi = e4m3x2(f[4 * j + 2] * inv, f[4 * j + 3] * inv);
            o[j] = lo | (hi << 16);
        }
        q[i * 2] = make_uint4(o[0], o[1], o[2], o[3]);
        q[i * 2 + 1] = make_uint4(o[4], o[5], o[6], o[7]);
        // tiled scale position: (128-row tile, 128-wide K block) -> row -> sub-block
        const long long tile = r / 128;
        const int kb = b / 4;
        sc[((tile * (K / 128) + kb) * 128 + (r % 128)) * 4 + (b % 4)] = static_cast<uint8_t>(e + 127);
    }
}

cudaError_t quantize_matrix(const void *w, long long rows, int K, void *out, int num_sms, cudaStream_t stream)
{
    const long long blocks = rows * (K / 32);
    long long grid = (blocks + kQuantThreads - 1) / kQuantThreads;
    if (grid > num_sms * 32LL)
        grid = num_sms * 32LL;
    if (grid < 1)
        grid = 1;
    uint8_t *q = static_cast<uint8_t *>(out);
    uint8_t *sc = q + rows * K;
    return launch_k(mx_quantize_kernel, dim3(static_cast<unsigned>(grid)), dim3(kQuantThreads), 0, stream, false,
                    static_cast<const uint4 *>(w), rows, K, reinterpret_cast<uint4 *>(q), sc);
}

}  // namespace

cudaError_t launch_quantize_weights_mxfp8(const void *W13, const void *W2, void *W13_mx, void *W2_mx, int E, int H,
                                          int I, int num_sms, cudaStream_t stream)
{
    cudaError_t e = quantize_matrix(W13, 2LL * E * I, H, W13_mx, num_sms, stream);
    if (e != cudaSuccess)
        return e;
    return quantize_matrix(W2, static_cast<long long>(E) * H, I, W2_mx, num_sms, stream);
}

}  // namespace moe
