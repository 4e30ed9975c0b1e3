// weights_pack.cu -- reorder row-major W13 / W2 into the access-ordered
// PACKED layout (include/moe.h), once, at model load.
//
// DeepGEMM PR #394 "MegaMoE: add cluster-paired FP4 weight packets",
// Summary / Motivation: store each routed expert's weight tile in the order
// the kernel reads it, so that the tiles a CTA streams are adjacent in
// memory. Here, without FP4 or scales: every (expert, 128-row weight tile,
// 64-wide K block) becomes the 16 KB image that a 128-byte-swizzled TMA load
// would leave in shared memory (line r = weight row r of the tile, its 16-byte
// chunk j = source chunk j ^ (r mod 8)), ordered expert -> tile -> K block; in
// W13 the gate tile and the matching up tile of a block sit side by side.
// The GEMMs then move each 16 KB image with an unswizzled TMA box.
#include "moe_internal.h"

namespace moe {

namespace {

// Destination index q runs over 16-byte chunks of the packed buffer in order.
__global__ void pack_w13_kernel(const uint4 *__restrict__ W13, uint4 *__restrict__ out, int E, int H, int I)
{
    const int KB = H / 64, NT = I / 128, row_chunks = H / 8;
    const long long total = static_cast<long long>(E) * 2 * I * row_chunks;
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < total;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(q & 7);
        const int line = static_cast<int>((q >> 3) % 256);          // 0..127 gate, 128..255 up
        const long long packet = (q >> 3) / 256;                    // (e, nt, kb)
        const int kb = static_cast<int>(packet % KB);
        const int nt = static_cast<int>((packet / KB) % NT);
        const int e = static_cast<int>(packet / (static_cast<long long>(KB) * NT));
        const int half = line >> 7, r = line & 127;
        const long long src_row = static_cast<long long>(e) * 2 * I + static_cast<long long>(half) * I + nt * 128 + r;
        out[q] = W13[src_row * row_chunks + kb * 8 + (j ^ (r & 7))];
    }
}

__global__ void pack_w2_kernel(const uint4 *__restrict__ W2, uint4 *__restrict__ out, int E, int H, int I)
{
    const int KB = I / 64, row_chunks = I / 8;
    const long long total = static_cast<long long>(E) * H * row_chunks;
    for (long long q = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; q < total;
         q += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(q & 7);
        const int r = static_cast<int>((q >> 3) & 127);
        const long long packet = (q >> 3) >> 7;                     // (e, nt, kb)
        const int kb = static_cast<int>(packet % KB);
        const long long tile = packet / KB;                         // e * NT + nt
        const long long src_row = tile * 128 + r;
        out[q] = W2[src_row * row_chunks + kb * 8 + (j ^ (r & 7))];
    }
}

}  // namespace

cudaError_t launch_pack_weights(const void *W13, const void *W2, void *W13_packed, void *W2_packed, int E, int H,
                                int I, int num_sms, cudaStream_t stream)
{
    const int blocks = num_sms * 8;
    pack_w13_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(W13), static_cast<uint4 *>(W13_packed), E,
                                                H, I);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    pack_w2_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(W2), static_cast<uint4 *>(W2_packed), E, H,
                                               I);
    return cudaGetLastError();
}

}  // namespace moe
