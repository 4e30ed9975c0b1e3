// dispatch_noalloc.cu -- moe_dispatch_noalloc: local dispatch with no
// caller workspace, for callers that cannot allocate device memory (a
// runtime whose device memory is fixed at start-up, or code running under
// stream capture, where cudaMalloc is illegal).
//
// The per-block slot counts and row bases that moe_dispatch keeps in the
// caller's workspace live here in one file-scope device array instead. Host
// code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the address is looked up once per device
// with cudaGetSymbolAddress, with that device current, and handed to the
// same kernels moe_dispatch launches. The address is kept with the CUDA
// context it was looked up in and looked up again when the device's current
// context is another one (after cudaDeviceReset, say).
#include <mutex>

#include "moe_internal.h"

namespace {

static __device__ __align__(256) int32_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_INTS];

constexpr int kErrWordInts = 64;   // error word, padded to 256 bytes
constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
int32_t *g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the
// library links the runtime only).
CtxGetCurrentFn ctx_get_current_fn()
{
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    return fn;
}

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call in each CUDA context of that device.
moe_status_t scratch_for_current_device(int32_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MOE_ERR_CUDA;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (!get_ctx)
        return MOE_ERR_CUDA;
    // no context yet on this thread: the symbol lookup below sets up the
    // device's primary context, which is then read again
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS)
        return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return MOE_ERR_CUDA;
        if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
            return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_dispatch_noalloc(const moe_problem_t *problem, const int32_t *topk_ids,
                                             const int32_t *d_num_tokens, int32_t *expert_offsets, int32_t *perm,
                                             int32_t *inv, const void *x, void *x_sorted, void *stream)
{
    moe_status_t st = moe::validate_problem(problem);
    if (st != MOE_OK)
        return st;
    const moe_problem_t &p = *problem;
    if (!topk_ids || !expert_offsets || !perm || !inv)
        return MOE_ERR_NULL;
    if ((x == nullptr) != (x_sorted == nullptr))
        return MOE_ERR_NULL;
    if (x && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x_sorted)) & 15u))
        return MOE_ERR_ALIGN;
    const long long n_blocks = moe::dispatch_blocks(p);
    const long long need = kErrWordInts + 2 * n_blocks * p.E;
    if (need > MOE_NOALLOC_SCRATCH_INTS)
        return MOE_ERR_WORKSPACE;
    if ((st = moe::validate_device()) != MOE_OK)
        return st;
    int32_t *scratch = nullptr;
    if ((st = scratch_for_current_device(&scratch)) != MOE_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *err = scratch;
    int32_t *block_counts = scratch + kErrWordInts;
    int32_t *block_base = block_counts + n_blocks * p.E;
    // the error word is the only state that must start from zero; counts and
    // bases are fully rewritten by every call before they are read
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (moe::launch_dispatch(topk_ids, d_num_tokens, p.T_max, p.k, p.E, block_counts, block_base, expert_offsets,
                             perm, inv, err, s, moe::use_pdl(p)) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (!x)
        return MOE_OK;
    if (moe::launch_gather_rows(x, perm, expert_offsets, p.E, p.k, p.H, moe::capacity_of(p), x_sorted,
                                moe::device_sm_count(), s, moe::use_pdl(p)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
