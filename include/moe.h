/*
 * moe.h -- C ABI of libmoe.so: routed Mixture-of-Experts expert execution on
 * one NVIDIA GB300 (sm_103a), BF16 weights and activations, fp32 accumulation.
 *
 * The operation is the one the TileOps page "[Refactor][MoE] Separate
 * dispatched expert compute" (PR #1738) composes in its Summary: routed
 * expert execution = local dispatch -> dispatched-expert MLP compute on a
 * tight (no-pad) expert-major batch -> combine with the routing weights.
 * Its Scope fixes BF16 tight/no-pad expert compute and leaves the rows past
 * the valid-row count unspecified; its Summary keeps valid-row counts on the
 * GPU behind a static capacity so that a whole call replays under a CUDA
 * Graph.
 *
 * Notation: T tokens (T <= T_max), E experts, k experts per token, H hidden
 * size, I intermediate size, R = T*k routed slots, slot s = t*k + j,
 * cap = capacity (rows of the sorted batch, >= T_max*k).
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument except `problem`, `bytes` and `host_code` is a
 *    DEVICE pointer on the current CUDA device, owned by the caller. The
 *    library never allocates or frees device memory and keeps no pointer
 *    after a call returns.
 *  - bf16 buffers are passed as `void*`: IEEE bfloat16, 2 bytes an element,
 *    row-major, rows contiguous. Every device buffer must be 16-byte aligned;
 *    the workspace 256-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *    only enqueue work on it: they never synchronise the host, never read a
 *    device value on the host, and are legal inside CUDA stream capture
 *    (after the first call of the host thread on a device, which sets up
 *    function attributes; make that first call outside capture).
 *  - Several host threads may call at once, each with its own workspace and
 *    its own output buffers (on one stream or several): the library keeps
 *    its launch caches per host thread and all of a call's device state in
 *    its workspace.
 *  - Host validation fails closed: a status other than MOE_OK means nothing
 *    was enqueued (DeepGEMM page "MegaMoE: add cluster-paired FP4 weight
 *    packets", Scope and fallback: unsupported shapes fail closed during host
 *    validation). MOE_ERR_CUDA means a launch failed; the stream may then
 *    hold part of the call.
 *  - Problems seen on the device (an expert id outside [0, E) other than -1,
 *    a pipeline wait that gave up) never stop a call: they set bits in a
 *    sticky error word at the start of the workspace, read with
 *    moe_last_device_error().
 *  - The path of the expert GEMMs (large-tile or M-small weight streaming)
 *    is chosen on the host from the static shape only (TileOps page, Review
 *    follow-up: one effective grouped-GEMM kernel resolved up front, no
 *    runtime row-policy branch), never from device row counts.
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULL = 1,        /* a required pointer is NULL */
    MOE_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
    MOE_ERR_ALIGN = 3,       /* H or I not a multiple of 64 (of 128 for the PACKED and MXFP8 weight
                                layouts, moe_pack_weights and moe_quantize_weights), or a misaligned
                                buffer */
    MOE_ERR_WORKSPACE = 4,   /* ws_bytes smaller than moe_workspace_size() */
    MOE_ERR_UNSUPPORTED = 5, /* no GB300-class device, or a path this build lacks */
    MOE_ERR_CUDA = 6         /* a CUDA call failed */
} moe_status_t;

/* Bits of the device error word (moe_last_device_error). */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1 /* an id outside [0, E) and not -1: slot dropped */
#define MOE_DEVERR_WAIT_TIMEOUT 0x2  /* a pipeline wait gave up: results of that call are invalid */
#define MOE_DEVERR_Y_RANGE 0x4       /* moe_forward, tiled paths: a down-GEMM output beyond the fp16
                                        range of its intermediate y was clipped to +-65504 */

/* Expert-GEMM path. AUTO picks from the static shape, a = T_max*k/E routed
 * rows per expert on average: M-small for a <= 8, single-CTA tiles for
 * 8 < a < 128, CTA-pair tiles for a >= 128 (MXFP8 weights: M-small at
 * every a). */
typedef enum moe_path {
    MOE_PATH_AUTO = 0,
    MOE_PATH_TILED = 1,       /* 256-row activation tiles x 256-row weight tiles on CTA pairs (cta_group::2) */
    MOE_PATH_SMALL_M = 2,     /* weights on the MMA M side, token tiles of 16..64 rows */
    MOE_PATH_TILED_1CTA = 3   /* 128 x 256 tiles on single CTAs */
} moe_path_t;

typedef struct moe_problem {
    int32_t T_max;    /* maximum tokens of one call, >= 1 (static) */
    int32_t E;        /* experts, 1..1024 */
    int32_t k;        /* experts per token, 1..E */
    int32_t H;        /* hidden size, multiple of 64 (of 128 for PACKED and MXFP8 weights) */
    int32_t I;        /* intermediate size, multiple of 64 (of 128 for PACKED and MXFP8 weights) */
    int32_t capacity; /* rows of the sorted batch; 0 means T_max*k; else >= T_max*k */
    int32_t path;     /* moe_path_t */
    int32_t weight_layout; /* moe_weight_layout_t of W13 and W2 */
    int32_t forward_form;  /* moe_forward_form_t */
} moe_problem_t;

/* How moe_forward launches decode-size batches (M-small path, 16-row token
 * tiles). ONE_KERNEL: dispatch, both GEMMs and the combine as one persistent
 * kernel (results bit-identical to SEPARATE); moe_forward and
 * moe_resolve_profile return MOE_ERR_UNSUPPORTED for a problem that is not
 * decode-size or whose tables do not fit that kernel's shared memory.
 * SEPARATE: dispatch, the two fused GEMMs and the combine as three kernels
 * chained by programmatic dependent launch (for a few tokens with bf16
 * weights the GEMM kernel also dispatches the slots itself, with the same
 * result, so that it need not wait for the dispatch kernel). AUTO: SEPARATE (measured at one
 * token, E=384, H=7168, I=3072, down GEMM in 4 K parts: 129.6 vs 131.5 us
 * with bf16 weights, 117.3 vs 121.8 us with MXFP8 weights). Other problems
 * ignore the field. */
typedef enum moe_forward_form {
    MOE_FORWARD_AUTO = 0,
    MOE_FORWARD_SEPARATE = 1,
    MOE_FORWARD_ONE_KERNEL = 2
} moe_forward_form_t;

/* Layout of W13 / W2 in memory.
 *  ROW_MAJOR: W13[E, 2I, H], W2[E, H, I] bf16, row-major.
 *  PACKED: the output of moe_pack_weights. Same bytes, reordered in the order
 *  the GEMMs read them (DeepGEMM page "MegaMoE: add cluster-paired FP4 weight
 *  packets", Summary and Motivation: a weight layout that follows the kernel's
 *  access order, loaded through TMA descriptors): expert -> 128-row weight
 *  tile -> 64-wide K block, each block stored as the 128-byte-swizzled
 *  shared-memory image of its 128 rows x 64 columns (16 KB), the gate and up
 *  tiles of one W13 block side by side (32 KB). Every path reads it; results
 *  are bitwise identical to ROW_MAJOR. */
typedef enum moe_weight_layout {
    MOE_WEIGHTS_ROW_MAJOR = 0,
    MOE_WEIGHTS_PACKED = 1,
    MOE_WEIGHTS_MXFP8 = 2
} moe_weight_layout_t;

/* MXFP8: the pages' MXFP8 path with prequantized expert weights (FlashInfer
 * moe_ep page, PR #3980; format 32 e4m3 x e8m0), OCP Microscaling v1.0. Each
 * 32 consecutive elements of a row along K (H for W13, I for W2) share one
 * E8M0 scale X = 2^e; each element is an FP8 E4M3 code P; the weight is X * P.
 * The output of moe_quantize_weights, one buffer per matrix:
 *   codes:  [E, 2I, H] (W13) or [E, H, I] (W2) bytes, row-major;
 *   scales: right after the codes, rows*K/32 bytes in the order the decode
 *           GEMMs read them: for each 128-row tile (rows counted over all
 *           experts), each 128-wide K block: 128 rows x 4 bytes, the scales of
 *           the row's four 32-element sub-blocks; scale code = e + 127.
 * moe_forward reads MXFP8 weights on the M-small path, which MOE_PATH_AUTO
 * takes for this layout at every batch size (token tiles of 16, 32 or 64
 * rows by a = T_max*k/E): it streams the 1-byte codes and expands X * P to
 * bf16 on the chip, exactly, then multiplies by the bf16 activations as for
 * bf16 weights. Activations, h and the output stay bf16 (SiLU(gate)*up
 * rounded to bf16 as before), so the result is the bf16 forward on the
 * dequantized weights. Each token tile of an expert expands its weight tiles
 * again, so MXFP8 weights pay off up to about a = 32 (prefill at E=384: 17-19%
 * faster than bf16 weights) and cost time beyond: a = 64 18% slower, a = 128
 * 1.75x, a = 512 2.9x. A tiled path asked for explicitly and
 * moe_expert_compute return MOE_ERR_UNSUPPORTED for this layout. Weights must
 * be finite with every block maximum in [2^-110, 2^24). */

/* Bytes of workspace every entry point below needs for `problem` (pure host
 * arithmetic, no CUDA call). The same workspace serves all entry points; it
 * holds the device error word, the GEMM kernels' counters (readiness counts
 * and the GPU-wide counts their CTAs take units from), dispatch scratch, the
 * activation h[cap, I] and, for moe_forward, the sorted batches. A new
 * workspace must be zero-filled (cudaMemset, or moe_clear_device_error)
 * before its first moe_forward or moe_expert_compute call: with stale
 * counters the GEMMs would skip units. Every call leaves its counters at zero
 * again, also after a timed-out wait (FlashInfer moe_ep page, launch-path
 * notes: workspaces allocated zeroed, counters cleaned by the kernel's tail),
 * so no per-call clearing is needed. */
moe_status_t moe_workspace_size(const moe_problem_t *problem, size_t *bytes);

/* Which expert-GEMM path `problem` resolves to (MOE_PATH_TILED,
 * MOE_PATH_SMALL_M or MOE_PATH_TILED_1CTA) and its activation-tile height
 * per CTA. Pure host. */
moe_status_t moe_resolve_path(const moe_problem_t *problem, int32_t *path, int32_t *tile_rows);

/* The full static launch profile of `problem` on the current device: every
 * choice the library makes from shapes alone (FlashInfer moe_ep page: tile,
 * schedule and token-back knobs keyed on the compile-time maximum token
 * count). Queries the current device's SM count; enqueues nothing. */
typedef struct moe_profile {
    int32_t path;          /* moe_path_t that runs (never AUTO) */
    int32_t tile_rows;     /* activation rows of one CTA's tile */
    int32_t down_split_k;  /* 1, 2 or 4: K parts of the down GEMM, in separate fp32 buffers summed in part order */
    int32_t pdl;           /* 1: kernels of a call use programmatic dependent launch */
    int32_t fused_gather;  /* 1: moe_forward's gate-up GEMM gathers rows from x (no x_sorted) */
    int32_t cta_pair;      /* 1: tiled GEMMs run on 2-CTA clusters */
    int32_t fused_mlp;     /* 1: moe_forward runs both GEMMs as one persistent kernel */
    int32_t megakernel;    /* 1: moe_forward is that one kernel, dispatch and combine included */
    int32_t kernel_launches; /* kernels one moe_forward call launches (memsets not counted) */
} moe_profile_t;

moe_status_t moe_resolve_profile(const moe_problem_t *problem, moe_profile_t *profile);

/*
 * Local dispatch: routing -> tight expert-major batch (TileOps page,
 * Summary: local dispatch; Scope: tight/no-pad batch, valid rows read from
 * expert_offsets[-1:]).
 *   topk_ids[T_max, k] int32  expert of each slot; -1 = dropped slot.
 *   d_num_tokens       int32* device scalar T (<= T_max) read on the GPU, so
 *                      a captured graph can replay with a new token count;
 *                      NULL means T = T_max.
 *   expert_offsets[E+1] int32 out: exclusive prefix sum of the per-expert
 *                      slot counts; expert_offsets[E] = valid rows.
 *   perm[cap]   int32  out: perm[row] = slot, for row < expert_offsets[E]
 *                      (later rows unspecified). Inside one expert the rows
 *                      follow ascending slot order (stable scatter).
 *   inv[T_max*k] int32 out: inv[slot] = row, -1 for a dropped slot (slots of
 *                      tokens >= T are not written).
 *   x[T_max, H], x_sorted[cap, H] bf16: optional (both NULL or both set);
 *                      when set, x_sorted[row] = x[perm[row] / k].
 * Results are bit-exact and deterministic.
 */
moe_status_t moe_dispatch(const moe_problem_t *problem, const int32_t *topk_ids,
                          const int32_t *d_num_tokens, int32_t *expert_offsets,
                          int32_t *perm, int32_t *inv, const void *x, void *x_sorted,
                          void *ws, size_t ws_bytes, void *stream);

/*
 * Dispatched-expert MLP on the tight batch (TileOps page, Summary: expert
 * compute for tight expert-major batches; Review follow-up: fused-gated
 * epilogue). For every expert e and row r in [expert_offsets[e],
 * expert_offsets[e+1]):
 *   h[r, n]  = bf16( SiLU(sum_h x_sorted[r,h] W13[e,n,h]) * sum_h x_sorted[r,h] W13[e,I+n,h] )
 *   y_sorted[r, m] = sum_n h[r,n] W2[e,m,n]                       (fp32)
 * with fp32 accumulation on the tensor cores; h lives in the workspace.
 *   x_sorted[cap, H] bf16, W13[E, 2I, H] bf16 (rows 0..I-1 gate, I..2I-1 up),
 *   W2[E, H, I] bf16, y_sorted[cap, H] fp32 out (rows past the valid count
 *   are not written), expert_offsets[E+1] as produced by moe_dispatch.
 * y_sorted stays fp32 so that the combine rounds to bf16 once, at the end.
 * ws: a zero-filled workspace (see moe_workspace_size), left with its
 * counters at zero.
 */
moe_status_t moe_expert_compute(const moe_problem_t *problem, const void *x_sorted,
                                const int32_t *expert_offsets, const void *W13, const void *W2,
                                float *y_sorted, void *ws, size_t ws_bytes, void *stream);

/*
 * Combine (TileOps page, Summary: routing weights kept outside expert
 * compute): out[t, m] = bf16( sum_{j=0..k-1} w[t,j] * y_sorted[inv[t*k+j], m] ),
 * fp32, j ascending, dropped slots (inv = -1) skipped; deterministic.
 *   topk_weights[T_max, k] fp32, inv[T_max*k] int32, y_sorted[cap, H] fp32,
 *   out[T_max, H] bf16 (rows >= T untouched), d_num_tokens as above.
 */
moe_status_t moe_combine(const moe_problem_t *problem, const float *y_sorted, const int32_t *inv,
                         const float *topk_weights, const int32_t *d_num_tokens, void *out,
                         void *stream);

/*
 * The whole routed expert execution in one call: dispatch (with the row
 * gather) -> expert compute -> combine, all on `stream`, with the sorted
 * batches and inv held in the workspace. Arguments as above; perm and
 * expert_offsets are still returned to the caller. On the tiled paths
 * (prefill- and large-batch shapes) the intermediate y between the down GEMM
 * and the combine is kept in fp16 (round to nearest, saturating at +-65504:
 * a clipped value sets MOE_DEVERR_Y_RANGE), which halves its HBM traffic;
 * the separate moe_expert_compute / moe_combine keep y in fp32. Decode-size
 * batches keep y in fp32. For decode-size batches
 * (moe_profile_t.megakernel) the call is a single persistent kernel: every
 * CTA dispatches the call's slots itself, then runs its share of both GEMMs
 * and of the combine; its CTAs wait on one another (bounded), so it expects
 * the GPU's SMs free for its CTAs, one per SM, when it starts. Results equal
 * those of the separate entry points bit for bit.
 */
moe_status_t moe_forward(const moe_problem_t *problem, const void *x, const int32_t *topk_ids,
                         const float *topk_weights, const int32_t *d_num_tokens, const void *W13,
                         const void *W2, int32_t *expert_offsets, int32_t *perm, void *out,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * moe_forward with stage timestamps: identical work, plus a cudaEventRecord of
 * stage_events[i] (cudaEvent_t, created by the caller with timing enabled)
 * at the 6 stage boundaries on `stream`: [0] before dispatch, [1] after the
 * dispatch kernels, [2] after the row gather, [3] after the gate-up GEMM,
 * [4] after the down GEMM, [5] after combine. Inside stream capture the
 * records become external event nodes of the graph (cudaEventRecordExternal),
 * so a replayed graph still reports per-stage times. No counterpart on the
 * pages: it exists to time each kernel from the host without a profiler.
 */
moe_status_t moe_forward_profiled(const moe_problem_t *problem, const void *x, const int32_t *topk_ids,
                                  const float *topk_weights, const int32_t *d_num_tokens, const void *W13,
                                  const void *W2, int32_t *expert_offsets, int32_t *perm, void *out,
                                  void *ws, size_t ws_bytes, void *stream, void *const *stage_events);

/*
 * moe_dispatch for callers that cannot allocate device memory. No counterpart
 * on the pages: some callers have no way to hand the library a workspace --
 * a runtime whose device memory is planned once at start-up and may not grow,
 * or code that runs under stream capture, where cudaMalloc is not allowed.
 * This variant takes no workspace: its per-block counts live in a static
 * device array of MOE_NOALLOC_SCRATCH_INTS int32 (1 MiB) inside libmoe.so,
 * which every GPU that loads the library keeps until the process exits.
 * Inputs and outputs are the caller's, exactly as in moe_dispatch, and the
 * results are identical to moe_dispatch's. Differences:
 *  - Returns MOE_ERR_WORKSPACE, before touching the device, when the problem
 *    needs more than the static array: 64 + 2 * ceil(T_max*k / 1024) * E ints.
 *  - The first call on a device looks up the array's device address with
 *    that device current, and looks it up again when the device's current
 *    context has changed since (cudaDeviceReset, a new primary context);
 *    make the first call in each context before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents
 *    (each call rewrites what it reads). Calls that overlap on the GPU --
 *    different streams without ordering between them -- race on it: order
 *    them on one stream.
 *  - An invalid expert id is dropped as in moe_dispatch, but its error bit
 *    goes to the static array and is not reported.
 * It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define MOE_NOALLOC_SCRATCH_INTS 262144
moe_status_t moe_dispatch_noalloc(const moe_problem_t *problem, const int32_t *topk_ids,
                                  const int32_t *d_num_tokens, int32_t *expert_offsets,
                                  int32_t *perm, int32_t *inv, const void *x, void *x_sorted,
                                  void *stream);

/*
 * Reorder W13 and W2 (row-major) into the PACKED layout, once, at model load.
 * W13_packed and W2_packed have the sizes of W13 and W2 and must not overlap
 * them. Only problem->E, H and I matter. Enqueued on `stream`.
 */
moe_status_t moe_pack_weights(const moe_problem_t *problem, const void *W13, const void *W2, void *W13_packed,
                              void *W2_packed, void *stream);

/* Bytes of W13 and W2 in `layout` (ROW_MAJOR and PACKED: 2 per element;
 * MXFP8: 1 per element plus one scale byte per 32). Pure host. */
moe_status_t moe_weight_bytes(const moe_problem_t *problem, int32_t layout, size_t *w13_bytes,
                              size_t *w2_bytes);

/* Quantize W13 and W2 (row-major bf16) to the MXFP8 layout, once, at model
 * load. W13_mx and W2_mx have moe_weight_bytes(MXFP8) bytes and must not
 * overlap the sources. Only problem->E, H and I matter. Enqueued on `stream`.
 * Bit-exact with the OCP MX definition above (round to nearest even,
 * saturation at 448). */
moe_status_t moe_quantize_weights(const moe_problem_t *problem, const void *W13, const void *W2,
                                  void *W13_mx, void *W2_mx, void *stream);

/* Read the sticky device error word of `ws` into *host_code (0 = none).
 * Synchronises `stream` (the only entry point that does). */
moe_status_t moe_last_device_error(const void *ws, void *stream, int32_t *host_code);

/* Clear the device error word and the GEMM kernels' counters (enqueued on
 * `stream`); also readies a workspace of unknown contents for moe_forward
 * and moe_expert_compute. */
moe_status_t moe_clear_device_error(void *ws, void *stream);

/* Human-readable name of a status. Never NULL. */
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H */
