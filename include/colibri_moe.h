/*
 * colibri_moe.h - C ABI of a GB300 (sm_103a) Mixture-of-Experts layer forward.
 *
 * One MoE layer:  router logits -> per-token top-k -> softmax over the k
 * selected logits -> dispatch (pairs grouped by expert) -> per-expert SwiGLU
 * FFN -> gate-weighted combine back into token order.
 *
 * The call shape (init / forward / free, status codes, caller-owned buffers)
 * follows the engine the source pages describe: pnsm.cn section 4.4
 * (colibri_init / colibri_forward / colibri_free), zskr.cn
 * "Colibri：面向MoE架构的C语言高效推理引擎解析" section 4.2 (caller-owned input
 * and output buffers, COLIBRI_ERR_INVALID_ARG), and pnsm.cn section 5.1
 * (init that fails returns no handle).
 *
 * Conventions for every entry point:
 *  - All pointers are plain addresses; nothing here is a framework type.
 *  - "device" pointers are CUDA device (or managed) memory on the handle's
 *    device; "host" pointers are ordinary host memory (pinned is faster).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device work is ordered on it; unless stated, a call returns
 *    without waiting for the device.
 *  - A handle is not thread-safe: use one handle per concurrently running
 *    stream.  Two forwards on one handle must be stream-ordered.
 *  - Every call returns a colibri_status_t; argument checks run on the host
 *    before any CUDA call, so an INVALID_ARG call has no side effect.
 */
#ifndef COLIBRI_MOE_H
#define COLIBRI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    COLIBRI_OK = 0,
    COLIBRI_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, misalignment, aliasing */
    COLIBRI_ERR_OOM = 2,          /* a device or pinned-host allocation failed (init only) */
    COLIBRI_ERR_CUDA = 3,         /* a CUDA runtime/launch error; the stream may hold garbage */
    COLIBRI_ERR_UNSUPPORTED = 4,  /* not an sm_103 device, or a shape this build cannot run */
    COLIBRI_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (see colibri_check) */
} colibri_status_t;

typedef enum {
    COLIBRI_DTYPE_FP32 = 0,       /* activations and weights float32, float32 arithmetic */
    COLIBRI_DTYPE_BF16 = 1        /* activations and weights bfloat16, float32 accumulation */
} colibri_dtype_t;

typedef enum {
    COLIBRI_EXEC_AUTO = 0,        /* choose from T and the shapes */
    COLIBRI_EXEC_STREAM = 1,      /* weight-streaming expert FFN on CUDA cores (decode sizes, fp32, int8) */
    COLIBRI_EXEC_GROUPED = 2      /* tcgen05 grouped GEMM expert FFN (bf16 only) */
} colibri_executor_t;

/* Layer shape.  d_model % 64 == 0, d_model <= 57856 (one token row of the
 * CUDA-core router in shared memory) and d_ff % 128 == 0 are required
 * (UNSUPPORTED otherwise); 1 <= top_k <= n_experts <= 256; top_k <= 8, or
 * top_k == n_experts.
 * top_k == n_experts selects soft routing (m.nxbn.cn section 2.2: a Soft MoE
 * router weights and fuses every expert's output instead of hard-selecting
 * k): every token goes to every expert, pair j of a token is expert j, and
 * the gate is the softmax over all E logits.  Otherwise routing is top-k. */
typedef struct {
    int32_t n_experts;   /* E */
    int32_t top_k;       /* k */
    int32_t d_model;     /* d */
    int32_t d_ff;        /* f, expert hidden size */
    int32_t max_tokens;  /* largest T any later call may pass; sizes the workspace */
    int32_t dtype;       /* colibri_dtype_t */
    int32_t device;      /* CUDA device ordinal */
    int32_t executor;    /* colibri_executor_t (can be changed with colibri_set_executor) */
} colibri_moe_config_t;

typedef struct colibri_moe colibri_moe_t;  /* opaque */

/*
 * colibri_init - build a layer handle: validate, copy and repack the weights
 * into the device layout, and allocate the whole workspace for max_tokens.
 *
 * Defines the layer of zskr.cn section 3.1/3.3 (router W_r, per-expert
 * gate_proj / up_proj / down_proj) in the row-major layouts:
 *   w_router     [d_model, E]           dtype
 *   router_bias  [E] float32 or NULL    added to the logits before top-k and
 *                                       softmax; -INFINITY masks an expert.
 *                                       Not a learned bias: a per-expert
 *                                       offset (e.g. a load skew or a mask).
 *   w_gate/w_up  [E, d_model, d_ff]     dtype  (x . W_gate[e] -> [T, d_ff])
 *   w_down       [E, d_ff, d_model]     dtype
 * weights_on_device: 0 = the five pointers are host memory, 1 = device.
 * The caller keeps ownership of its arrays and may free them once init
 * returns (init synchronises the device before returning).
 * On any failure *out is set to NULL and everything allocated is freed.
 */
colibri_status_t colibri_init(const colibri_moe_config_t* cfg,
                              const void* w_router, const float* router_bias,
                              const void* w_gate, const void* w_up, const void* w_down,
                              int weights_on_device, colibri_moe_t** out);

/*
 * Weight-only int8 expert weights (m.nxbn.cn section 3.1: every expert
 * matrix cut into 64x64 blocks, each quantised from its own min and max into
 * an int8 weight buffer and a scale buffer, dequantised inside the GEMM;
 * pnsm.cn section 3.1: min-max to [-127, 127], converted on the CPU; pnsm.cn
 * section 5.2: w = (q - zp) * scale with an int32 zero point).
 *
 * Per 64x64 block b of a matrix (rows and columns multiples of 64):
 *   lo = min(min(b), 0), hi = max(max(b), 0)
 *   scale = float32((hi - lo) / 254)           (1 for a block of zeros)
 *   zp    = round(-127 - lo / scale)           in [-127, 127]
 *   q     = clamp(round(w / scale) + zp, -127, 127)
 * with round = nearest, ties to even, evaluated in double precision from the
 * float32 scale.  Dequantised weight: (q - zp) * scale, within scale / 2 of w.
 */
typedef struct {
    const int8_t* q;       /* [E, R, C] codes, in the float weight's layout */
    const float* scale;    /* [E, R/64, C/64] */
    const int32_t* zp;     /* [E, R/64, C/64] */
} colibri_int8_weights_t;

/*
 * colibri_quantize_int8_block64 - the converter: quantise one row-major
 * [rows, cols] matrix (host memory, dtype FP32 or BF16) block by block as
 * above into caller-owned host arrays q [rows, cols], scale and zp
 * [rows/64, cols/64].  Runs on the calling CPU thread; no device work.
 * INVALID_ARG for NULL pointers, rows or cols not positive multiples of 64,
 * or a non-finite weight.
 */
colibri_status_t colibri_quantize_int8_block64(const void* w, int32_t dtype, int32_t rows,
                                               int32_t cols, int8_t* q, float* scale,
                                               int32_t* zp);

/*
 * colibri_init_int8 - a layer handle whose expert weights are int8 blocks:
 *   w_gate, w_up  R = d_model, C = d_ff   (as colibri_init's [E, d_model, d_ff])
 *   w_down        R = d_ff,    C = d_model
 * w_router / router_bias / cfg as in colibri_init (cfg->dtype is the
 * activation and router type).  Executors: GROUPED (bf16 activations)
 * streams the int8 codes into shared memory with TMA, converter warps
 * dequantise them (to f16) and the tcgen05 MMAs read them; STREAM runs on
 * CUDA cores: for bf16 batches of at most three tokens the codes stream
 * through shared memory by bulk copies and multiply 16-bit integer
 * activations (one per 64-wide block, scaled by a power of two) with integer
 * dot products, otherwise each row's codes are dequantised in registers (the
 * only executor for fp32 activations).  AUTO picks STREAM for bf16 batches
 * of at most three tokens whose gate/up stage has at least one 64-unit item
 * per SM (top_k * d_ff / 64 >= SMs), GROUPED otherwise.  weights_on_device
 * applies to every array.
 */
colibri_status_t colibri_init_int8(const colibri_moe_config_t* cfg,
                                   const void* w_router, const float* router_bias,
                                   const colibri_int8_weights_t* w_gate,
                                   const colibri_int8_weights_t* w_up,
                                   const colibri_int8_weights_t* w_down,
                                   int weights_on_device, colibri_moe_t** out);

/*
 * colibri_forward - y = MoE(x) for T tokens (zskr.cn section 3.3 stages 2-5).
 *   x  [T, d_model] device, dtype, 16-byte aligned, read only
 *   y  [T, d_model] device, dtype, 16-byte aligned, written; must not overlap x
 *   0 <= T <= max_tokens; T == 0 is a no-op.
 * Allocates nothing and does not synchronise the host.  Routing results of
 * the last forward stay in the workspace until the next call (see
 * colibri_get_routing).
 */
colibri_status_t colibri_forward(colibri_moe_t* h, const void* x, int32_t T, void* y,
                                 void* stream);

/*
 * colibri_forward_host - the same layer on host buffers: copies x to the
 * device, runs colibri_forward, copies y back and waits until y_host holds
 * the result.
 *   x_host, y_host [T, d_model] host memory (pinned recommended), dtype.
 * Uses the workspace's own device copies of x and y (no allocation).
 */
colibri_status_t colibri_forward_host(colibri_moe_t* h, const void* x_host, int32_t T,
                                      void* y_host, void* stream);

/*
 * colibri_forward_host_async - colibri_forward_host without the wait, for
 * pipelining a sequence of batches: the upload of x and the download of y run
 * on two copy streams of the handle, and successive calls alternate between
 * two staging slots, so that one call's upload and the previous call's
 * download overlap the layer of another.  The layer itself runs on `stream`
 * after the upload; every call on one handle must pass the same stream.
 * x_host must stay unchanged and y_host must not be read until
 * colibri_host_wait returns.  With pageable host memory the copies are not
 * asynchronous (pin both buffers).  Returns an error without waiting.
 */
colibri_status_t colibri_forward_host_async(colibri_moe_t* h, const void* x_host, int32_t T,
                                            void* y_host, void* stream);

/*
 * colibri_host_wait - wait until every colibri_forward_host_async call on the
 * handle has finished and written its y_host.
 */
colibri_status_t colibri_host_wait(colibri_moe_t* h);

/*
 * colibri_forward_stack_layer - one layer of a pre-norm decode stack
 * (pnsm.cn section 2.2: residual around the MoE block):
 *   u = bf16(RMSNorm(hidden) * gamma),  hidden <- bf16(hidden + MoE(u))
 * RMSNorm(h) = h / sqrt(mean(h^2) + eps), in float32; the residual sum is
 * formed in float32 from the float32 combine result and rounded once.
 *   hidden [T, d_model] device, dtype, updated in place
 *   gamma  [d_model] device, dtype
 * Requires dtype BF16 or FP32 matching the handle; allocates nothing.
 */
colibri_status_t colibri_forward_stack_layer(colibri_moe_t* h, void* hidden, int32_t T,
                                             const void* gamma, float eps, void* stream);

/*
 * colibri_get_routing - copy the last forward's routing decisions out
 * (zskr.cn section 3.3 stage 2 outputs, and the stage 3 grouping):
 *   topk_idx [T, k] int32   expert ids, descending logit, ties -> lower id
 *   topk_w   [T, k] float32 softmax over the k selected logits
 *   counts   [E]    int32   pairs per expert
 *   perm     [T*k]  int32   perm[p] = t*k + j of the p-th pair in expert order
 * All device pointers; any may be NULL to skip it.  Stream-ordered after the
 * forward on the same stream.  T is the last forward's T.
 */
colibri_status_t colibri_get_routing(colibri_moe_t* h, int32_t* topk_idx, float* topk_w,
                                     int32_t* counts, int32_t* perm, void* stream);

/*
 * colibri_set_capacity - hard expert capacity for later forwards (cf-1.com
 * section 2.3: an expert's capacity is the most tokens it handles in one
 * batch; section 4.2: --expert-capacity is a hard limit and tokens past it are
 * dropped; zskr.cn section 2.2: hard_capacity).  Each expert accepts at most
 * `capacity` (token, slot) pairs, in token order and then slot order; a
 * dropped pair adds nothing to its token's output and the token's other gates
 * are left unchanged.  capacity < 0 (the default) removes the limit; 0 drops
 * every pair (y = 0, or y = hidden for the residual layer).
 * colibri_get_routing still reports every routed pair: counts are before the
 * limit, and expert e kept perm[offsets[e] .. offsets[e] + min(counts[e],
 * capacity)) with offsets the exclusive prefix sum of counts.
 */
colibri_status_t colibri_set_capacity(colibri_moe_t* h, int32_t capacity);

/* colibri_set_executor - choose the expert executor for later forwards.
 * GROUPED needs dtype BF16 (UNSUPPORTED otherwise). */
colibri_status_t colibri_set_executor(colibri_moe_t* h, int32_t executor);

/*
 * colibri_check - wait for `stream`, then report the first failure of any
 * earlier call on this handle: COLIBRI_ERR_CUDA for a CUDA error,
 * COLIBRI_ERR_TIMEOUT when a bounded device-side wait (an mbarrier wait in the
 * grouped GEMM) gave up.  Clears the recorded device status.
 */
colibri_status_t colibri_check(colibri_moe_t* h, void* stream);

/* colibri_launch_count - kernels this handle has launched since init
 * (counted on the host, one per kernel launch). */
colibri_status_t colibri_launch_count(const colibri_moe_t* h, uint64_t* n);

/* colibri_workspace_bytes - device bytes held by the handle (weights + workspace). */
colibri_status_t colibri_workspace_bytes(const colibri_moe_t* h, uint64_t* weights,
                                         uint64_t* workspace);

/* Stages of one forward, for colibri_profile_read. */
typedef enum {
    COLIBRI_STAGE_ROUTER = 0,     /* logits + top-k + softmax */
    COLIBRI_STAGE_DISPATCH = 1,   /* histogram, scan, permutation, tile list */
    COLIBRI_STAGE_GATHER = 2,     /* token rows into expert order (grouped executor) */
    COLIBRI_STAGE_EXPERT_UP = 3,  /* gate/up projection + SiLU * up */
    COLIBRI_STAGE_EXPERT_DOWN = 4,/* down projection */
    COLIBRI_STAGE_COMBINE = 5,    /* gate-weighted sum (+ residual) */
    COLIBRI_STAGE_RMSNORM = 6,    /* stack layers only */
    COLIBRI_NUM_STAGES = 7
} colibri_stage_t;

/*
 * colibri_profile_enable - when enable != 0, every later forward records a
 * CUDA event pair around each stage's kernel on the caller's stream (events
 * come from a host-side pool; no device memory is allocated).  0 turns it
 * off and drops what was recorded.
 */
colibri_status_t colibri_profile_enable(colibri_moe_t* h, int enable);

/*
 * colibri_profile_read - wait for the recorded events, then add each stage's
 * total device time (milliseconds) and number of kernel launches since the
 * last read into total_ms[COLIBRI_NUM_STAGES] and launches[COLIBRI_NUM_STAGES]
 * (host arrays, overwritten), and clear the record.
 */
colibri_status_t colibri_profile_read(colibri_moe_t* h, double* total_ms, uint64_t* launches);

/*
 * colibri_route_static - the routing stage of a layer (router logits, top-k,
 * softmax over the k, dispatch permutation) for callers that cannot allocate
 * device memory and have no handle.  The source pages have no counterpart of
 * this call.
 *
 * Who needs it: code that may not call cudaMalloc — while a stream is being
 * captured into a CUDA graph, inside a framework whose caching allocator owns
 * the device memory, or in a loop that cannot take the device-wide
 * synchronisation an allocation may cause.  Nothing is allocated: the call's
 * intermediate data lives in one fixed file-scope device array inside the
 * library (about 4.6 MiB, held by every GPU that loads the library until the
 * process exits).
 *
 *   x           [T, d_model] device, dtype
 *   w_router    [d_model, n_experts] device, dtype (the layout colibri_init takes)
 *   router_bias [n_experts] device float32, or NULL (same meaning as in colibri_init)
 *   topk_idx    [T, top_k] device int32, written (as colibri_get_routing)
 *   topk_w      [T, top_k] device float32, written
 *   counts      [n_experts] device int32, written
 *   perm        [T * top_k] device int32, written
 * Limits of the fixed array: d_model * n_experts <= 1048576 and
 * T * top_k <= 131072; larger sizes return COLIBRI_ERR_INVALID_ARG before any
 * CUDA call.  Shape rules as colibri_init (d_model % 64 == 0, d_model <=
 * 57856, n_experts <= 256, top_k <= 8 or top_k == n_experts (soft routing, as
 * in colibri_moe_config_t): COLIBRI_ERR_UNSUPPORTED otherwise, before any
 * CUDA call).
 *
 * Runs on the current device, ordered on `stream`, without waiting for it.
 * The first call on a device looks up the array's device address and checks
 * the architecture; make that first call before any stream capture.  The
 * address is kept for the life of the process: after cudaDeviceReset the
 * library's module is reloaded and the kept address is stale, so
 * cudaDeviceReset is not supported in a process that calls this entry point.
 * All calls on a device share the array and it keeps the last call's
 * contents: calls that overlap on the GPU (different streams, or unordered
 * graph nodes) race and give wrong results.
 *
 * The logits are computed by the CUDA-core router kernel.  A handle
 * computes them with other kernels (a many-CTA decode router with the dot
 * products cut into slices, or the tensor cores from 512 tokens), which add
 * the products in other orders: the gates may differ from
 * colibri_get_routing's in the last bits, and top-k may differ on tokens
 * whose deciding logits lie within float32 rounding of each other.  Counts
 * and perm are always the dispatch of the returned topk_idx.  A failure the dispatch detects on the device
 * (an expert id out of range, which the router never writes) sets every
 * counts[e] to -1.
 */
colibri_status_t colibri_route_static(const void* x, const void* w_router,
                                      const float* router_bias, int32_t T, int32_t d_model,
                                      int32_t n_experts, int32_t top_k, int32_t dtype,
                                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                                      int32_t* perm, void* stream);

/*
 * Expert parallelism: the experts of a layer split across the GPUs of one
 * machine, the token rows exchanged with an all-to-all (cf-1.com section 4.1:
 * GPU-to-GPU bandwidth for the communication between experts on several
 * cards; section 4.3: several GPUs of one machine).  The exchange itself is
 * the caller's (a collective library); these calls are the steps on each
 * side of it.  The source side routes its tokens (colibri_route_static) and
 * gathers the rows into expert order (colibri_gather_rows), so that the rows
 * bound for each owner are one contiguous range; after the exchange back it
 * combines the returned rows (colibri_combine_rows).  An owner runs its
 * experts on the rows it received (colibri_forward_routed on a handle
 * holding only its experts).
 */

/*
 * colibri_forward_routed - colibri_forward with the caller's routing instead
 * of the router: y[t] = sum_j topk_w[t, j] * FFN_{topk_idx[t, j]}(x[t]), j in
 * order, float32, then rounded once to dtype.  Dispatch, expert GEMMs and
 * combine are those of colibri_forward.
 *   x, y      [T, d_model] device, dtype, 16-byte aligned, not overlapping
 *   topk_idx  [T, k] device int32, expert ids of this handle (0 .. n_experts-1)
 *   topk_w    [T, k] device float32
 * T * k may not exceed max_tokens * top_k of the handle's configuration
 * (COLIBRI_ERR_INVALID_ARG).  An id out of range is reported by colibri_check
 * (COLIBRI_ERR_CUDA) after the stream reaches it.  Allocates nothing.
 */
colibri_status_t colibri_forward_routed(colibri_moe_t* h, const void* x, int32_t T, int32_t k,
                                        const int32_t* topk_idx, const float* topk_w, void* y,
                                        void* stream);

/*
 * colibri_gather_rows - xp[p] = x[perm[p] / k] for p < npairs: the token rows
 * in the expert order of a dispatch permutation (perm as colibri_route_static
 * and colibri_get_routing give it).
 *   x [x_rows, d_model], xp [npairs, d_model] device, dtype, 16-byte aligned
 *   perm [npairs] device int32; a value outside 0 .. x_rows*k-1 gathers a
 *   zero row (every access stays in bounds)
 * d_model * element size a multiple of 16 bytes.  Runs on the current
 * device, ordered on `stream`; allocates nothing.
 */
colibri_status_t colibri_gather_rows(const void* x, int32_t x_rows, const int32_t* perm, int32_t k,
                                     int32_t npairs, int32_t d_model, int32_t dtype, void* xp,
                                     void* stream);

/*
 * colibri_combine_rows - y[t] = sum_j topk_w[t, j] * rows[p(t, j)], j in
 * order, float32, rounded once to dtype, where p(t, j) is the position of
 * pair t*k + j in perm (rows in expert order, one per pair).
 *   rows        [T * k, d_model] device: float32 (rows_dtype FP32), or bf16
 *               (rows_dtype BF16, with dtype BF16); 16-byte aligned
 *   topk_w      [T, k] device float32
 *   perm        [T * k] device int32, a permutation of 0 .. T*k-1 (a pair
 *               whose position no value names adds nothing; values out of
 *               range are skipped, so every access stays in bounds)
 *   inv_scratch [T * k] device int32, overwritten (the inverse of perm)
 *   y           [T, d_model] device, dtype, 16-byte aligned
 * d_model % 8 == 0 and T * k <= INT32_MAX (COLIBRI_ERR_INVALID_ARG
 * otherwise).  Runs on the current device, ordered on `stream`.
 */
colibri_status_t colibri_combine_rows(const void* rows, int32_t rows_dtype, const float* topk_w,
                                      const int32_t* perm, int32_t T, int32_t k, int32_t d_model,
                                      int32_t dtype, int32_t* inv_scratch, void* y, void* stream);

/* colibri_free - release everything the handle holds; NULL is allowed.
 * Synchronises the handle's device first. */
void colibri_free(colibri_moe_t* h);

/* colibri_status_str - a static, never-NULL description of a status. */
const char* colibri_status_str(colibri_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* COLIBRI_MOE_H */
