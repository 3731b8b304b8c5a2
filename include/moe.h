/*
 * moe.h -- C ABI of the GB300 (sm_103a) fused mixture-of-experts layer
 * forward: router -> top-k gate -> dispatch -> expert FFN -> combine.
 *
 * The operation is the five-step MoE forward of the page "用Ascend C写一个
 * MoE融合算子" (Writing a fused MoE operator in Ascend C), section
 * "MoE的计算流程":
 *   1. Routing   scores  = TopK(x × W_router)
 *   2. Gating    weights = Softmax(scores)            (over the k selected)
 *   3. Dispatch  x_e     = x[tokens assigned to e]
 *   4. Expert    y_e     = GELU(x_e × W1_e) × W2_e    (section "2. Dispatch +
 *                          Expert + Combine 流水线", listing "Expert计算")
 *   5. Combine   y       = Σ_j weights_j × y_{e_j}     (listing "Scatter + 加权")
 * with an optional capacity factor (article "CANN ops-transformer MoE",
 * section 4.3, capacity_factor = 1.2) that drops an overloaded expert's
 * assignments in ascending token order (page "CANN ops-transformer：MoE
 * 路由算子的负载均衡策略", section "负载不均衡的根源", token dropping).
 *
 * Readings fixed by this library where the pages are silent:
 *   - TopK: descending logit; equal logits -> lower expert index first.
 *     Column j of ids/weights is the j-th best expert.
 *   - Router logits and the gate softmax are fp32 (bf16 inputs, fp32
 *     accumulation); an optional fp32 bias b[E] is added to the logits.
 *     The gate weights follow moe_shape.gating (default: softmax over the
 *     k selected logits).
 *   - GELU is the exact form 0.5 z (1 + erf(z / sqrt 2)).
 *   - capacity C = ceil(capacity_factor * T * k / E - 1e-9) when
 *     capacity_factor > 0, else unlimited.  The first C assignments of each
 *     expert in ascending (token, slot) order are kept; dropped ones are not
 *     re-routed and the survivors keep their softmax weight; a token whose
 *     slots are all dropped gets y = 0.
 *   - The expert hidden activation h and the expert output are rounded to
 *     bf16 in the workspace; y is bf16 (round to nearest even) from an fp32
 *     combine summed in slot order j = 0..k-1.  With k = 1 the combine is
 *     done by the second expert GEMM itself: y[t] = w[t] * (h W2) is formed
 *     from the fp32 accumulator and rounded to bf16 once (no bf16 rounding
 *     of the expert output in between).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *     contiguous, 16-byte aligned.  bf16 tensors are passed as uint16_t bit
 *     patterns.  The library never allocates, frees or retains memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream: they only enqueue work and never
 *     synchronise the host, except moe_get_device_status.
 *   - `ws` is a caller-owned device workspace of `ws_bytes` bytes, at least
 *     moe_workspace_size() for moe_forward / moe_expert_ffn_combine and at
 *     least moe_route_workspace_size() for moe_route / moe_dispatch; its
 *     first bytes hold the device status word of the most recent call.
 *     Concurrent calls must not share a workspace.
 *   - Return value: MOE_OK or an MOE_ERR_* code.  Arguments are validated on
 *     the host before anything is enqueued; on an error nothing is launched
 *     and moe_last_error_string() describes the problem.
 *   - Faults found on the device (a bounded wait that ran out, an expert id
 *     out of range) do not trap: kernels set bits in the status word, which
 *     moe_get_device_status() reads back.
 *
 * Limits (MOE_ERR_UNSUPPORTED beyond them): 1 <= E <= 256,
 * 1 <= k <= min(8, E), H % 8 == 0, F % 8 == 0, H >= 8, F >= 8,
 * T * k <= 2^24.  T == 0 is accepted and only clears counts/offsets.
 * When E % 8 != 0 the rows of W_router are not 16-byte aligned; the route
 * then first copies W_router into the workspace with its rows padded to a
 * multiple of 8 experts (zeros, never selected).
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1 /* null/misaligned pointer, bad size, small workspace */
#define MOE_ERR_UNSUPPORTED 2 /* shape outside the limits above */
#define MOE_ERR_CUDA 3        /* a CUDA runtime/driver call failed */
#define MOE_ERR_TIMEOUT 4     /* moe_get_device_status: a device wait ran out */
#define MOE_ERR_DEVICE 5      /* moe_get_device_status: another device fault bit */

/* Device status bits (the word moe_get_device_status returns). */
#define MOE_DEV_TIMEOUT 0x1 /* a kernel's bounded wait gave up */
#define MOE_DEV_BAD_ID 0x2  /* an expert id outside [0, E) reached dispatch */

/* Smallest workspace accepted by moe_get_device_status and
 * moe_selftest_wait_timeout. */
#define MOE_WS_MIN_BYTES 256

/* Gate weights (moe_shape.gating).
 * MOE_GATE_TOPK_SOFTMAX (0, default): softmax over the k selected logits
 *   (the router kernel of "用Ascend C写一个MoE融合算子", section "1. Routing +
 *   Gating 合并": Softmax over the top-k scores only).
 * MOE_GATE_SOFTMAX_TOPK (1): softmax over all E logits, then the k selected
 *   probabilities as they are (the Softmax -> Top-k order of section 2.1 of
 *   the article "CANN ops-transformer MoE"); a token's weights sum to less
 *   than 1 unless k = E.
 * MOE_GATE_SOFTMAX_TOPK_RENORM (2): as 1, then the k probabilities divided
 *   by their sum (mathematically equal to 0; computed in this order).
 * The selected experts are the same in all three modes. */
#define MOE_GATE_TOPK_SOFTMAX 0
#define MOE_GATE_SOFTMAX_TOPK 1
#define MOE_GATE_SOFTMAX_TOPK_RENORM 2

/* Expert FFN (moe_shape.expert_act).
 * MOE_EXPERT_GELU (0, default): y_e = GELU(x W1[e]) W2[e], W1 [E, H, F]
 *   (listing "Expert计算" of "用Ascend C写一个MoE融合算子").
 * MOE_EXPERT_SWIGLU (1): y_e = (SiLU(x W_gate[e]) * (x W_up[e])) W2[e], with
 *   W1 [E, H, 2F] = [W_gate | W_up] along the last dimension (the gated
 *   experts of the Llama 3 / Mixtral / DeepSeek models the page names);
 *   SiLU(z) = z / (1 + exp(-z)).  W2 is [E, F, H] in both. */
#define MOE_EXPERT_GELU 0
#define MOE_EXPERT_SWIGLU 1

typedef struct moe_shape {
  int32_t T; /* tokens */
  int32_t H; /* hidden size */
  int32_t F; /* expert FFN width (ignored by moe_route / moe_dispatch) */
  int32_t E; /* experts */
  int32_t k; /* experts per token */
  double capacity_factor; /* <= 0 or NaN: no capacity limit */
  int32_t gating; /* MOE_GATE_*; 0 (zero-initialised) = softmax over the k selected */
  int32_t expert_act; /* MOE_EXPERT_*; 0 (zero-initialised) = GELU FFN */
} moe_shape;

/* Library version, (major << 16) | minor. */
MOE_API int moe_version(void);

/* Message describing the last error returned on this host thread. */
MOE_API const char* moe_last_error_string(void);

/* Expert capacity C for the shape (see above), or -1 for no limit. */
MOE_API int64_t moe_expert_capacity(const moe_shape* s);

/* Workspace bytes needed by moe_forward and moe_expert_ffn_combine (and
 * enough for every other entry point): a 1 KB status block, per-128-token
 * expert counts [ceil(T/128), E] int32, the padded W_router copy when
 * E % 8 != 0 (see moe_route_workspace_size), the fused route's per-CTA
 * expert counts (bytes, at most 256 rows of E rounded up to 16) for the
 * batches it serves, h [T*k, F] bf16, a [T*k, H] bf16
 * region that holds first the token rows in dispatch order, then the
 * expert outputs, and for T*k <= 64 rows fp32 partial expert outputs of up
 * to 4 K splits [4, T*k, H] (the small-batch second GEMM).  Returns 0 for
 * an invalid shape. */
MOE_API size_t moe_workspace_size(const moe_shape* s);

/* Workspace bytes needed by moe_route and moe_dispatch (status block,
 * per-128-token expert counts, when E % 8 != 0 the padded copy of W_router
 * [H, E rounded up to 8], and the fused route's per-CTA counts; F is
 * ignored).  Returns 0 for an invalid shape. */
MOE_API size_t moe_route_workspace_size(const moe_shape* s);

/*
 * Which kernels moe_forward (and moe_route) launch for this shape; no
 * counterpart on the pages, for callers that count or profile kernels.
 * Host only: depends on the shape alone.
 *   *dispatch_in_router = 1 when the dispatch (step 3) runs in the router's
 *     launch: small batches (T <= 128 and E <= 64, logits on the CUDA
 *     cores) and batches of up to 128 tiles of 128 tokens (T <= 16384; the
 *     fused tensor-core route, on a GPU that holds one such CTA per SM for
 *     at least 128 SMs, as every sm_103 part does); 0: the tensor-core
 *     cluster router, then a dispatch kernel.
 *   *combine_in_gemm = 1 for k = 1: the combine runs inside the second
 *     expert GEMM; 0: a separate combine kernel.
 * Returns MOE_OK, or MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad
 * shape or a null output.
 */
MOE_API int moe_forward_plan(const moe_shape* s, int32_t* dispatch_in_router,
                             int32_t* combine_in_gemm);

/*
 * The launch shape of the one-launch tensor-core route on the current
 * device, for callers that profile the route; no counterpart on the pages.
 *   *tile_tokens = tokens per tile (64 or 128), *splits = K splits per tile
 *     (the thread-block cluster size: 1, 2, 4 or 8) -- the pair that
 *     minimises the bytes each CTA streams among those whose clusters all
 *     fit on the device at once; both 0 when the shape routes otherwise
 *     (small batch on the CUDA cores, or router + dispatch kernels).
 * Sets up the current device (as every entry point does).  Returns MOE_OK,
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad shape or a null
 * output, MOE_ERR_CUDA if the device cannot be set up.
 */
MOE_API int moe_route_plan(const moe_shape* s, int32_t* tile_tokens, int32_t* splits);

/*
 * Steps 1-3 (the router kernel "MoERouterKernel::Process": x × W_router on
 * the tensor cores, per-token TopK, Softmax over the k scores; then the
 * dispatch of GatherTokensByExpert) for all T tokens.  Up to 128 tiles of
 * 128 tokens this is one launch that splits the logit GEMM along H across
 * the CTAs of a thread-block cluster (tiles of 64 or 128 tokens, up to 8
 * splits, spread over the SMs) and dispatches in the same kernel; every
 * wait inside it on memory or on other clusters is
 * bounded (a CTA that could not become resident, e.g. behind another
 * stream's long kernel, ends the call with MOE_DEV_TIMEOUT, not a hang).
 *   x        [T, H]  bf16        w_router [H, E] bf16 (E contiguous)
 *   b_router [E]     fp32 or NULL (added to the logits)
 * Outputs (device, caller-owned):
 *   ids      [T, k]  int32   selected experts, best first
 *   weights  [T, k]  fp32    softmax over the k selected logits
 *   counts   [E]     int32   kept assignments per expert (after capacity)
 *   offsets  [E+1]   int32   exclusive prefix sum of counts
 *   perm     [T*k]   int32   perm[offsets[e] + r] = t*k + j of the r-th kept
 *                            assignment of expert e, tokens ascending;
 *                            entries >= offsets[E] are -1
 *   slot     [T, k]  int32   row of assignment (t, j) in perm, -1 if dropped
 * The router logits never leave the chip.
 */
MOE_API int moe_route(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
              const float* b_router, int32_t* ids, float* weights, int32_t* counts,
              int32_t* offsets, int32_t* perm, int32_t* slot, void* ws, size_t ws_bytes,
              void* stream);

/*
 * Step 3 alone (GatherTokensByExpert as a stable counting sort plus the
 * capacity clip): ids [T, k] -> counts, offsets, perm, slot as in moe_route.
 * Ids outside [0, E) are treated as dropped and set MOE_DEV_BAD_ID.
 */
MOE_API int moe_dispatch(const moe_shape* s, const int32_t* ids, int32_t* counts, int32_t* offsets,
                 int32_t* perm, int32_t* slot, void* ws, size_t ws_bytes, void* stream);

/*
 * Steps 4-5 (the expert kernel "MoEExpertKernel::Process" and its
 * ScatterWithWeights, written as a gather): for every kept assignment,
 * h = GELU(x[t] × W1[e]) and y_e = h × W2[e]; then
 * y[t] = Σ_{j: slot[t,j] >= 0} weights[t,j] × y_e(t,j).
 *   x [T, H] bf16, W1 [E, H, F] bf16 (F contiguous; [E, H, 2F] for
 *   MOE_EXPERT_SWIGLU), W2 [E, F, H] bf16 (H contiguous); weights, offsets,
 *   perm, slot as produced by moe_route.
 *   y [T, H] bf16 (output).
 * The kept token rows are first copied in dispatch order into the
 * workspace (row r = x[perm[r] / k], the dispatch step's x_i of section
 * "MoE的计算流程"), which both expert GEMMs then read with TMA.
 * perm/offsets must describe a valid dispatch (0 <= perm < T*k, offsets
 * non-decreasing, offsets[E] <= T*k); the library does not re-validate them
 * (a token index outside [0, T) is clamped, never dereferenced).
 */
MOE_API int moe_expert_ffn_combine(const moe_shape* s, const uint16_t* x, const uint16_t* w1,
                           const uint16_t* w2, const float* weights, const int32_t* offsets,
                           const int32_t* perm, const int32_t* slot, uint16_t* y, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * The steps of moe_expert_ffn_combine one at a time, for callers that move
 * rows between the steps themselves -- e.g. expert parallelism, where each
 * GPU holds some of the experts and the dispatched rows travel to their
 * expert's GPU and back (the article's section 3 all-to-all).
 *
 * moe_dispatch_rows: the dispatch step's regrouped tokens x_i of section
 * "MoE的计算流程" (step 3): xp[r] = x[perm[r] / k] for r < offsets[E], in
 * dispatch order (expert-major); rows of xp past offsets[E] are not written.
 *   x [T, H] bf16, perm / offsets as produced by moe_route, xp [T*k, H] bf16.
 * Uses no workspace; perm entries outside [0, T*k) are clamped, never
 * dereferenced.
 */
MOE_API int moe_dispatch_rows(const moe_shape* s, const uint16_t* x, const int32_t* perm,
                              const int32_t* offsets, uint16_t* xp, void* stream);

/*
 * moe_expert_ffn: step 4 (listing "Expert计算") on rows already grouped:
 * rows [seg_offsets[i], seg_offsets[i+1]) of xp form segment i, computed by
 * expert i % E:  Y[r] = act(xp[r] · W1[e]) · W2[e]  (GELU, or SwiGLU with
 * W1 = [W_gate | W_up]), h and Y rounded to bf16.
 *   s: H, F, E (the experts whose weights W1 / W2 hold, 1..256),
 *     expert_act; T*k is the row
 *     capacity of xp and Y (e.g. T = rows, k = 1); gating is ignored.
 *   n_segments: 1..256; seg_offsets [n_segments+1] int32 (device), non-
 *     decreasing, seg_offsets[n_segments] <= T*k (not re-validated).
 *   xp [T*k, H] bf16, W1 [E, H, F] (or [E, H, 2F]), W2 [E, F, H], Y [T*k, H]
 *   bf16 (rows outside every segment are not written).
 * With E experts per GPU and rows received from G sources, each source's
 * rows grouped by expert, n_segments = G * E and segment i = (source i / E,
 * expert i % E): the received buffer is used as it arrives.
 * ws as for moe_expert_ffn_combine (moe_workspace_size of the same s).
 */
MOE_API int moe_expert_ffn(const moe_shape* s, int32_t n_segments, const uint16_t* xp,
                           const uint16_t* w1, const uint16_t* w2, const int32_t* seg_offsets,
                           uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_combine: step 5 (listing "Scatter + 加权", written as a gather):
 * y[t] = sum over j with slot[t,j] >= 0 of weights[t,j] * Y[slot[t,j]],
 * fp32 in slot order, rounded to bf16; 0 when every slot was dropped.
 *   Y [T*k, H] bf16 in dispatch order, weights [T, k] fp32, slot [T, k]
 *   int32 as produced by moe_route, y [T, H] bf16.  No workspace.
 */
MOE_API int moe_combine(const moe_shape* s, const uint16_t* Y, const float* weights,
                        const int32_t* slot, uint16_t* y, void* stream);

/*
 * The whole layer (the op "MoEFusion::Compute(x, w_router, expert_weights,
 * y)" of section "3. 完整调用流程"): moe_route followed by
 * moe_expert_ffn_combine on `stream` with no host synchronisation: a small
 * kernel that clears the status block, then router, dispatch, permute,
 * expert GEMM1, expert GEMM2 and combine -- seven kernels, one fewer when
 * the router also dispatches (moe_forward_plan: up to 128 tiles of 128
 * tokens), one fewer when GEMM2 also combines (k = 1), and one more (a
 * W_router copy padded to 8-expert rows) when E % 8 != 0.  The routing
 * outputs are written as in moe_route.
 */
MOE_API int moe_forward(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                const float* b_router, const uint16_t* w1, const uint16_t* w2, uint16_t* y,
                int32_t* ids, float* weights, int32_t* counts, int32_t* offsets, int32_t* perm,
                int32_t* slot, void* ws, size_t ws_bytes, void* stream);

/*
 * Bytes of the library's built-in device scratch used by
 * moe_expert_ffn_combine_noalloc (held on every GPU that loads the library
 * until the process exits).
 */
#define MOE_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * moe_expert_ffn_combine for callers that cannot allocate device memory.
 * The pages have no counterpart: it exists for hosts that own only their
 * input and output buffers -- e.g. a runtime that reserves all device memory
 * at start-up and forbids cudaMalloc afterwards, or a plain C caller with no
 * device allocator at hand -- and so cannot provide the `ws` workspace.
 * Same arguments and results as moe_expert_ffn_combine, without `ws`: the
 * hidden activations and expert outputs live in a static device array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes inside the library.
 *   - Shapes whose workspace (moe_workspace_size) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ERR_UNSUPPORTED.  The
 *     workspace is about T*k*(F+H)*2 bytes, plus T*k*H*16 bytes of fp32
 *     split-K partials when T*k <= 64 rows: at H = 4096, F = 14336 the limit
 *     is about 900 rows of T*k (a 32-token, k = 2 decode step needs 6.4 MB).
 *   - Nothing is allocated or freed.  The first call on a device looks up
 *     the scratch's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture.
 *   - Every call on a device shares the one scratch array: calls that
 *     overlap on the GPU (different streams, or different host threads)
 *     race and corrupt each other's results; serialise them.
 *   - Device status bits of these calls are kept in the scratch; read (and
 *     clear) them with moe_noalloc_device_status, not moe_get_device_status.
 */
MOE_API int moe_expert_ffn_combine_noalloc(const moe_shape* s, const uint16_t* x,
                                           const uint16_t* w1, const uint16_t* w2,
                                           const float* weights, const int32_t* offsets,
                                           const int32_t* perm, const int32_t* slot, uint16_t* y,
                                           void* stream);

/*
 * The device status word of moe_expert_ffn_combine_noalloc's built-in
 * scratch on the current device (no counterpart on the pages): synchronises
 * `stream`, reads the word into *status and clears it, with the return codes
 * of moe_get_device_status.  Allocates nothing.
 */
MOE_API int moe_noalloc_device_status(void* stream, int32_t* status);

/*
 * moe_forward with timing hooks (no counterpart on the pages): `events`
 * points to 7 cudaEvent_t handles (any may be NULL; `events` itself may be
 * NULL), recorded on `stream` before the router kernel (after the status
 * clear) and after each of the six steps: router, dispatch, permute (token
 * rows into dispatch order), expert GEMM1, expert GEMM2, combine.  A step
 * that runs inside another kernel (dispatch in the small-batch router,
 * combine in GEMM2 when k = 1) has its two events recorded back to back.
 * The events are caller-owned; the library only records them.
 */
MOE_API int moe_forward_profiled(const moe_shape* s, const uint16_t* x, const uint16_t* w_router,
                                 const float* b_router, const uint16_t* w1, const uint16_t* w2,
                                 uint16_t* y, int32_t* ids, float* weights, int32_t* counts,
                                 int32_t* offsets, int32_t* perm, int32_t* slot, void* ws,
                                 size_t ws_bytes, void* stream, void* const* events);

/*
 * Synchronises `stream`, reads the device status word of the workspace into
 * *status and clears it.  Returns MOE_OK when the word is 0,
 * MOE_ERR_TIMEOUT when MOE_DEV_TIMEOUT is set, MOE_ERR_DEVICE for other
 * bits, MOE_ERR_CUDA if the copy fails.
 */
MOE_API int moe_get_device_status(void* ws, void* stream, int32_t* status);

/*
 * Self-test of the bounded-wait machinery, no counterpart on the pages:
 * launches one CTA that waits on an mbarrier nobody arrives on, with a
 * limit of `limit_ns` nanoseconds (1e3 .. 1e10), then records
 * MOE_DEV_TIMEOUT in the workspace status word and returns.  Used by the
 * failure-detection test; nothing traps or hangs.
 */
MOE_API int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H */
