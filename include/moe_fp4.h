/*
 * moe_fp4.h — C ABI of the FP4 routed mixture-of-experts layer for GB300 (sm_103a).
 *
 * The layer is the routed-expert block of DeepSeek-V4-Flash-style inference
 * ("DeepSeek-V4-Flash on AMD gfx90a: Correctness Recovery and Inference
 * Performance Engineering", abstract: FP4 routed mixture-of-experts with packed
 * FP4 weights and expert sorting; the "MXFP4 MoE" path of the vLLM-on-MI300X
 * write-up).  Per token it
 *   1. picks the top-k experts of the router logits, ordered by (logit desc,
 *      expert index asc), and weights them by the softmax over the k picked
 *      logits (fp32 comparison, ties to the lower expert id: MI250 correctness
 *      blog, section 4.1 table and section 4.2);
 *   2. sorts the T*k (token, slot) pairs by expert with a stable counting sort
 *      and builds per-expert offsets ("retuned expert sorting");
 *   3. for every expert, multiplies its tokens by the packed-FP4 W13 (gate and
 *      up) and applies SwiGLU, h = bf16(silu(g) * u);
 *   4. multiplies h by the packed-FP4 W2 (down) and combines the k expert
 *      outputs of each token with its routing weights (by default added into
 *      out in the W2 kernel's epilogue in no fixed order; in slot order with
 *      MOE_FP4_FLAG_DETERMINISTIC).
 *
 * Formats (MXFP4, OCP Microscaling v1.0):
 *   - weights: two E2M1 codes per byte along K, the LOW nibble holds the even
 *     K element; code bit 3 = sign, bits 0..2 index {0, .5, 1, 1.5, 2, 3, 4, 6};
 *   - scales: E8M0 bytes, value 2^(s-127), one per 32 consecutive K elements
 *     of a row; s in [0, 253].  Bytes 254 and 255 (NaN), and scales that push
 *     a product or sum past the fp32 range, are outside the contract: results
 *     are unspecified, nothing faults.
 *   - x is bf16 (raw IEEE binary32 upper halves), router logits and all
 *     outputs are fp32 except h (bf16).  Router logits must be finite.
 *
 * Tensor layouts (all row-major, C-contiguous, device memory unless stated):
 *   x              bf16   [T, d]
 *   router_logits  fp32   [T, E]
 *   w13            uint8  [E, 2I, d/2]   rows [0, I) = gate, rows [I, 2I) = up
 *   w13_scale      uint8  [E, 2I, d/32]
 *   w2             uint8  [E, d, I/2]    row n = output feature n, packed along I
 *   w2_scale       uint8  [E, d, I/32]
 *   out            fp32   [T, d]         fully overwritten
 *   topk_ids       int32  [T, k]         slot 0 = highest logit
 *   topk_weights   fp32   [T, k]
 *   expert_offsets int32  [E + 1]        expert e owns sorted rows [off[e], off[e+1])
 *   sorted_slot    int32  [T*k]          sorted row r -> flat slot t*k + j,
 *                                        increasing within each expert
 *   h              bf16   [T*k, I]       SwiGLU output in sorted-row order
 *
 * Ownership and threading: the caller owns every buffer and the stream.  The
 * library allocates nothing; all scratch lives in the caller's workspace
 * (moe_fp4_workspace_bytes).  moe_fp4_route and moe_fp4_forward only enqueue
 * work on the given stream and never synchronise.  Calls that use different
 * workspaces may run concurrently; calls sharing a workspace must be ordered
 * on one stream.  Inside a call the kernels after routing are launched with
 * programmatic dependent launch (each waits on the device for the one before
 * it); the call as a whole keeps ordinary stream order with the caller's work:
 * its first kernel starts after everything enqueued before it, and the last
 * kernel of moe_fp4_forward lets no later kernel start early.  (The routing
 * kernel of moe_fp4_route, T <= 32, does let a following kernel that the
 * caller launches early start before it ends; such a kernel must wait on the
 * device, griddepcontrol.wait, before it reads the routing outputs, as any
 * early-launched kernel must.)
 *
 * Errors: every function returns a moe_fp4_status.  Argument checks happen on
 * the host before anything is enqueued; on error nothing is launched.  A
 * failed launch returns MOE_FP4_ERR_CUDA (the CUDA error is left for the
 * caller's next CUDA call to see).  Kernels never trap.
 */
#ifndef MOE_FP4_H_
#define MOE_FP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Problem sizes.  T tokens, d hidden size, I expert intermediate size,
 * E experts, k experts per token. */
typedef struct moe_fp4_dims {
  int32_t T, d, I, E, k;
} moe_fp4_dims;

typedef enum moe_fp4_status {
  MOE_FP4_OK = 0,
  MOE_FP4_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer */
  MOE_FP4_ERR_UNSUPPORTED = -2,  /* sizes the kernels do not cover (see moe_fp4_workspace_bytes) */
  MOE_FP4_ERR_WORKSPACE = -3,    /* workspace too small */
  MOE_FP4_ERR_CUDA = -4,         /* a CUDA runtime call failed */
  MOE_FP4_ERR_DEVICE = -5        /* a kernel reported an error word (moe_fp4_check) */
} moe_fp4_status;

/* Flags for moe_fp4_forward.  Both expert paths give results within the same
 * tolerance of the definition; the default picks by shape (expected rows per
 * expert = T*k/E): the streaming GEMV path for few rows, the tensor-core path
 * otherwise. */
#define MOE_FP4_FLAG_FORCE_GEMV 0x1u    /* streaming path: weights streamed once, warp-level mma.sync
                                           (d, I multiples of 1024) */
#define MOE_FP4_FLAG_FORCE_TC   0x2u    /* tcgen05 tensor-core path */
/* On the streaming path: both projections in one persistent launch (W13 +
 * SwiGLU, a grid-wide arrival counter with a bounded wait, then W2), one CTA
 * per SM launched cooperatively, instead of two launches (the paper's
 * per-layer synchronisation and launch cost, abstract: limits).  The same
 * results; in moe_fp4_forward_profiled the W13 stage then covers both
 * projections and the W2 stage is empty.  May be combined with
 * MOE_FP4_FLAG_FORCE_GEMV; ignored on the tensor-core path. */
#define MOE_FP4_FLAG_PERSISTENT 0x4u
/* On the tensor-core path: run both projections on pairs of SMs (tcgen05
 * cta_group::2: one MMA instruction covers M = 256 weight rows, 128 from each
 * CTA's tensor memory, with the token tile split between the two CTAs), and
 * the weighted combine inside the W2 kernel (per-token counters; the CTA
 * that completes a token's k slots sums them in slot order, deterministic).
 * The same results within the layer's tolerance; slower than the default
 * one-SM kernels on GB300 (the dequantisers' tensor-memory stores wait while
 * the pair's MMAs read both SMs' tensor memory).  Ignored on the streaming
 * path. */
#define MOE_FP4_FLAG_CTA_PAIRS 0x8u
/* The weighted combine.  By default the W2 kernel adds each slot's weighted
 * output row into out in its epilogue (fp32 atomic adds, out zeroed first):
 * no y buffer round trip and no separate pass, but the k terms of an output
 * element are summed in whatever order the slots finish, so results may
 * differ in the last bits between calls.  With this flag the W2 kernel writes
 * y and a separate pass sums the k rows of each token in slot order:
 * bitwise reproducible.  CTA pairs always use their own in-epilogue combine in
 * slot order (reproducible); the fallback paths for sizes outside the
 * streaming kernel's use the separate pass. */
#define MOE_FP4_FLAG_DETERMINISTIC 0x10u

/* Bytes of device workspace a call with these sizes needs (256-byte aligned
 * base required).  Returns 0 when the sizes are invalid or unsupported:
 * T >= 1, 1 <= k <= min(E, 32), 1 <= E <= 1024, d and I multiples of 128,
 * 128 <= d <= 16384, 128 <= I <= 16384, T*k < 2^31, T*k*max(d, I) < 2^40. */
size_t moe_fp4_workspace_bytes(const moe_fp4_dims* dims);

/* Steps 1-2 only (routing and the expert sort), so that routing can be
 * checked bit-exactly on its own (the paper's fixed-token and hash checks).
 * topk_ids, topk_weights, expert_offsets and sorted_slot are required
 * device outputs.  Pointers: 4-byte aligned; workspace 256-byte aligned. */
int moe_fp4_route(const moe_fp4_dims* dims, const float* router_logits,
                  int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                  int32_t* sorted_slot, void* workspace, size_t workspace_bytes,
                  void* cuda_stream);

/* The whole layer (steps 1-4) on device buffers.  out is required; the
 * routing outputs and h are optional (NULL: kept in the workspace only).
 * x, w13, w13_scale, w2, w2_scale, out and h must be 16-byte aligned,
 * the routing outputs 4-byte aligned, the workspace 256-byte aligned.  flags: 0 or one MOE_FP4_FLAG_FORCE_*,
 * optionally with MOE_FP4_FLAG_PERSISTENT. */
int moe_fp4_forward(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                    const uint8_t* w13, const uint8_t* w13_scale,
                    const uint8_t* w2, const uint8_t* w2_scale, float* out,
                    int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                    int32_t* sorted_slot, void* h_bf16, unsigned flags,
                    void* workspace, size_t workspace_bytes, void* cuda_stream);

/* The router (gate) projection, the step ahead of top-k routing:
 *   router_logits[t, e] = sum_K x[t, K] * w_gate[e, K]
 * with bf16 x [T, d] and bf16 w_gate [E, d] (row e = expert e's gate
 * vector), every product exact, fp32 accumulation, fp32 logits [T, E] (the
 * MI250 correctness blog, section 4.1: low-precision inputs with FP32
 * accumulation for the gate network, FP32 values for the top-k comparison).
 * The sum order is fixed, so the logits are the same on every call.  x and
 * w_gate 16-byte aligned, router_logits 4-byte aligned; dims as for
 * moe_fp4_forward (I and k are not used).  One kernel is enqueued; no
 * workspace. */
int moe_fp4_router(const moe_fp4_dims* dims, const void* x_bf16, const void* w_gate_bf16,
                   float* router_logits, void* cuda_stream);

/* The whole layer starting from x and the router weights: moe_fp4_router
 * writes router_logits (a required [T, E] fp32 device buffer owned by the
 * caller), then moe_fp4_forward runs on them.  Same arguments, checks and
 * results as moe_fp4_forward otherwise; every argument is checked before
 * anything is enqueued. */
int moe_fp4_forward_gated(const moe_fp4_dims* dims, const void* x_bf16, const void* w_gate_bf16,
                          float* router_logits, const uint8_t* w13, const uint8_t* w13_scale,
                          const uint8_t* w2, const uint8_t* w2_scale, float* out,
                          int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                          int32_t* sorted_slot, void* h_bf16, unsigned flags,
                          void* workspace, size_t workspace_bytes, void* cuda_stream);

/* moe_fp4_forward that also records caller-created CUDA events (cudaEvent_t
 * handles, MOE_FP4_NUM_STAGE_EVENTS of them) on the stream between its
 * stages, so that a caller can time each kernel in place:
 *   events[0] before routing and the expert sort (3 kernels)
 *   events[1] before the token gather (tensor-core path only; else empty)
 *   events[2] before W13 + SwiGLU
 *   events[3] before W2
 *   events[4] before the combine pass
 *   events[5] after the combine pass (empty when the W2 kernel does the
 *   combine in its epilogue, the default)
 * Same arguments, checks and results as moe_fp4_forward. */
#define MOE_FP4_NUM_STAGE_EVENTS 6
int moe_fp4_forward_profiled(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                             const uint8_t* w13, const uint8_t* w13_scale,
                             const uint8_t* w2, const uint8_t* w2_scale, float* out,
                             int32_t* topk_ids, float* topk_weights, int32_t* expert_offsets,
                             int32_t* sorted_slot, void* h_bf16, unsigned flags,
                             void* workspace, size_t workspace_bytes, void* cuda_stream,
                             void* const* stage_events);

/* Bytes of device workspace moe_fp4_forward_host needs: the forward workspace
 * plus device staging for x, router_logits and out. */
size_t moe_fp4_host_workspace_bytes(const moe_fp4_dims* dims);

/* The whole layer with HOST x, router_logits and out (weights stay on the
 * device).  Copies x to device staging inside the workspace, runs
 * moe_fp4_forward and synchronises the stream before returning.  Host buffers
 * may be pageable or pinned (pinned is faster).  router_logits and out in
 * memory the device can address (page-locked by the CUDA allocator or
 * registered with it; out 16-byte aligned) are used in place: the routing
 * kernel reads the logits and the combine writes out over the host link, with
 * no copy.  Otherwise they go through device staging too. */
int moe_fp4_forward_host(const moe_fp4_dims* dims, const void* x_bf16_host,
                         const float* router_logits_host,
                         const uint8_t* w13, const uint8_t* w13_scale,
                         const uint8_t* w2, const uint8_t* w2_scale, float* out_host,
                         unsigned flags, void* workspace, size_t workspace_bytes,
                         void* cuda_stream);

/* The whole layer without any workspace argument, for callers that cannot
 * allocate device memory: runtimes without an allocator, callers that must
 * not call cudaMalloc inside a stream-ordered or captured region, plugins
 * that are handed only input and output pointers.  (The paper has no
 * counterpart; this is a deployment convenience.)
 *
 * Scratch: a fixed device array of MOE_FP4_NOALLOC_SCRATCH_BYTES inside this
 * library, which every GPU that loads the library holds until the process
 * exits.  Problems whose moe_fp4_workspace_bytes exceeds it are rejected with
 * MOE_FP4_ERR_WORKSPACE before anything is enqueued.  With E = 256 and k = 8
 * that allows T <= 72 tokens at d = 4096, I = 2048 (the T = 32 decode batch
 * needs about 7.4 MB) and T <= 44 at d = 7168, I = 2048; prefill-sized
 * batches need a workspace (moe_fp4_forward).
 * The array's device address is looked up (with the call's device current)
 * on every call made outside a stream capture, so a device reset between calls
 * is harmless; a call made during a capture uses the address of the last call
 * outside one, so make one call on each device before capturing.
 * All calls share the array and it keeps the last call's contents: calls
 * that overlap on the GPU (other streams, other host threads) race and give
 * wrong results; order them on one stream.  Otherwise the same arguments,
 * checks and results as moe_fp4_forward, with no optional outputs.  The
 * device error word lives in the internal array: moe_fp4_noalloc_check reads
 * it. */
#define MOE_FP4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int moe_fp4_forward_noalloc(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                            const uint8_t* w13, const uint8_t* w13_scale,
                            const uint8_t* w2, const uint8_t* w2_scale, float* out,
                            unsigned flags, void* cuda_stream);

/* moe_fp4_check for the internal array of moe_fp4_forward_noalloc:
 * synchronises the stream, reads the device error word left by the calls
 * enqueued before it (bits as in moe_fp4_check) and clears it.  Returns
 * MOE_FP4_OK, MOE_FP4_ERR_DEVICE or MOE_FP4_ERR_CUDA.  Allocates nothing. */
int moe_fp4_noalloc_check(void* cuda_stream);

/* MXFP8 quantisation of bf16 rows: the activation operand of a block-scaled
 * (MX) tensor-core product.  The paper quantises its decode activations
 * (abstract: INT8 activation quantisation) and the MI250 blog names
 * block-wise FP8 quantisation as the next gain; this is the MX form, with
 * the blocks of the weights (OCP Microscaling v1.0 conversion, E4M3 element).
 * For each 32 consecutive elements of a row, with amax their largest
 * magnitude:
 *   scale byte  s = floor(log2(amax)) - 8 + 127, at least 0; an all-zero
 *               block gets 0 (the scale is 2^(s-127));
 *   codes       E4M3 (OCP FP8 "FN": bias 7, no infinities, largest 448) of
 *               x / 2^(s-127), rounded to nearest even, saturated at +-448;
 *               a negative zero gives 0x80.
 * Layouts (row-major, device memory):
 *   x_bf16  bf16   [rows, K]      16-byte aligned; K a positive multiple of 32
 *   codes   uint8  [rows, K]      16-byte aligned; fully overwritten
 *   scales  uint8  [rows, K/32]   fully overwritten
 * The caller owns the buffers and the stream.  One kernel is enqueued; for
 * rows = 0 nothing is, and the pointers may be null.  The call never
 * synchronises.  Returns MOE_FP4_ERR_INVALID_ARG, with nothing enqueued, for
 * rows < 0, K not a positive multiple of 32, or (rows > 0) a null pointer or
 * a misaligned x_bf16 / codes; MOE_FP4_ERR_CUDA if the launch fails. */
int moe_fp4_mxfp8_quantize(const void* x_bf16, int64_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                           void* cuda_stream);

/* Workspace bytes of moe_fp4_forward_mx (256-byte aligned base); 0 for the
 * sizes moe_fp4_workspace_bytes rejects. */
size_t moe_fp4_mx_workspace_bytes(const moe_fp4_dims* dims);

/* The layer with MXFP8 activations into both projections, on block-scaled
 * tensor cores (tcgen05.mma kind::mxf8f6f4: the E2M1 weights and their E8M0
 * scales as stored, E4M3 activations with one E8M0 scale per 32 elements,
 * fp32 accumulation).  Steps as in moe_fp4_forward, with two quantisations
 * added (the MXFP8 conversion of moe_fp4_mxfp8_quantize):
 *   x_q = MXFP8(x) per token row (blocks of 32 along d) before W13;
 *   h   = bf16(silu(g) * u) as in moe_fp4_forward, then
 *   h_q = MXFP8(h) per slot row (blocks of 32 along I) before W2;
 *   y   = h_q . W2_e^T; out = sum_j w_j y_j.
 * The paper quantises its decode activations (abstract: INT8 activation
 * quantisation) and the MI250 blog names block-wise FP8 as the next gain;
 * this is that layer in the weights' own MX block format, not the exact
 * layer: out differs from moe_fp4_forward by the activation rounding.
 * Routing and the sort are those of moe_fp4_route, bit for bit.
 * Arguments as in moe_fp4_forward, except: w13 and w2 must be 32-byte
 * aligned; there are no flags; the optional outputs (NULL: kept in the
 * workspace only) are, in sorted-row order (S = T*k, row r = the r-th row of
 * the expert sort):
 *   h_bf16    bf16  [S, I]     16-byte aligned
 *   h_codes   uint8 [S, I]     E4M3 codes of h_q, 16-byte aligned
 *   h_scales  uint8 [S, I/32]  E8M0 scales of h_q
 *   x_codes   uint8 [S, d]     E4M3 codes of x_q of the row's token, 16-byte aligned
 *   x_scales  uint8 [S, d/32]  E8M0 scales of x_q
 * Enqueues the routing kernel, the quantising gather, the W13 projection,
 * the quantiser of h, the W2 projection and the combine; never synchronises.  A block of x or h that
 * holds an infinity or a NaN gets the NaN scale 0xFF and NaN codes, and the
 * rows it feeds come out NaN.
 * stage_events: NULL, or 6 cudaEvent_t handles recorded on the stream as in
 * moe_fp4_forward_profiled (before routing, after routing, after the
 * quantising gather, after W13, after the quantiser of h and W2, after the
 * combine). */
int moe_fp4_forward_mx(const moe_fp4_dims* dims, const void* x_bf16, const float* router_logits,
                       const uint8_t* w13, const uint8_t* w13_scale, const uint8_t* w2, const uint8_t* w2_scale,
                       float* out, void* h_bf16, uint8_t* h_codes, uint8_t* h_scales, uint8_t* x_codes,
                       uint8_t* x_scales, void* workspace, size_t workspace_bytes, void* cuda_stream,
                       void* const* stage_events);

/* Fault injection, for tests of the failure path only (the layer's own
 * failure handling: every pipeline wait in the kernels is bounded, and a wait
 * that runs out sets bit 2 of the device error word, releases the kernel's
 * other roles, lets every copy and MMA in flight finish, frees tensor memory
 * and returns).  While a site other than MOE_FP4_FAULT_NONE is set, every
 * later moe_fp4_forward* call in this process, from any thread, plants the
 * fault on the host's instruction, and every pipeline wait gives up after
 * wait_limit_us microseconds instead of 2 s:
 *   MOE_FP4_FAULT_TC_TOKEN_TILE   the tensor-core W13 kernel's first CTA never
 *                                 loads its first token tile (in
 *                                 moe_fp4_forward_mx: the block-scaled W13
 *                                 kernel's first CTA never loads its first
 *                                 stage);
 *   MOE_FP4_FAULT_STREAM_STAGE    the streaming W13 kernel's first CTA never
 *                                 loads its first weight stage.
 * Nothing faults, traps or hangs: the waiting threads give up, the outputs of
 * that call are incomplete, and moe_fp4_check reports MOE_FP4_ERR_DEVICE.
 * MOE_FP4_FAULT_NONE (wait_limit_us ignored) restores normal operation.
 * Returns MOE_FP4_ERR_INVALID_ARG for an unknown site or a zero limit. */
#define MOE_FP4_FAULT_NONE 0
#define MOE_FP4_FAULT_TC_TOKEN_TILE 1
#define MOE_FP4_FAULT_STREAM_STAGE 2
int moe_fp4_set_fault_injection(int site, uint32_t wait_limit_us);

/* Synchronises the stream and reads the device error word of the workspace,
 * which the kernels OR bits into: 1 = an index out of range (e.g. a corrupted
 * expert id, whose slot is dropped); 2 = a pipeline wait gave up after 2 s
 * (the kernel skipped the rest of its work, so the outputs are incomplete).
 * Returns MOE_FP4_OK, MOE_FP4_ERR_DEVICE or MOE_FP4_ERR_CUDA, and clears the
 * word. */
int moe_fp4_check(void* workspace, void* cuda_stream);

/* Static text for a status code. */
const char* moe_fp4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP4_H_ */
