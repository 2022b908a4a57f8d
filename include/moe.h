/*
 * libroutedmoe: routed mixture-of-experts layer for speculative-decode verify steps and
 * prefill chunks on GB300 (sm_103a).  C ABI over plain pointers; no C++ or torch types.
 *
 * The layer (token t, hidden x_t in BF16, router logits l_t in FP32):
 *   1. router   p = softmax(l_t) over E experts; the k largest logits are selected
 *               (larger first, equal values -> lower expert index); the selected
 *               probabilities are renormalised to sum to one.
 *   2. experts  for each selected expert e with weight w:
 *                 g = x W13[e][0:F]^T,  u = x W13[e][F:2F]^T,  h = silu(g) * u,
 *                 y = h W2[e]^T
 *   3. un-route out_t = residual_t + sum_{j<k} w_j y_j   (slots summed in order, BF16 out)
 * Expert weights are NVFP4: E2M1 codes (two per byte, element 2i in the low nibble),
 * one E4M3 scale per 16 consecutive elements along the reduction dimension, and one
 * FP32 scale per tensor.
 *
 * Passages that define the operations (pages on the Qwen3.8-Flash-Next MoE path):
 *   - "How I forked vLLM and made Qwen3.8-Flash-Next decode 1.6x faster on one GPU":
 *     section "The model and the constraint" (512 experts, top-10, NVFP4 experts) and
 *     section "5. Hand-written kernels", paragraph "Fused MoE routing" (warp-per-token
 *     softmax, top-k arg-max on float keys, lowest id wins ties, counts / scan /
 *     scatter of routes to experts).
 *   - "Persistent execution for Flash-Next GGUF on SM70": section "First implementation
 *     boundary" (router GEMV outside the boundary; compact expert-presence list with
 *     route positions; workers over (expert, output stripe) tasks that load each
 *     expert's weights once; gate/up with SiLU*multiply publishing per-expert
 *     readiness; down fused with the weighted unroute, routes summed in a fixed order,
 *     no arrival-ordered float atomics); section "MonoMoE" (precomputed router logits
 *     are the input; explicit ordering, valid zero intermediates, deterministic output
 *     reduction); the paragraph on epoch/workspace ownership under graph replays.
 *   - "How I forked vLLM ...", section "5. Hand-written kernels", paragraph "PDL
 *     weight-prefetch GEMV": fixed-size workspace that CUDA graphs never see replaced.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major, 16-byte aligned, owned by the
 *     caller; the library allocates no device memory and keeps no per-call state
 *     outside the caller's workspace (only a read-only per-device property cache).
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream); no
 *     host synchronisation, no device-to-host copy, no host-visible size depends on
 *     data, so every call can be captured in a CUDA graph.
 *   - Host-detectable errors (null pointers, unsupported shapes, misalignment, a
 *     workspace that is too small) return a negative moe_status before anything is
 *     enqueued.  Device-detected conditions (an expert id out of range, a bounded wait
 *     that gave up, hidden values outside FP16 range, an FP16 intermediate that
 *     saturated) are OR-ed into a status word inside the workspace; read it with
 *     moe_read_device_status after synchronising the stream.
 *   - Calls on distinct workspaces may run concurrently; calls sharing a workspace
 *     must be ordered on one stream.
 */
#ifndef ROUTED_MOE_H
#define ROUTED_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2, /* shape outside what the kernels implement (see moe_shape) */
  MOE_ERR_WORKSPACE = -3,   /* workspace null, misaligned or smaller than moe_workspace_bytes */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (no device, launch error) */
  MOE_ERR_DEVICE = -5       /* moe_read_device_status found device-side error bits */
} moe_status;

/* Device status bits (OR-ed into the workspace status word by kernels). */
#define MOE_DEV_BAD_EXPERT_ID 0x1u  /* a routing id was outside [0, E) in moe_plan */
#define MOE_DEV_TIMEOUT 0x2u        /* a bounded wait in the expert kernel gave up */
#define MOE_DEV_HIDDEN_RANGE 0x4u   /* |hidden| exceeded the FP16 range (65504) */
#define MOE_DEV_H_SATURATED 0x8u    /* |silu(g)*u| exceeded 2^4 * 65504 and was clamped */
#define MOE_DEV_Y_SATURATED 0x10u   /* MOE_ALGO_WIDE: a per-route down output exceeded 2^4 * 65504
                                       and was clamped */

/* Layer shape.  T tokens (rows of the call), d hidden size, ffn expert intermediate
 * size, E experts, k experts per token.  Supported: 1 <= T <= 65536, 1 <= k <= 32,
 * k <= E <= 1024, d % 128 == 0, ffn % 128 == 0, 128 <= d <= 16384, 128 <= ffn <= 8192. */
typedef struct moe_shape {
  int32_t T, d, ffn, E, k;
} moe_shape;

/* Expert-kernel selection for moe_forward_algo. */
typedef enum moe_algo {
  MOE_ALGO_AUTO = 0,     /* MOE_ALGO_WIDE when the routes average at least 32 rows per expert
                            (T * k >= 32 * E, e.g. prefill chunks), else MOE_ALGO_MMA where it
                            applies (d and ffn powers of two from 256 to 2048), else
                            MOE_ALGO_TCGEN05 */
  MOE_ALGO_TCGEN05 = 1,  /* persistent stripe kernel: TMA weight stream, in-register NVFP4
                            dequantisation into tensor memory, tcgen05 MMA (FP32 accumulate),
                            16-row column groups, readiness counters between gate/up and down */
  MOE_ALGO_SIMT = 2,     /* CUDA-core kernels, one launch per stage (ablation baseline) */
  MOE_ALGO_MMA = 3,      /* persistent stripe kernel: TMA weight stream, in-register NVFP4
                            dequantisation into the A fragments of warp-level m16n8k16 tensor-core
                            MMAs (weights stationary, routed rows as the 8-wide operand, FP32
                            accumulate), gate and up of one F index in one warp, readiness
                            counters between gate/up and down; needs d and ffn powers of two from
                            256 to 2048 (MOE_ERR_UNSUPPORTED otherwise) */
  MOE_ALGO_WIDE = 4      /* persistent stripe kernel for many routed rows per expert (prefill
                            chunks): as MOE_ALGO_TCGEN05, but up to 192 routed rows per weight
                            pass in one tcgen05 MMA per 16-element K step (N = rows rounded up
                            to 16), two tensor-memory accumulators so that a task's epilogue
                            overlaps the next task's MMAs */
} moe_algo;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_string(int status);

/* Message of the last failed CUDA call made by this library on the calling host thread
 * (empty string if none).  Static thread-local storage, never NULL. */
MOE_API const char* moe_last_cuda_error(void);

/* Bytes of device workspace needed for `shape` (0 if the shape is unsupported).
 * The workspace holds the routing plan, per-call counters, the FP16 copy of the
 * hidden rows, the gate/up intermediate, per-route down outputs and the status word.
 * It must be 256-byte aligned.  Pure host function: needs no GPU. */
MOE_API size_t moe_workspace_bytes(const moe_shape* shape);

/* Zero the status block and the decode kernel's two counter sets (the first 8960 bytes, or
 * all of a smaller buffer) of a freshly allocated workspace (enqueued on `stream`).  Call
 * once after allocation; every other field is (re)written by moe_plan / moe_forward, and the
 * counter sets are left zeroed by every call that uses them. */
MOE_API int moe_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Check a shape without touching the GPU: MOE_OK, MOE_ERR_INVALID_ARG or
 * MOE_ERR_UNSUPPORTED. */
MOE_API int moe_check_shape(const moe_shape* shape);

/* The expert kernel MOE_ALGO_AUTO selects for a shape (MOE_ALGO_WIDE, MOE_ALGO_MMA or
 * MOE_ALGO_TCGEN05),
 * or a negative status when the shape is invalid.  Pure host function: needs no GPU. */
MOE_API int moe_auto_algo(const moe_shape* shape);

/* 1 if moe_forward_experts / moe_forward_algo / moe_layer with `algo` run the weighted
 * un-route inside the expert kernel (the decode kernel does so for T <= 8: trailing
 * un-route tasks that wait for the down tasks of their 128-column stripe), 0 if it runs as
 * a kernel of its own after the expert kernel, or a negative status for an invalid shape
 * or algo.  The two give identical bits.  Pure host function: needs no GPU. */
MOE_API int moe_unroute_fused(const moe_shape* shape, int algo);

/* Number of kernel launches one moe_layer call makes for `shape` (1 for the one-launch
 * layer of at most eight tokens), or a negative status for an invalid shape.  Pure host
 * function: needs no GPU. */
MOE_API int moe_layer_launches(const moe_shape* shape);

/* Step 1, router ("Fused MoE routing"; "Router: selection and expert-task production").
 *   logits  [T, E]  float32, finite values (non-finite logits are outside the contract)
 *   ids     [T, k]  int32 out: selected experts in selection order (value desc, ties to
 *                   the lower index; -0 and +0 compare equal)
 *   weights [T, k]  float32 out: renormalised softmax probabilities of the selection
 * One warp per token. */
MOE_API int moe_route_topk(const moe_shape* shape, const float* logits, int32_t* ids, float* weights,
                   moe_stream_t stream);

/* Step 2, bucketing ("First implementation boundary", step 1): per-expert route counts,
 * their exclusive prefix sum, the ascending list of touched experts, each route's
 * position in expert-major order, the per-expert task prefix sums used by the expert
 * kernel, and a copy of the routing weights, all written into `workspace`.
 *   ids     [T, k] int32, values in [0, E) (violations set MOE_DEV_BAD_EXPERT_ID)
 *   weights [T, k] float32
 * One 1024-thread CTA for T * k up to 16384 routes; above that three launches (per-slice
 * histograms of 4096 routes, one scan CTA, per-slice positions).  The order of the routes
 * inside one expert's bucket is not fixed (results do not depend on it).
 * Must precede every moe_forward whose routing changed. */
MOE_API int moe_plan(const moe_shape* shape, const int32_t* ids, const float* weights, void* workspace,
             size_t workspace_bytes, moe_stream_t stream);

/* Steps 3-4, experts and un-route, using the plan in `workspace`:
 *   hidden     [T, d]          BF16, |values| <= 65504
 *   w13_codes  [E, 2*ffn, d/2] uint8 E2M1 pairs; rows [0, ffn) gate, [ffn, 2*ffn) up
 *   w13_scales [E, 2*ffn, d/16] uint8 E4M3 block scales
 *   w13_scale  FP32 tensor scale of W13
 *   w2_codes   [E, d, ffn/2]   uint8 E2M1 pairs
 *   w2_scales  [E, d, ffn/16]  uint8 E4M3 block scales
 *   w2_scale   FP32 tensor scale of W2
 *   residual   [T, d] BF16 or NULL (treated as zero)
 *   out        [T, d] BF16; may alias residual (each element is read before written)
 * Every moe_forward re-zeroes the counters it uses, so it may be repeated on one plan.
 * moe_forward is moe_forward_algo(..., MOE_ALGO_AUTO). */
MOE_API int moe_forward(const moe_shape* shape, const void* hidden, const uint8_t* w13_codes,
                const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes,
                const uint8_t* w2_scales, float w2_scale, const void* residual, void* out,
                void* workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API int moe_forward_algo(const moe_shape* shape, const void* hidden, const uint8_t* w13_codes,
                     const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes,
                     const uint8_t* w2_scales, float w2_scale, const void* residual, void* out,
                     void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream);

/* The two halves of moe_forward_algo, for callers that schedule them separately:
 * moe_forward_prepare zeroes the counters of the call and stages `hidden` as FP16 in the
 * workspace (one small kernel); moe_forward_experts runs the expert kernel(s) on that
 * staging and the plan.  Arguments as for moe_forward_algo. */
MOE_API int moe_forward_prepare(const moe_shape* shape, const void* hidden, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream);
MOE_API int moe_forward_experts(const moe_shape* shape, const uint8_t* w13_codes,
                                const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes,
                                const uint8_t* w2_scales, float w2_scale, const void* residual,
                                void* out, void* workspace, size_t workspace_bytes, int algo,
                                moe_stream_t stream);

/* moe_forward_experts in two launches' worth of parts, for callers that want to time or
 * schedule them apart: moe_forward_expert_kernels runs only the expert kernel(s) (gate/up,
 * SiLU·mul, down projection into the per-route outputs of the workspace: FP32, or
 * FP16(y * 2^-4) from MOE_ALGO_WIDE, recorded in the plan for the un-route);
 * moe_forward_unroute runs only the weighted un-route (out = residual + the token's routes
 * in slot order, "fuses down with weighted unroute" in "Persistent execution for
 * Flash-Next GGUF on SM70").  Arguments as for moe_forward_experts. */
MOE_API int moe_forward_expert_kernels(const moe_shape* shape, const uint8_t* w13_codes,
                                       const uint8_t* w13_scales, float w13_scale,
                                       const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                       void* workspace, size_t workspace_bytes, int algo,
                                       moe_stream_t stream);
MOE_API int moe_forward_unroute(const moe_shape* shape, const void* residual, void* out, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/* Steps 1-2 together with moe_forward_prepare's staging: the router (ids/weights written
 * to the caller's [T, k] buffers), the plan in `workspace`, the FP16 copy of `hidden` and
 * the reset of the expert kernel's counters.  For T * k up to 16384 this is one fused
 * launch (the last CTA to finish routing builds the plan); larger batches run
 * moe_route_topk + moe_plan + moe_forward_prepare.  Afterwards moe_forward_experts (or
 * moe_forward_expert_kernels + moe_forward_unroute) completes the layer.  Arguments as for
 * moe_route_topk, moe_plan and moe_forward_prepare; returns MOE_OK or an error code. */
MOE_API int moe_front(const moe_shape* shape, const float* logits, const void* hidden, int32_t* ids,
                      float* weights, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Whole layer: router, plan and forward on one stream, with ids/weights written to the
 * caller's [T, k] buffers.  For T <= 8 (T * k <= 256, E <= 1024) where MOE_ALGO_AUTO picks
 * the warp-MMA decode kernel, the whole layer is ONE launch: every CTA of the decode kernel
 * routes the T tokens and builds the plan in shared memory before its weight stream starts
 * (results identical to the split steps), and the routing, the plan and the FP16 hidden rows
 * are still written into the workspace for later calls.  Otherwise, for T * k up to 16384
 * the router, the FP16 staging of hidden and the plan run as one fused launch (moe_front),
 * and moe_layer is moe_front followed by moe_forward_experts with MOE_ALGO_AUTO.  Where the
 * expert kernel that MOE_ALGO_AUTO picks does not read the plan's task table (the decode
 * kernel above eight tokens, the wide kernel), the layer leaves the table unwritten and its
 * task counts at 0: a later moe_forward_experts on that plan must use MOE_ALGO_AUTO (another
 * algorithm would find no tasks). */
MOE_API int moe_layer(const moe_shape* shape, const float* logits, const void* hidden,
              const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
              const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
              const void* residual, void* out, int32_t* ids, float* weights, void* workspace,
              size_t workspace_bytes, moe_stream_t stream);

/* Expert-parallel shard of moe_layer: the layer restricted to the experts [e_begin, e_end),
 * for a deployment that splits the experts over GPUs ("TokenSpeed: Qwen3.8-Flash-Next
 * optimisations", section on the benchmark settings: expert parallelism of 4 on 4x GB300).
 * Routing runs over all E experts (ids/weights as moe_layer, identical on every shard); only
 * the routes to local experts are planned and computed, so
 *     out = residual + sum over the token's slots j with e_begin <= id_j < e_end of w_j y_j,
 * slots in order, FP32, one BF16 rounding.  Summing the shards' outputs (residual passed to
 * one shard only, NULL to the others) gives the layer up to those per-shard roundings.
 *   w13_codes/w13_scales/w2_codes/w2_scales hold the local experts only: entry e - e_begin
 *   is expert e ([e_end - e_begin, 2*ffn, d/2] and so on).
 * Other arguments, ownership and errors as moe_layer; 0 <= e_begin < e_end <= E, else
 * MOE_ERR_INVALID_ARG.  The range is an argument of this call only: nothing is kept
 * between calls. */
MOE_API int moe_layer_expert_range(const moe_shape* shape, int e_begin, int e_end, const float* logits,
                                   const void* hidden, const uint8_t* w13_codes, const uint8_t* w13_scales,
                                   float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales,
                                   float w2_scale, const void* residual, void* out, int32_t* ids,
                                   float* weights, void* workspace, size_t workspace_bytes,
                                   moe_stream_t stream);

/* moe_layer_expert_range as a plan / forward pair, for expert-parallel callers that run
 * the router themselves (moe_route_topk) and schedule the steps apart:
 *   moe_plan_expert_range             moe_plan restricted to the experts [e_begin, e_end):
 *                                     routes to other experts get no position and add
 *                                     nothing;
 *   moe_forward_experts_expert_range  moe_forward_experts on that plan with the local
 *                                     weights (entry e - e_begin holds expert e).
 * moe_forward_prepare stages the hidden rows in between, as for the full layer.  Both
 * calls of one layer must be given the same range (the plan holds positions for the local
 * experts only; the expert kernels index the local weights by e - e_begin).  Arguments,
 * ownership and errors as moe_plan / moe_forward_experts; 0 <= e_begin < e_end <= E, else
 * MOE_ERR_INVALID_ARG. */
MOE_API int moe_plan_expert_range(const moe_shape* shape, int e_begin, int e_end, const int32_t* ids,
                                  const float* weights, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream);
MOE_API int moe_forward_experts_expert_range(const moe_shape* shape, int e_begin, int e_end,
                                             const uint8_t* w13_codes, const uint8_t* w13_scales,
                                             float w13_scale, const uint8_t* w2_codes,
                                             const uint8_t* w2_scales, float w2_scale, const void* residual,
                                             void* out, void* workspace, size_t workspace_bytes, int algo,
                                             moe_stream_t stream);

/* moe_layer with one FP32 tensor scale per expert for each weight tensor instead of one for
 * all experts: expert e's W13 is scaled by w13_scales_e[e] and its W2 by w2_scales_e[e]
 * (device arrays of E floats; NVFP4 checkpoints that quantise each expert separately carry
 * such per-expert global scales).  Other arguments, ownership and errors as moe_layer. */
MOE_API int moe_layer_expert_scales(const moe_shape* shape, const float* logits, const void* hidden,
                                    const uint8_t* w13_codes, const uint8_t* w13_scales, const float* w13_scales_e,
                                    const uint8_t* w2_codes, const uint8_t* w2_scales, const float* w2_scales_e,
                                    const void* residual, void* out, int32_t* ids, float* weights,
                                    void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Router projection, the producer of the router logits ("Persistent execution for Flash-Next
 * GGUF on SM70", section "Router: selection and expert-task production": the projection whose
 * results the selection consumes, with an explicit hand-off to the final producer):
 *   logits[t][e] = sum_c hidden[t][c] * router_w[e][c]   (BF16 inputs, FP32 sums)
 *   hidden   [T, d] BF16;  router_w [E, d] BF16 (row e = expert e);  logits [T, E] FP32 out.
 * Written as the weight-prefetch GEMV of "How I forked vLLM and made Qwen3.8-Flash-Next decode
 * 1.6x faster on one GPU" (section 5, paragraph "PDL weight-prefetch GEMV"): each CTA copies its
 * 16 router-weight rows into shared memory before it waits for the preceding kernel in the
 * stream, so under programmatic dependent launch the weights stream while that kernel (the
 * previous layer) finishes; the partial sums of its four K quarters are added in a fixed order
 * (no atomics), so the logits, and the routing, are the same on every run.  Supported: E a
 * multiple of 16, d a multiple of 64 up to 4096.  MOE_ERR_UNSUPPORTED otherwise. */
MOE_API int moe_router_logits(const moe_shape* shape, const void* hidden, const void* router_w, float* logits,
                              moe_stream_t stream);

/* moe_router_logits followed by moe_layer on its logits: the layer from the hidden states and
 * the router weight.  `logits` [T, E] FP32 is the caller's buffer for the projection (also an
 * output).  Other arguments, ownership and errors as moe_layer. */
MOE_API int moe_layer_from_hidden(const moe_shape* shape, const void* hidden, const void* router_w, float* logits,
                                  const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                                  const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                  const void* residual, void* out, int32_t* ids, float* weights, void* workspace,
                                  size_t workspace_bytes, moe_stream_t stream);

/* Gated residual update and the next normalisation, in place of the plain un-route, for a
 * model whose residual stream has G branches ("TokenSpeed: Qwen3.8-Flash-Next optimisations",
 * section "Residual update and normalization fusion").  With O[t] = sum_j w_{t,j} y_{t,j} the
 * token's weighted routes (slots in order, FP32, from the per-route outputs that
 * moe_forward_expert_kernels left in `workspace`), for every token t and branch g < G:
 *   residual_out[g][t] = BF16(residual[g][t] + 2 sigmoid(inject_logits[t][g]) O[t])
 *   normed_out[g][t]   = GemmaRMSNorm(residual_out[g][t], norm_weight[g])
 *   GemmaRMSNorm(x, w)_c = x_c / sqrt(mean_c(x_c^2) + eps) * (1 + w_c)
 * The normalisation reads the updated residual after its rounding to BF16 (kept on chip; both
 * outputs are stored).  One CTA per token.
 *   residual      [G, T, d] BF16 (16-byte aligned)
 *   inject_logits [T, G]    FP32
 *   norm_weight   [G, d]    BF16
 *   eps           >= 0 (the pages give none; Gemma's own is 1e-6)
 *   residual_out  [G, T, d] BF16, may alias residual;  normed_out [G, T, d] BF16
 * Supported: 1 <= G <= 8, d <= 4096 (MOE_ERR_UNSUPPORTED otherwise).  Errors as moe_forward. */
MOE_API int moe_forward_unroute_gated(const moe_shape* shape, int G, const void* residual,
                                      const float* inject_logits, const void* norm_weight, float eps,
                                      void* residual_out, void* normed_out, void* workspace,
                                      size_t workspace_bytes, moe_stream_t stream);

/* Whole layer with the gated epilogue: moe_front, moe_forward_expert_kernels (MOE_ALGO_AUTO) and
 * moe_forward_unroute_gated.  Arguments as those calls; ids/weights as moe_layer. */
MOE_API int moe_layer_gated(const moe_shape* shape, int G, const float* logits, const void* hidden,
                            const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                            const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                            const void* residual, const float* inject_logits, const void* norm_weight, float eps,
                            void* residual_out, void* normed_out, int32_t* ids, float* weights, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/* The whole layer (moe_layer) with its scratch in a fixed device array of the library
 * instead of a caller-provided workspace.  The pages have no counterpart for this entry
 * point.  It is for callers that cannot allocate device memory: code running while a
 * CUDA graph is being captured (cudaMalloc is not capturable), plug-ins whose host
 * framework owns all device memory through its own allocator, and latency-critical
 * loops where cudaMalloc's implicit device synchronisation is not acceptable.  Such
 * callers still pass every input and output (logits, hidden, weights, residual, out,
 * ids, weights) exactly as for moe_layer; this call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine).
 *   - Scratch: a file-scope 16 MiB (16777216-byte) device array in the library, present
 *     on every GPU that loads the library until the process exits.  Shapes with
 *     moe_workspace_bytes(shape) larger than that return MOE_ERR_WORKSPACE (with a
 *     message in moe_last_cuda_error); this covers the decode-verify shapes (e.g.
 *     T = 4 or 32 with d = 2048, ffn = 512, E = 512, k = 10), not large prefill chunks.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before any
 *     stream capture.  The address is kept for the life of the process and belongs to the
 *     device's primary context: do not use this entry point after cudaDeviceReset or from
 *     another context on the same device.
 *   - Sharing: every call uses the same array and leaves its contents behind; the call
 *     clears what must start at zero (status word, counters) itself.  Calls whose work
 *     overlaps on the GPU (different streams, or several host threads) race on the
 *     array: serialise them.  Device-side status bits are not returned by this call; read
 *     them with moe_static_workspace_read_status after it.
 * Returns as moe_layer. */
MOE_API int moe_layer_static_workspace(const moe_shape* shape, const float* logits,
                                       const void* hidden, const uint8_t* w13_codes,
                                       const uint8_t* w13_scales, float w13_scale,
                                       const uint8_t* w2_codes, const uint8_t* w2_scales,
                                       float w2_scale, const void* residual, void* out,
                                       int32_t* ids, float* weights, moe_stream_t stream);

/* The device status word of moe_layer_static_workspace's array, as moe_read_device_status
 * reads a caller workspace's: blocking copy on `stream`, cleared when `clear` is non-zero,
 * MOE_OK if no bit is set, MOE_ERR_DEVICE if any is.  Each static call starts by clearing
 * the word, so read it after a call and before the next. */
MOE_API int moe_static_workspace_read_status(int clear, uint32_t* status_bits, moe_stream_t stream);

/* Copy the device status word to *status_bits (blocking copy on `stream`; call after the
 * work of interest has been enqueued) and clear it when `clear` is non-zero.  Returns
 * MOE_OK if no bit is set, MOE_ERR_DEVICE if any is. */
MOE_API int moe_read_device_status(const void* workspace, int clear, uint32_t* status_bits,
                           moe_stream_t stream);

/* Read back the plan summary: number of touched experts U and the largest per-expert
 * row count (blocking copy on `stream`; diagnostic use, e.g. for byte accounting). */
MOE_API int moe_plan_summary(const moe_shape* shape, const void* workspace, int32_t* touched_experts,
                     int32_t* max_rows, moe_stream_t stream);

/* Device-side plan arrays inside the workspace, for tests: pointers to counts [E],
 * offsets [E+1], touched [E] (first U valid), route_pos [T*k] (position of route
 * t*k+j in expert-major order) and pos_token [T*k].  Returns MOE_OK or an error. */
MOE_API int moe_plan_views(const moe_shape* shape, void* workspace, int32_t** counts, int32_t** offsets,
                   int32_t** touched, int32_t** route_pos, int32_t** pos_token);

#ifdef __cplusplus
}
#endif

#endif /* ROUTED_MOE_H */
