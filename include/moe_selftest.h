/*
 * Self-test entry points of libroutedmoe: each runs one building block of the expert
 * kernel in isolation so that tests can check it against host-computed expectations.
 * They are not part of the layer; the paper has no counterpart for them.
 *
 * All pointers are device pointers owned by the caller; work is enqueued on `stream`.
 * Return values are moe_status codes (see moe.h).
 */
#ifndef ROUTED_MOE_SELFTEST_H
#define ROUTED_MOE_SELFTEST_H

#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* NVFP4 decode as used by the dequantisation warps.
 *   words     [n] uint32: eight E2M1 codes each (element 2i in the low nibble of byte i)
 *   out       [4n] uint32: hardware conversion, f16x2 out[4w + b] = (element 2b, element 2b+1)
 *   pairs     [m] uint32: two E4M3 bytes in the low 16 bits (low byte -> low half)
 *   sout      [m] uint32: f16x2 of the two scale values */
MOE_API int moe_selftest_decode(const uint32_t* words, int n, uint32_t* out, const uint32_t* pairs, int m,
                                uint32_t* sout, moe_stream_t stream);

/* One TMA load of a 64-byte x 64-row box of a [rows, row_bytes] uint8 matrix at byte
 * column x (a multiple of 16) and row y, with the 64-byte swizzle the expert kernel
 * uses; out [4096] receives the raw shared-memory image. */
MOE_API int moe_selftest_tma(const uint8_t* src, int rows, int row_bytes, int x, int y, uint8_t* out,
                             moe_stream_t stream);

/* One 128 x 16 x 128 product on the tensor core the way the expert kernel issues it:
 * A [128, 128] FP16 (row-major) written to tensor memory by 128 threads, B [16, 128]
 * FP16 (row-major) stored in shared memory in 128-byte swizzled K-major atoms, eight
 * kind::f16 MMAs with FP32 accumulation, result D [128, 16] FP32 (row-major) = A B^T. */
MOE_API int moe_selftest_mma(const void* A, const void* B, float* D, moe_stream_t stream);

/* The expert kernel and the un-route kernel exactly as moe_forward_experts runs them with
 * MOE_ALGO_AUTO (after moe_plan and moe_forward_prepare), with a timeline recorded into
 * `trace`: per CTA 8 roles x 1024 uint64 events (event code << 56 | index << 40 | low 40
 * bits of %globaltimer in ns); zero-initialise the buffer (multiProcessorCount x 65536 bytes).
 * Warp-MMA kernel: role 0 weight producer (1 task published, 2 chunk issued), 1 activation
 * producer (3 readiness met, 4 chunk issued), 2 and 3 first and last compute warp (5 task
 * taken, index bit 15 = down task; 6 chunks done; 12 un-route wait begins, 13 wait met),
 * 4 publisher (9 task released), 5 CTA (10 start, 11 end).  Decode kernel for at most eight
 * tokens: as the warp-MMA kernel, with role 1 event 3 = a down task's h rows requested, role 2
 * events 7 / 8 = a barrier round of two chunks begins / its data has landed, role 5 event 14 =
 * kernel entry (before the wait for the preceding kernel).  tcgen05 kernel: roles 0 and 1 as
 * above, 2 first dequantisation warp (5 chunk landed, 6 chunk in tensor memory), 3 MMA (7 chunk issued),
 * 4 epilogue (8 accumulator ready, 9 task done), 5 CTA (10 start, 11 end). */
MOE_API int moe_selftest_expert_trace(const moe_shape* shape, const uint8_t* w13_codes,
                                      const uint8_t* w13_scales, float w13_scale,
                                      const uint8_t* w2_codes, const uint8_t* w2_scales,
                                      float w2_scale, const void* residual, void* out,
                                      void* workspace, size_t workspace_bytes,
                                      unsigned long long* trace, moe_stream_t stream);

/* moe_layer with the same timeline as moe_selftest_expert_trace recorded by its expert
 * kernel.  For T <= 8 that is the one-launch layer, whose prologue routes and plans: role 5
 * event 10 is then taken after that prologue, and it adds role 6 events 16 (token 0 routed),
 * 18 (routes in shared memory), 19 (route positions done), role 7 event 17 (hidden rows
 * converted), and role 0 events 20 (first task entry and tokens known), 21 (first task slot
 * free), 22 / 23 (before / after the first weight copy is issued). */
MOE_API int moe_selftest_layer_trace(const moe_shape* shape, const float* logits, const void* hidden,
                                     const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                                     const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                     const void* residual, void* out, int32_t* ids, float* weights,
                                     void* workspace, size_t workspace_bytes, unsigned long long* trace,
                                     moe_stream_t stream);

/* The failure path of the expert kernels' bounded waits, for tests.  After moe_front (or
 * moe_route_topk + moe_plan + moe_forward_prepare) has left a plan in `workspace`, the down task
 * number `dn_task` of the table the chosen kernel reads is rewritten to wait for the readiness
 * counter of a touched-expert index that no gate/up task publishes (U, one past the last
 * touched expert, which needs U < E); then the expert kernel and the un-route run as
 * moe_forward_experts(algo) does, with every bounded wait limited to `wait_limit_cycles`
 * clock cycles (the library's own limit is 2^33).  The wait that cannot be met gives up, the
 * CTA sets MOE_DEV_TIMEOUT in the workspace status word and stops, its roles drain the copies
 * they started (tensor memory is released in the tcgen05 kernels), and the other CTAs stop in
 * turn when they wait for work the stopped CTA had claimed: the launch completes, outputs are
 * undefined.  The plan must be rebuilt before the workspace is used again (moe_front or
 * moe_plan).  Blocking: synchronises `stream` to read and rewrite the table entry.
 *   algo: MOE_ALGO_AUTO, MOE_ALGO_MMA, MOE_ALGO_TCGEN05 or MOE_ALGO_WIDE.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (no such down task, U == E, algo MOE_ALGO_SIMT, limit
 * not positive) or another moe_status. */
MOE_API int moe_selftest_expert_timeout(const moe_shape* shape, const uint8_t* w13_codes,
                                        const uint8_t* w13_scales, float w13_scale,
                                        const uint8_t* w2_codes, const uint8_t* w2_scales,
                                        float w2_scale, const void* residual, void* out,
                                        void* workspace, size_t workspace_bytes, int algo, int dn_task,
                                        long long wait_limit_cycles, moe_stream_t stream);

/* moe_forward_expert_kernels in two parts, so that the expert kernel can be timed alone:
 * part 0 launches the kernels that prepare its input (for MOE_ALGO_WIDE, or AUTO choosing
 * it: the hidden rows gathered into route order and the wide kernel's task table; nothing
 * for the other kernels), part 1 the expert kernel itself, which reads what part 0 left in the
 * workspace.  Part 0 followed by part 1 on the same stream equals moe_forward_expert_kernels.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (part not 0 or 1) or another moe_status. */
MOE_API int moe_selftest_expert_part(const moe_shape* shape, const uint8_t* w13_codes,
                                     const uint8_t* w13_scales, float w13_scale,
                                     const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                     void* workspace, size_t workspace_bytes, int algo, int part,
                                     moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ROUTED_MOE_SELFTEST_H */
