/*
 * CPU oracle for the routed mixture-of-experts layer (softmax router, top-k with
 * renormalised weights, NVFP4 gate/up + SiLU*mul, NVFP4 down projection, weighted
 * un-route into a BF16 residual).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * code; it exists so that tests, the smoke check and the CPU baseline of the bench
 * can check the CUDA path against a plain, slow, obviously correct implementation.
 * It shares no code, header, table or constant with the CUDA sources.
 *
 * Precision: the layer is specified as "dequantise NVFP4 to FP32 and compute in
 * FP32"; every function therefore exists in an FP32 form (the parity reference) and
 * an FP64 shadow form built from the same template, used to bound the FP32 form's
 * own rounding error.
 *
 * Sources (pages on the Qwen3.8-Flash-Next routed MoE path):
 *  - "How I forked vLLM and made Qwen3.8-Flash-Next decode 1.6x faster on one GPU",
 *    section "5. Hand-written kernels", paragraph "Fused MoE routing": softmax per
 *    token, top-k by arg-max on float keys, lowest expert id wins ties, routing that
 *    matches the reference exactly.  Section "The model and the constraint": 512
 *    experts, top-10, NVFP4 experts.
 *  - "Persistent execution for Flash-Next GGUF on SM70", section "Router: selection
 *    and expert-task production": repeated maxima in a warp, ties to the lowest
 *    expert index, selection plus normalisation; section "First implementation
 *    boundary": compact expert-presence list, fused gate/up with SiLU/multiply, down
 *    fused with the weighted unroute, routes summed in a fixed order.
 *  - "TokenSpeed: Qwen3.8-Flash-Next optimisations", section "Residual update and
 *    normalization fusion": R' = R + 2 sigmoid(a) O per residual branch, then
 *    GemmaRMSNorm(R', w) of the consuming mixer, the residual rounded to its storage type
 *    before the normalisation reads it.
 *  - NVFP4 bit formats: the pages only name "NVFP4"; the element format follows the
 *    OCP Microscaling (MX) v1.0 definitions of E2M1 (FP4, exponent bias 1, no
 *    inf/NaN) and E4M3 (FP8, bias 7, no infinities, S.1111.111 = NaN), with one E4M3
 *    scale per 16 consecutive elements and one FP32 tensor scale.
 *
 * All arrays are host memory, row-major, owned by the caller.  BF16 tensors are
 * passed as uint16 bit patterns.  Functions never allocate visible state and report
 * invalid arguments by returning a negative value.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* E2M1 value of the low 4 bits of `nibble` (sign bit 3, exponent bits 2..1, mantissa bit 0). */
float oracle_e2m1_value(uint32_t nibble);

/* E4M3 value of `byte` (sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0);
 * exponent 0 is subnormal 2^-6 * m/8; 0x7F / 0xFF decode to NaN. */
float oracle_e4m3_value(uint32_t byte);

/* Dequantised weight row: out[c] = E2M1(code nibble c) * E4M3(scale[c/16]) * tensor_scale
 * for c < K.  `codes` holds K/2 bytes (element 2i in the low nibble of byte i). */
int oracle_dequant_row(const uint8_t* codes, const uint8_t* scales, float tensor_scale,
                       int K, float* out);

/* Router: for every token t < T, softmax over the E logits, the k largest logits
 * (larger first, equal values -> lower index, -0 == +0), and the selected
 * probabilities renormalised to sum to one.  ids/weights are [T, k] in selection
 * order.  Returns 0, or -1 on invalid sizes. */
int oracle_route_topk_f32(int T, int E, int k, const float* logits, int32_t* ids, float* weights);
int oracle_route_topk_f64(int T, int E, int k, const float* logits, int32_t* ids, double* weights);

/* Bucketing: counts[e] = number of routes to expert e, offsets[0..E] their exclusive
 * prefix sum, touched[0..U) the experts with counts > 0 in ascending order.  Returns U,
 * or -1 on invalid input (an id outside [0, E)). */
int oracle_plan(int T, int E, int k, const int32_t* ids, int32_t* counts, int32_t* offsets,
                int32_t* touched);

/* The expert part of the layer for the tokens t with token_mask[t] != 0 (all tokens if
 * token_mask is NULL):
 *   g = x W13[e][0:F]^T, u = x W13[e][F:2F]^T, h = silu(g) * u, y = h W2[e]^T,
 *   out[t] = residual[t] + sum_j weights[t][j] * y_{t,j}   (j = 0..k-1 in slot order)
 * with weights dequantised to the accumulation type and every sum in ascending index
 * order.  `residual` may be NULL (treated as zero).  out is [T, d] in the accumulation
 * type; rows of unmasked tokens are left untouched.  Returns 0, or -1 on bad input. */
int oracle_moe_experts_f32(int T, int d, int F, int E, int k,
                           const uint16_t* hidden_bf16, const int32_t* ids, const float* weights,
                           const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_ts,
                           const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_ts,
                           const uint16_t* residual_bf16, const uint8_t* token_mask, float* out);
int oracle_moe_experts_f64(int T, int d, int F, int E, int k,
                           const uint16_t* hidden_bf16, const int32_t* ids, const double* weights,
                           const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_ts,
                           const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_ts,
                           const uint16_t* residual_bf16, const uint8_t* token_mask, double* out);

/* BF16 bit pattern of `x`, round to nearest, ties to even (NaN stays NaN). */
uint16_t oracle_bf16_round(float x);

/* Router projection: logits[t][e] = sum_c hidden[t][c] * router_w[e][c] (BF16 inputs, sums in
 * the accumulation type, ascending c).  hidden [T, d], router_w [E, d], logits [T, E].
 * Returns 0, or -1 on invalid sizes. */
int oracle_router_logits_f32(int T, int d, int E, const uint16_t* hidden_bf16, const uint16_t* router_w_bf16,
                             float* logits);
int oracle_router_logits_f64(int T, int d, int E, const uint16_t* hidden_bf16, const uint16_t* router_w_bf16,
                             double* logits);

/* Gated residual update and normalisation for G residual branches:
 *   R'[g][t] = BF16(R[g][t] + 2 sigmoid(a[t][g]) O[t]),
 *   N[g][t]  = R'[g][t] / sqrt(mean(R'[g][t]^2) + eps) * (1 + w[g])
 * moe_out O [T, d] (the sublayer output), residual R [G, T, d] BF16, inject_logits a [T, G],
 * norm_w w [G, d] BF16; residual_out R' [G, T, d] BF16, normed N [G, T, d].  Returns 0 or -1. */
int oracle_gated_residual_norm_f32(int T, int d, int G, const float* moe_out, const uint16_t* residual_bf16,
                                   const float* inject_logits, const uint16_t* norm_w_bf16, float eps,
                                   uint16_t* residual_out_bf16, float* normed);
int oracle_gated_residual_norm_f64(int T, int d, int G, const double* moe_out, const uint16_t* residual_bf16,
                                   const float* inject_logits, const uint16_t* norm_w_bf16, float eps,
                                   uint16_t* residual_out_bf16, double* normed);

/* oracle_moe_experts_f32 with one FP32 tensor scale per expert and weight tensor:
 * w13_ts_e [E] and w2_ts_e [E] (entry e scales expert e's W13 / W2). */
int oracle_moe_experts_ts_f32(int T, int d, int F, int E, int k, const uint16_t* hidden_bf16, const int32_t* ids,
                              const float* weights, const uint8_t* w13_codes, const uint8_t* w13_scales,
                              const float* w13_ts_e, const uint8_t* w2_codes, const uint8_t* w2_scales,
                              const float* w2_ts_e, const uint16_t* residual_bf16, const uint8_t* token_mask,
                              float* out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
