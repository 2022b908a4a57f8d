// CPU oracle for the routed MoE layer.  TEST INFRASTRUCTURE ONLY: see moe_oracle.h.
//
// Plain single-threaded C++17.  Every step follows the definition it cites, in the
// order the definition states it; no blocking, fusion or reordering.  Sums run in
// ascending index order in the accumulation type (float for the parity reference,
// double for the shadow that bounds the float version's rounding error).
#include "moe_oracle.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace {

// E2M1 (OCP MX v1.0 FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
// Exponent field 0 is subnormal: value = 2^(1-1) * (m / 2) = m / 2.
// Otherwise value = 2^(e-1) * (1 + m / 2).  No infinities or NaN.
double e2m1_exact(uint32_t nibble) {
  const uint32_t s = (nibble >> 3) & 1u;
  const uint32_t e = (nibble >> 1) & 3u;
  const uint32_t m = nibble & 1u;
  double mag;
  if (e == 0) {
    mag = 0.5 * static_cast<double>(m);
  } else {
    mag = std::ldexp(1.0 + 0.5 * static_cast<double>(m), static_cast<int>(e) - 1);
  }
  return s ? -mag : mag;
}

// E4M3 (OCP MX v1.0 FP8 "FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
// Exponent field 0 is subnormal: 2^(1-7) * (m / 8).  S.1111.111 is NaN; there are no
// infinities, so exponent field 15 with m < 7 is an ordinary normal number (max 448).
double e4m3_exact(uint32_t byte) {
  const uint32_t s = (byte >> 7) & 1u;
  const uint32_t e = (byte >> 3) & 15u;
  const uint32_t m = byte & 7u;
  if (e == 15u && m == 7u) return std::nan("");
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(m) / 8.0, -6);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, static_cast<int>(e) - 7);
  }
  return s ? -mag : mag;
}

// BF16 is the upper half of an IEEE binary32 pattern.
float bf16_to_float(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// The two decode functions tabulated once (16 and 256 entries): the tables hold exactly
// the values of e2m1_exact / e4m3_exact, so lookups change nothing but speed.
struct DecodeTables {
  double e2m1[16];
  double e4m3[256];
  DecodeTables() {
    for (uint32_t i = 0; i < 16; ++i) e2m1[i] = e2m1_exact(i);
    for (uint32_t i = 0; i < 256; ++i) e4m3[i] = e4m3_exact(i);
  }
};
const DecodeTables& tables() {
  static const DecodeTables t;
  return t;
}

// One NVFP4 weight: code nibble c of a row (element 2i in the low nibble of byte i),
// its block scale (one E4M3 per 16 consecutive elements) and the tensor scale.  The
// product of an E2M1 value, an E4M3 value and an FP32 scale is formed in Acc; for
// float it is exact whenever the tensor scale is a power of two (6 significant bits).
template <typename Acc>
Acc nvfp4_weight(const DecodeTables& tb, const uint8_t* codes, const uint8_t* scales, float tensor_scale, int c) {
  const uint32_t byte = codes[c >> 1];
  const uint32_t nib = (c & 1) ? (byte >> 4) : (byte & 15u);
  const Acc v = static_cast<Acc>(tb.e2m1[nib]);
  const Acc s = static_cast<Acc>(tb.e4m3[scales[c >> 4]]);
  return v * s * static_cast<Acc>(tensor_scale);
}

// Router for one token (routing paragraph of "Fused MoE routing"; selection paragraph
// of "Router: selection and expert-task production"):
//   1. softmax over the E logits: p_e = exp(l_e - max) / sum_e exp(l_e - max);
//   2. choose k experts by repeated maxima of the logits, larger first, ties to the
//      lower expert index (the strict '>' keeps the first, i.e. lowest, index; float
//      comparison treats -0 and +0 as equal);
//   3. renormalise: w_j = p_{s_j} / sum_{i<k} p_{s_i}.
// Selecting on the logits instead of the rounded probabilities gives the same order
// in exact arithmetic (softmax is strictly increasing) and keeps the ids independent
// of the exponential's rounding.
template <typename Acc>
void route_token(int E, int k, const float* l, int32_t* ids, Acc* w) {
  float mx = l[0];
  for (int e = 1; e < E; ++e) mx = (l[e] > mx) ? l[e] : mx;
  std::vector<Acc> ex(E);
  Acc z = 0;
  for (int e = 0; e < E; ++e) {
    ex[e] = std::exp(static_cast<Acc>(l[e]) - static_cast<Acc>(mx));
    z += ex[e];
  }
  std::vector<Acc> p(E);
  for (int e = 0; e < E; ++e) p[e] = ex[e] / z;

  std::vector<char> used(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (used[e]) continue;
      if (best < 0 || l[e] > l[best]) best = e;
    }
    used[best] = 1;
    ids[j] = best;
  }
  Acc sel = 0;
  for (int j = 0; j < k; ++j) sel += p[ids[j]];
  for (int j = 0; j < k; ++j) w[j] = p[ids[j]] / sel;
}

template <typename Acc>
int route_topk(int T, int E, int k, const float* logits, int32_t* ids, Acc* weights) {
  if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
  for (int t = 0; t < T; ++t) {
    route_token<Acc>(E, k, logits + static_cast<size_t>(t) * E, ids + static_cast<size_t>(t) * k,
                     weights + static_cast<size_t>(t) * k);
  }
  return 0;
}

// Expert FFN plus weighted un-route for every selected token ("First implementation
// boundary", steps 2-4: gate/up with SiLU*multiply, down projection, routes summed in
// a fixed order).  For token t and slot j with expert e:
//   g_n = sum_c x_c Wg[e][n][c],  u_n = sum_c x_c Wu[e][n][c]           (n < F)
//   h_n = silu(g_n) * u_n,        silu(z) = z / (1 + exp(-z))
//   y_r = sum_n h_n W2[e][r][n]                                         (r < d)
//   out[t][r] = residual[t][r] + sum_{j=0..k-1} w_{t,j} y_{t,j,r}
// The FP32 tensor scale of each weight tensor is either one value for all experts or, when
// the per-expert array is given, entry e for expert e (one scale per expert's W13 and W2).
template <typename Acc>
int moe_experts(int T, int d, int F, int E, int k, const uint16_t* hidden, const int32_t* ids,
                const Acc* weights, const uint8_t* w13c, const uint8_t* w13s, float w13_ts,
                const uint8_t* w2c, const uint8_t* w2s, float w2_ts, const uint16_t* residual,
                const uint8_t* mask, Acc* out, const float* w13_ts_e = nullptr, const float* w2_ts_e = nullptr) {
  if (T < 0 || d <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E || d % 16 || F % 16) return -1;
  const DecodeTables& tb = tables();
  const size_t d2 = static_cast<size_t>(d) / 2, d16 = static_cast<size_t>(d) / 16;
  const size_t f2 = static_cast<size_t>(F) / 2, f16 = static_cast<size_t>(F) / 16;
  std::vector<Acc> x(d), g(F), u(F), h(F), y(d), acc(d);
  for (int t = 0; t < T; ++t) {
    if (mask && !mask[t]) continue;
    for (int c = 0; c < d; ++c) x[c] = static_cast<Acc>(bf16_to_float(hidden[static_cast<size_t>(t) * d + c]));
    for (int r = 0; r < d; ++r) acc[r] = 0;
    for (int j = 0; j < k; ++j) {
      const int e = ids[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) return -1;
      const float ts13 = w13_ts_e ? w13_ts_e[e] : w13_ts;
      const float ts2 = w2_ts_e ? w2_ts_e[e] : w2_ts;
      for (int n = 0; n < F; ++n) {
        const size_t rg = static_cast<size_t>(e) * 2 * F + n;      // gate row
        const size_t ru = static_cast<size_t>(e) * 2 * F + F + n;  // up row
        Acc sg = 0, su = 0;
        for (int c = 0; c < d; ++c) sg += x[c] * nvfp4_weight<Acc>(tb, w13c + rg * d2, w13s + rg * d16, ts13, c);
        for (int c = 0; c < d; ++c) su += x[c] * nvfp4_weight<Acc>(tb, w13c + ru * d2, w13s + ru * d16, ts13, c);
        g[n] = sg;
        u[n] = su;
      }
      for (int n = 0; n < F; ++n) h[n] = g[n] / (static_cast<Acc>(1) + std::exp(-g[n])) * u[n];
      for (int r = 0; r < d; ++r) {
        const size_t rr = static_cast<size_t>(e) * d + r;
        Acc s = 0;
        for (int n = 0; n < F; ++n) s += h[n] * nvfp4_weight<Acc>(tb, w2c + rr * f2, w2s + rr * f16, ts2, n);
        y[r] = s;
      }
      const Acc wj = weights[static_cast<size_t>(t) * k + j];
      for (int r = 0; r < d; ++r) acc[r] += wj * y[r];
    }
    for (int r = 0; r < d; ++r) {
      const Acc res = residual ? static_cast<Acc>(bf16_to_float(residual[static_cast<size_t>(t) * d + r])) : 0;
      out[static_cast<size_t>(t) * d + r] = res + acc[r];
    }
  }
  return 0;
}

// BF16 of a binary32 value, round to nearest, ties to even (the rounding a BF16 store of a
// float performs); NaN stays NaN (quiet), infinities and zeros keep their sign.
uint16_t bf16_round(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// Router projection ("Router: selection and expert-task production": the projection whose
// results feed selection): logits[t][e] = sum_c x[t][c] * Wr[e][c] with the BF16 hidden row
// and the BF16 router weight row, in the accumulation type, ascending c.
template <typename Acc>
int router_logits(int T, int d, int E, const uint16_t* hidden, const uint16_t* wr, Acc* logits) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      Acc s = 0;
      for (int c = 0; c < d; ++c)
        s += static_cast<Acc>(bf16_to_float(hidden[static_cast<size_t>(t) * d + c])) *
             static_cast<Acc>(bf16_to_float(wr[static_cast<size_t>(e) * d + c]));
      logits[static_cast<size_t>(t) * E + e] = s;
    }
  }
  return 0;
}

// Gated residual update and the next normalisation (TokenSpeed, "Residual update and
// normalization fusion"), per token t and residual branch g < G:
//   R'[g][t] = R[g][t] + 2 sigmoid(a[t][g]) O[t]          stored (and kept) as BF16
//   N[g][t]  = GemmaRMSNorm(R'[g][t], w[g])
//   GemmaRMSNorm(x, w)_c = x_c / sqrt(mean_c(x_c^2) + eps) * (1 + w_c)
// O is the sublayer's output (here the routed-MoE sum over the token's routes, without a
// residual); the normalisation reads the residual after its rounding to the storage type.
// sigmoid(z) = 1 / (1 + exp(-z)).  Sums ascend in c.
template <typename Acc>
int gated_residual_norm(int T, int d, int G, const Acc* O, const uint16_t* R, const float* a, const uint16_t* w,
                        float eps, uint16_t* r_out, Acc* n_out) {
  if (T < 0 || d <= 0 || G <= 0) return -1;
  std::vector<Acc> rr(d);
  for (int t = 0; t < T; ++t) {
    for (int g = 0; g < G; ++g) {
      const Acc z = static_cast<Acc>(a[static_cast<size_t>(t) * G + g]);
      const Acc gate = static_cast<Acc>(2) * (static_cast<Acc>(1) / (static_cast<Acc>(1) + std::exp(-z)));
      const size_t row = (static_cast<size_t>(g) * T + t) * d;
      Acc ss = 0;
      for (int c = 0; c < d; ++c) {
        const Acc v = static_cast<Acc>(bf16_to_float(R[row + c])) + gate * O[static_cast<size_t>(t) * d + c];
        const uint16_t b = bf16_round(static_cast<float>(v));
        r_out[row + c] = b;
        rr[c] = static_cast<Acc>(bf16_to_float(b));
        ss += rr[c] * rr[c];
      }
      const Acc inv = static_cast<Acc>(1) / std::sqrt(ss / static_cast<Acc>(d) + static_cast<Acc>(eps));
      for (int c = 0; c < d; ++c) {
        const Acc wc = static_cast<Acc>(bf16_to_float(w[static_cast<size_t>(g) * d + c]));
        n_out[row + c] = rr[c] * inv * (static_cast<Acc>(1) + wc);
      }
    }
  }
  return 0;
}

}  // namespace

extern "C" {

uint16_t oracle_bf16_round(float x) { return bf16_round(x); }

int oracle_router_logits_f32(int T, int d, int E, const uint16_t* hidden_bf16, const uint16_t* router_w_bf16,
                             float* logits) {
  return router_logits<float>(T, d, E, hidden_bf16, router_w_bf16, logits);
}

int oracle_router_logits_f64(int T, int d, int E, const uint16_t* hidden_bf16, const uint16_t* router_w_bf16,
                             double* logits) {
  return router_logits<double>(T, d, E, hidden_bf16, router_w_bf16, logits);
}

int oracle_gated_residual_norm_f32(int T, int d, int G, const float* moe_out, const uint16_t* residual_bf16,
                                   const float* inject_logits, const uint16_t* norm_w_bf16, float eps,
                                   uint16_t* residual_out_bf16, float* normed) {
  return gated_residual_norm<float>(T, d, G, moe_out, residual_bf16, inject_logits, norm_w_bf16, eps,
                                    residual_out_bf16, normed);
}

int oracle_gated_residual_norm_f64(int T, int d, int G, const double* moe_out, const uint16_t* residual_bf16,
                                   const float* inject_logits, const uint16_t* norm_w_bf16, float eps,
                                   uint16_t* residual_out_bf16, double* normed) {
  return gated_residual_norm<double>(T, d, G, moe_out, residual_bf16, inject_logits, norm_w_bf16, eps,
                                     residual_out_bf16, normed);
}

int oracle_moe_experts_ts_f32(int T, int d, int F, int E, int k, const uint16_t* hidden_bf16, const int32_t* ids,
                              const float* weights, const uint8_t* w13_codes, const uint8_t* w13_scales,
                              const float* w13_ts_e, const uint8_t* w2_codes, const uint8_t* w2_scales,
                              const float* w2_ts_e, const uint16_t* residual_bf16, const uint8_t* token_mask,
                              float* out) {
  if (!w13_ts_e || !w2_ts_e) return -1;
  return moe_experts<float>(T, d, F, E, k, hidden_bf16, ids, weights, w13_codes, w13_scales, 1.0f, w2_codes,
                            w2_scales, 1.0f, residual_bf16, token_mask, out, w13_ts_e, w2_ts_e);
}

float oracle_e2m1_value(uint32_t nibble) { return static_cast<float>(e2m1_exact(nibble & 15u)); }

float oracle_e4m3_value(uint32_t byte) { return static_cast<float>(e4m3_exact(byte & 255u)); }

int oracle_dequant_row(const uint8_t* codes, const uint8_t* scales, float tensor_scale, int K,
                       float* out) {
  if (K <= 0 || K % 16) return -1;
  for (int c = 0; c < K; ++c) out[c] = nvfp4_weight<float>(tables(), codes, scales, tensor_scale, c);
  return 0;
}

int oracle_route_topk_f32(int T, int E, int k, const float* logits, int32_t* ids, float* weights) {
  return route_topk<float>(T, E, k, logits, ids, weights);
}

int oracle_route_topk_f64(int T, int E, int k, const float* logits, int32_t* ids, double* weights) {
  return route_topk<double>(T, E, k, logits, ids, weights);
}

// Bucketing of routes by expert (the compact expert-presence list of "First
// implementation boundary", step 1): per-expert counts, their exclusive prefix sum,
// and the touched experts in ascending order.
int oracle_plan(int T, int E, int k, const int32_t* ids, int32_t* counts, int32_t* offsets,
                int32_t* touched) {
  if (T < 0 || E <= 0 || k <= 0) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (size_t r = 0; r < static_cast<size_t>(T) * k; ++r) {
    const int e = ids[r];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int U = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] > 0) touched[U++] = e;
  }
  return U;
}

int oracle_moe_experts_f32(int T, int d, int F, int E, int k, const uint16_t* hidden_bf16,
                           const int32_t* ids, const float* weights, const uint8_t* w13_codes,
                           const uint8_t* w13_scales, float w13_ts, const uint8_t* w2_codes,
                           const uint8_t* w2_scales, float w2_ts, const uint16_t* residual_bf16,
                           const uint8_t* token_mask, float* out) {
  return moe_experts<float>(T, d, F, E, k, hidden_bf16, ids, weights, w13_codes, w13_scales, w13_ts,
                            w2_codes, w2_scales, w2_ts, residual_bf16, token_mask, out);
}

int oracle_moe_experts_f64(int T, int d, int F, int E, int k, const uint16_t* hidden_bf16,
                           const int32_t* ids, const double* weights, const uint8_t* w13_codes,
                           const uint8_t* w13_scales, float w13_ts, const uint8_t* w2_codes,
                           const uint8_t* w2_scales, float w2_ts, const uint16_t* residual_bf16,
                           const uint8_t* token_mask, double* out) {
  return moe_experts<double>(T, d, F, E, k, hidden_bf16, ids, weights, w13_codes, w13_scales, w13_ts,
                             w2_codes, w2_scales, w2_ts, residual_bf16, token_mask, out);
}

}  // extern "C"
