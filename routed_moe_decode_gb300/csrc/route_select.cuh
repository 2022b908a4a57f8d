// Router selection of one token by one warp: softmax over the E logits, top-k by arg-max
// rounds on order-preserving float keys (lowest expert id wins ties), renormalised weights
// ("Fused MoE routing" in "How I forked vLLM and made Qwen3.8-Flash-Next decode 1.6x faster
// on one GPU", section 5; "Router: selection and expert-task production" in "Persistent
// execution for Flash-Next GGUF on SM70").  Used by the router kernels and by the decode
// kernel that routes its own tokens.
#pragma once

#include <cfloat>

#include "moe_common.cuh"

namespace moe {

constexpr uint32_t kFull = 0xffffffffu;

// Inverse of float_key: the float whose key is `k` (+0 for the shared key of +-0).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Insert key `x` of slot `i` into the descending list c[0..C) (slots in s[]); slots arrive in
// ascending order and only a strictly larger key moves ahead, so equal keys keep the lower
// slot (the lower expert id) first.
template <int C>
__device__ __forceinline__ void cache_insert(uint32_t (&c)[C], int (&s)[C], uint32_t x, int i) {
#pragma unroll
  for (int m = C - 1; m > 0; --m) {
    const bool above = x > c[m - 1], here = x > c[m];
    s[m] = above ? s[m - 1] : (here ? i : s[m]);
    c[m] = above ? c[m - 1] : (here ? x : c[m]);
  }
  s[0] = x > c[0] ? i : s[0];
  c[0] = x > c[0] ? x : c[0];
}

// Exact selection by k rounds over all of a lane's keys (no list): the fallback of
// route_token when a lane runs out of listed keys.  Same ordering and tie rule; lane l holds
// the ids [NPL l, NPL l + NPL).
template <int NPL>
__device__ __forceinline__ void select_scan(const uint32_t (&key)[NPL], int k, uint32_t& my_key, int& my_id) {
  const int lane = threadIdx.x & 31;
  uint32_t used = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (!((used >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t kmax = __reduce_max_sync(kFull, bk);
    const uint32_t cand = bk == kmax ? static_cast<uint32_t>(NPL * lane + bi) : 0xffffffffu;
    const uint32_t idx = __reduce_min_sync(kFull, cand);
    if (static_cast<int>(idx / NPL) == lane) used |= 1u << (idx % NPL);
    if (lane == j) {
      my_key = kmax;
      my_id = static_cast<int>(idx);
    }
  }
}

// Route token t (one warp): top-k by k rounds of arg-max selection, softmax weights
// renormalised over the selection.  Writes ids[t, :k] and weights[t, :k] (when ids is not
// null) and the shared-memory copies s_ids/s_w at row s_row (when s_ids is not null).
//
// Lane l holds the logits [NPL l, NPL l + NPL) (16-byte loads when E is a multiple of 4) and
// keeps its best min(NPL, 4) keys in a sorted register list; a round is one warp max over the
// lanes' heads, one warp min over the expert ids holding that key (the lowest id wins ties),
// and a shift of the winner's list.  If a lane gave away its whole list while holding further
// keys, the rounds may have missed one of those, and the selection is redone by full scans.
// The selected logit is recovered from its key (the key is a bijection of the float bits).
// Weights: w_j = exp(l_j - l_max) / sum over the selection of exp(l_i - l_max) -- the softmax
// probabilities renormalised over the selection, whose common denominator over all E experts
// cancels in the renormalisation, so it is not formed.
template <int NPL>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ weights,
                                            int* s_ids = nullptr, float* s_w = nullptr, int s_row = 0) {
  constexpr int C = NPL < 4 ? NPL : 4;
  const int lane = threadIdx.x & 31;
  const float* row = logits + static_cast<size_t>(t) * E;
  const int base = NPL * lane;
  const int nvalid = max(0, min(NPL, E - base));
  float v[NPL];
  uint32_t key[NPL];
  if (NPL % 4 == 0 && (E & 3) == 0 && nvalid == NPL) {
    const float4* r4 = reinterpret_cast<const float4*>(row + base);
#pragma unroll
    for (int j = 0; j < NPL / 4; ++j) {
      const float4 q = __ldg(r4 + j);
      v[4 * j] = q.x;
      v[4 * j + 1] = q.y;
      v[4 * j + 2] = q.z;
      v[4 * j + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NPL; ++i) v[i] = i < nvalid ? __ldg(row + base + i) : -FLT_MAX;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) key[i] = i < nvalid ? float_key(v[i]) : 0u;  // 0: below every real key
  uint32_t ck[C];
  int cs[C];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    ck[c] = 0u;
    cs[c] = 0;
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) cache_insert<C>(ck, cs, key[i], i);

  int nused = 0;
  uint32_t my_key = 0;
  int my_id = 0;
  uint32_t kmax0 = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t kmax = __reduce_max_sync(kFull, ck[0]);
    if (j == 0) kmax0 = kmax;
    const uint32_t cand = ck[0] == kmax ? static_cast<uint32_t>(base + cs[0]) : 0xffffffffu;
    const uint32_t idx = __reduce_min_sync(kFull, cand);
    if (lane == j) {
      my_key = kmax;
      my_id = static_cast<int>(idx);
    }
    const bool own = static_cast<int>(idx / NPL) == lane;
    nused += own ? 1 : 0;
#pragma unroll
    for (int c = 0; c + 1 < C; ++c) {
      ck[c] = own ? ck[c + 1] : ck[c];
      cs[c] = own ? cs[c + 1] : cs[c];
    }
    ck[C - 1] = own ? 0u : ck[C - 1];
  }
  if constexpr (NPL > C) {
    if (__any_sync(kFull, nused >= C && nvalid > C)) select_scan<NPL>(key, k, my_key, my_id);
  }
  // the largest logit is the first selected; renormalise over the selection
  const float mx = key_float(kmax0);
  const float p = lane < k ? expf(key_float(my_key) - mx) : 0.f;
  float sel = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sel += __shfl_xor_sync(kFull, sel, o);
  if (lane < k) {
    if (ids != nullptr) {
      ids[static_cast<size_t>(t) * k + lane] = my_id;
      weights[static_cast<size_t>(t) * k + lane] = p / sel;
    }
    if (s_ids != nullptr) {
      s_ids[s_row * k + lane] = my_id;
      s_w[s_row * k + lane] = p / sel;
    }
  }
}

}  // namespace moe
