// Router (softmax + top-k + renormalisation) and bucketing (plan) kernels.
//
// Router: one warp per token ("Fused MoE routing" in "How I forked vLLM and made
// Qwen3.8-Flash-Next decode 1.6x faster on one GPU", section 5; "Router: selection and
// expert-task production" in "Persistent execution for Flash-Next GGUF on SM70").  Lane
// l holds logits l + 32 i.  The softmax denominator is a warp reduction; selection is k
// rounds of a warp arg-max on order-preserving float keys with the lowest expert id
// winning ties (redux.sync max of the key, then redux.sync min of the candidate ids).
// Selection compares the logits; softmax is monotone, so this is the same selection as
// on probabilities and keeps the ids independent of the exponential's rounding.
//
// Plan: one CTA.  Per-expert counts (shared-memory atomics), exclusive scan, the
// ascending touched-expert list, each route's position in expert-major order, and the
// expert kernel's task table (all gate/up tasks, then all down tasks) ("First
// implementation boundary", step 1: compact expert-presence list plus the original
// route positions; no gather of token features).
#include <cfloat>

#include "moe_common.cuh"
#include "moe_kernels.cuh"

namespace moe {

constexpr uint32_t kFull = 0xffffffffu;

// Route token t (one warp): softmax over the E logits, k rounds of arg-max selection,
// renormalised weights.  Writes ids[t, :k] and weights[t, :k].
template <int NPL>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ weights,
                                            int* s_ids = nullptr, float* s_w = nullptr, int s_row = 0) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[NPL];
  uint32_t key[NPL];
  float mx = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    const bool ok = e < E;
    v[i] = ok ? __ldg(row + e) : -FLT_MAX;
    key[i] = ok ? float_key(v[i]) : 0u;  // 0 is below every real key: never selected
    mx = fmaxf(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    if (lane + 32 * i < E) s += expf(v[i] - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  const float z = s;

  uint32_t used = 0;
  int my_id = 0;
  float my_p = 0.f;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (!((used >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t kmax = __reduce_max_sync(kFull, bk);
    const uint32_t cand = (bi >= 0 && bk == kmax) ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
    const uint32_t idx = __reduce_min_sync(kFull, cand);
    const int owner = static_cast<int>(idx & 31u);
    const int slot = static_cast<int>(idx >> 5);
    if (lane == owner) used |= 1u << slot;
    float lv = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) lv = (i == slot) ? v[i] : lv;
    lv = __shfl_sync(kFull, lv, owner);
    if (lane == j) {
      my_id = static_cast<int>(idx);
      my_p = expf(lv - mx) / z;
    }
  }
  // renormalise over the selection, summed in slot order
  float sel = 0.f;
  for (int j = 0; j < k; ++j) sel += __shfl_sync(kFull, my_p, j);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_id;
    weights[static_cast<size_t>(t) * k + lane] = my_p / sel;
    if (s_ids != nullptr) {
      s_ids[s_row * k + lane] = my_id;
      s_w[s_row * k + lane] = my_p / sel;
    }
  }
}

template <int NPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ weights) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<NPL>(logits, t, E, k, ids, weights);
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* weights,
                              cudaStream_t stream) {
  const int npl = (E + 31) / 32;
  const dim3 grid((T + 7) / 8), block(256);
  void (*kern)(const float*, int, int, int, int32_t*, float*) =
      npl <= 1 ? route_topk_kernel<1> : npl <= 2 ? route_topk_kernel<2> : npl <= 4 ? route_topk_kernel<4>
      : npl <= 8 ? route_topk_kernel<8> : npl <= 16 ? route_topk_kernel<16> : route_topk_kernel<32>;
  return launch_pdl(kern, grid, block, 0, stream, logits, T, E, k, ids, weights);
}

// Exclusive scan of one int per thread across a 1024-thread block; returns the total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int out = warp_sums[warp] + incl - v;
  total = warp_sums[32];
  __syncthreads();
  return out;
}

// The plan for all T * k routes, computed by one 1024-thread CTA.  ids/weights are read past
// L1: in the fused front they were written by other CTAs of the same launch.
__device__ __forceinline__ void plan_block(const PlanArgs& a) {
  __shared__ int s_counts[1024];
  __shared__ int s_cursor[1024];
  __shared__ int s_scan[33];
  const int tid = threadIdx.x;
  const int E = a.E, R = a.T * a.k;
  if (tid < E) s_counts[tid] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = __ldcg(a.ids + r);
    a.route_w[r] = __ldcg(a.weights + r);
    if (e < 0 || e >= E) {
      atomicOr(a.status, static_cast<int>(MOE_DEV_BAD_EXPERT_ID));
    } else {
      atomicAdd(&s_counts[e], 1);
    }
  }
  __syncthreads();
  const int cnt = tid < E ? s_counts[tid] : 0;
  int total = 0;
  const int off = block_exclusive_scan(cnt, s_scan, total);
  const int flag = cnt > 0 ? 1 : 0;
  int U = 0;
  const int rank = block_exclusive_scan(flag, s_scan, U);
  if (tid < E) {
    a.counts[tid] = cnt;
    a.offsets[tid] = off;
    s_cursor[tid] = off;
    if (flag) a.touched[rank] = tid;
  }
  if (tid == 0) a.offsets[E] = total;
  // per touched expert: passes of kRowsPerPass rows; gate/up and down task counts
  const int npass = flag ? (cnt + kRowsPerPass - 1) / kRowsPerPass : 0;
  const int ngu = npass * a.S_gu;
  const int ndn = npass * a.S_dn;
  __syncthreads();
  if (flag) s_counts[rank] = ngu;  // gather per-touched values at index `rank`
  __syncthreads();
  int gu_total = 0;
  const int gu_v = tid < U ? s_counts[tid] : 0;
  const int gu_start = block_exclusive_scan(gu_v, s_scan, gu_total);
  __syncthreads();
  if (flag) s_counts[rank] = ndn;
  __syncthreads();
  int dn_total = 0;
  const int dn_v = tid < U ? s_counts[tid] : 0;
  const int dn_start = block_exclusive_scan(dn_v, s_scan, dn_total);
  if (tid < U) {
    a.gu_start[tid] = gu_start;
    a.dn_start[tid] = dn_start;
  }
  if (tid == 0) {
    a.gu_start[U] = gu_total;
    a.dn_start[U] = dn_total;
  }
  // the task table: all gate/up tasks (touched order, pass, stripe), then all down tasks
  __syncthreads();
  if (flag) {
    s_counts[rank] = tid;  // expert of touched index `rank`
  }
  __syncthreads();
  if (tid < U) {
    const int e = s_counts[tid];
    const int m = a.counts[e];
    const int base = a.offsets[e];
    const int np = (m + kRowsPerPass - 1) / kRowsPerPass;
    int gi = gu_start;
    int di = gu_total + dn_start;
    for (int p = 0; p < np; ++p) {
      const int rows = min(kRowsPerPass, m - p * kRowsPerPass);
      const int row0 = base + p * kRowsPerPass;
      const int z = rows | (np > 1 ? 1 << 17 : 0);
      for (int s2 = 0; s2 < a.S_gu; ++s2) a.tasks[gi++] = TaskEntry{e | (tid << 16), row0, z, s2};
      for (int s2 = 0; s2 < a.S_dn; ++s2) a.tasks[di++] = TaskEntry{e | (tid << 16), row0, z | (1 << 16), s2};
    }
  }
  // largest row count over the experts
  int mx = cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(kFull, mx, o));
  if ((tid & 31) == 0) s_scan[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    int m = 0;
    for (int w = 0; w < 32; ++w) m = max(m, s_scan[w]);
    a.meta[META_U] = U;
    a.meta[META_NGU] = gu_total;
    a.meta[META_NDN] = dn_total;
    a.meta[META_MAXROWS] = m;
  }
  __syncthreads();
  // route positions in expert-major order
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = __ldcg(a.ids + r);
    if (e < 0 || e >= E) {
      a.route_pos[r] = -1;
      continue;
    }
    const int pos = atomicAdd(&s_cursor[e], 1);
    a.route_pos[r] = pos;
    a.pos_tok[pos] = r / a.k;
  }
}

// The plan for up to kPlanCached * 1024 routes in one 1024-thread CTA, with one pass over
// the routes (each thread keeps its routes' experts and in-bucket ranks in registers) and one
// block scan of (count, touched flag, passes) packed in 64 bits.  ids/weights come from
// shared memory (from_smem) or from global memory past L1 (written by other CTAs).  Route
// positions within a bucket follow shared-memory atomic order (outputs do not depend on it).
constexpr int kPlanCached = 16;

__device__ __forceinline__ long long block_exclusive_scan64(long long v, long long* warp_sums, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const long long w = warp_sums[lane];
    long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - w;
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  total = warp_sums[32];
  return warp_sums[warp] + incl - v;
}

__device__ __forceinline__ void plan_block_cached(const PlanArgs& a, const int* ids_src, const float* w_src,
                                                  bool from_smem) {
  __shared__ int s_off[1024];
  __shared__ int s_num[1024];
  __shared__ long long s_scan64[33];
  const int tid = threadIdx.x;
  const int E = a.E, R = a.T * a.k;
  if (tid < E) s_num[tid] = 0;
  __syncthreads();
  int ev[kPlanCached], rk[kPlanCached];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kPlanCached; ++j) {
    const int r = tid + j * 1024;
    ev[j] = -1;
    rk[j] = 0;
    if (r < R) {
      const int e = from_smem ? ids_src[r] : __ldcg(ids_src + r);
      a.route_w[r] = from_smem ? w_src[r] : __ldcg(w_src + r);
      if (e < 0 || e >= E) {
        bad = true;
        a.route_pos[r] = -1;
      } else {
        ev[j] = e;
        rk[j] = atomicAdd(&s_num[e], 1);
      }
    }
  }
  if (bad) atomicOr(a.status, static_cast<int>(MOE_DEV_BAD_EXPERT_ID));
  __syncthreads();
  // count (bits 0..21), touched flag (22..33), passes (34..63)
  const int cnt = tid < E ? s_num[tid] : 0;
  const int flag = cnt > 0 ? 1 : 0;
  const int np = (cnt + kRowsPerPass - 1) / kRowsPerPass;
  long long tot = 0;
  const long long pre = block_exclusive_scan64(
      static_cast<long long>(cnt) | (static_cast<long long>(flag) << 22) | (static_cast<long long>(np) << 34), s_scan64,
      tot);
  const int off = static_cast<int>(pre & 0x3fffff);
  const int rank = static_cast<int>((pre >> 22) & 0xfff);
  const int pass0 = static_cast<int>(pre >> 34);
  const int total = static_cast<int>(tot & 0x3fffff);
  const int U = static_cast<int>((tot >> 22) & 0xfff);
  const int passes = static_cast<int>(tot >> 34);
  if (tid < E) {
    a.counts[tid] = cnt;
    a.offsets[tid] = off;
    s_off[tid] = off;
    if (flag) {
      a.touched[rank] = tid;
      a.gu_start[rank] = pass0 * a.S_gu;
      a.dn_start[rank] = pass0 * a.S_dn;
    }
  }
  // largest row count over the experts
  int mx = cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(kFull, mx, o));
  if ((tid & 31) == 0) s_scan64[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    long long m = 0;
    for (int w = 0; w < 32; ++w) m = max(m, s_scan64[w]);
    a.offsets[E] = total;
    a.gu_start[U] = passes * a.S_gu;
    a.dn_start[U] = passes * a.S_dn;
    a.meta[META_U] = U;
    a.meta[META_NGU] = passes * a.S_gu;
    a.meta[META_NDN] = passes * a.S_dn;
    a.meta[META_MAXROWS] = static_cast<int>(m);
  }
  // route positions in expert-major order
#pragma unroll
  for (int j = 0; j < kPlanCached; ++j) {
    const int r = tid + j * 1024;
    if (ev[j] >= 0) {
      const int pos = s_off[ev[j]] + rk[j];
      a.route_pos[r] = pos;
      a.pos_tok[pos] = r / a.k;
    }
  }
  // the task table: all gate/up tasks (touched order, pass, stripe), then all down tasks;
  // each touched expert's thread writes its own entries
  if (tid < E && flag) {
    int gi = pass0 * a.S_gu, di = passes * a.S_gu + pass0 * a.S_dn;
    for (int p = 0; p < np; ++p) {
      const int rows = min(kRowsPerPass, cnt - p * kRowsPerPass);
      const int row0 = off + p * kRowsPerPass;
      const int z = rows | (np > 1 ? 1 << 17 : 0);
      for (int s2 = 0; s2 < a.S_gu; ++s2) a.tasks[gi++] = TaskEntry{tid | (rank << 16), row0, z, s2};
      for (int s2 = 0; s2 < a.S_dn; ++s2) a.tasks[di++] = TaskEntry{tid | (rank << 16), row0, z | (1 << 16), s2};
    }
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  if (a.T * a.k <= kPlanCached * 1024) plan_block_cached(a, a.ids, a.weights, false);
  else plan_block(a);
}

// ---------------------------------------------------------------------------------
// Fused front for moderate T * k: each 1024-thread CTA routes 32 tokens (one per warp) and
// converts their hidden rows to FP16; CTA 0 zeroes the expert kernel's counters.  With one
// CTA it builds the plan itself from its routes in shared memory; otherwise the last CTA to
// finish (arrival counter, reset by that CTA for the next call) builds it.
// ---------------------------------------------------------------------------------
// hidden rows [t0, t0 + nt) -> FP16 by threads `first` + i * `stride`, flagging values
// outside the FP16 range
__device__ __forceinline__ void convert_hidden(const FrontArgs& f, int t0, int nt, int first, int stride) {
  const size_t n8 = static_cast<size_t>(nt) * f.d / 8;
  const uint4* src = reinterpret_cast<const uint4*>(f.hidden + static_cast<size_t>(t0) * f.d);
  uint4* dst = reinterpret_cast<uint4*>(f.x16 + static_cast<size_t>(t0) * f.d);
  bool bad = false;
  for (size_t i = first; i < n8; i += stride) {
    const uint4 raw = src[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 v = __bfloat1622float2(b[q]);
      bad |= !(fabsf(v.x) <= 65504.f) || !(fabsf(v.y) <= 65504.f);
      h[q] = __floats2half2_rn(v.x, v.y);
    }
    dst[i] = o;
  }
  if (bad) atomicOr(f.plan.status, static_cast<int>(MOE_DEV_HIDDEN_RANGE));
}

template <int NPL>
__global__ void __launch_bounds__(1024) front_kernel(FrontArgs f) {
  __shared__ int s_last;
  __shared__ int s_ids[1024];  // one CTA: its routes, handed to the plan through shared memory
  __shared__ float s_w[1024];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const PlanArgs& a = f.plan;
  const int t0 = blockIdx.x * 32, nt = min(32, a.T - t0);
  const bool single = gridDim.x == 1;
  // warps 0..nt-1 route one token each; the other warps stage the hidden rows meanwhile
  if (warp < nt)
    route_token<NPL>(f.logits, t0 + warp, a.E, a.k, const_cast<int32_t*>(a.ids), const_cast<float*>(a.weights),
                     single ? s_ids : nullptr, s_w, warp);
  if (nt < 32) {
    if (warp >= nt) convert_hidden(f, t0, nt, threadIdx.x - nt * 32, (32 - nt) * 32);
  } else {
    convert_hidden(f, t0, nt, threadIdx.x, blockDim.x);
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) f.ready[i] = 0u;
    if (threadIdx.x == 0) *f.ticket = 0u;
  }
  if (single) {
    __syncthreads();
    plan_block_cached(a, s_ids, s_w, true);
    return;
  }
  // the last CTA to arrive sees every route
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(f.done, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (a.T * a.k <= kPlanCached * 1024) plan_block_cached(a, a.ids, a.weights, false);
  else plan_block(a);
  if (threadIdx.x == 0) *f.done = 0u;
}

cudaError_t launch_front(const FrontArgs& f, cudaStream_t stream) {
  const int npl = (f.plan.E + 31) / 32;
  const dim3 grid((f.plan.T + 31) / 32), block(1024);
  void (*kern)(FrontArgs) = npl <= 1 ? front_kernel<1> : npl <= 2 ? front_kernel<2> : npl <= 4 ? front_kernel<4>
                           : npl <= 8 ? front_kernel<8> : npl <= 16 ? front_kernel<16> : front_kernel<32>;
  return launch_pdl(kern, grid, block, 0, stream, f);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, a);
}

}  // namespace moe
