// Router (softmax + top-k + renormalisation) and bucketing (plan) kernels.
//
// Router: one warp per token ("Fused MoE routing" in "How I forked vLLM and made
// Qwen3.8-Flash-Next decode 1.6x faster on one GPU", section 5; "Router: selection and
// expert-task production" in "Persistent execution for Flash-Next GGUF on SM70"), in
// route_select.cuh.  Lane l holds a contiguous block of E / 32 logits; selection is k rounds
// of a warp arg-max on order-preserving float keys with the lowest expert id winning ties
// (redux.sync max of the key, then redux.sync min of the candidate ids).  Selection compares
// the logits; softmax is monotone, so this is the same selection as on probabilities and
// keeps the ids independent of the exponential's rounding.
//
// Plan: one CTA.  Per-expert counts (shared-memory atomics), exclusive scan, the
// ascending touched-expert list, each route's position in expert-major order, and the
// expert kernel's task table (all gate/up tasks, then all down tasks) ("First
// implementation boundary", step 1: compact expert-presence list plus the original
// route positions; no gather of token features).
#include <cfloat>

#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "route_select.cuh"

namespace moe {

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

// Expert-parallel sharding: a call plans (and computes) only the routes of the experts in
// [e_lo, e_hi); the other routes get no bucket and route position -1, which the un-route
// skips, so the call's output is the partial sum over its experts.
__device__ __forceinline__ bool local_expert(const PlanArgs& a, int e) { return e >= a.e_lo && e < a.e_hi; }

// Everything of the plan that follows from the per-expert counts (thread e of a 1024-thread
// CTA holds count cnt of expert e): offsets, touched list, task-pass prefix sums, the task
// table and the meta words.  s_counts is scratch of 1024 ints.  Returns expert tid's offset.
// write_table: also write the task table from this block (one CTA writes a few hundred KB
// slowly; the multi-CTA plan leaves it to its scatter kernel, spread over all its CTAs).
__device__ __forceinline__ int plan_from_counts(const PlanArgs& a, int cnt, int* s_counts, int* s_scan,
                                                int* s_pass0, int* s_cnt, int* s_off, bool write_table) {
  const int tid = threadIdx.x;
  const int E = a.E;
  int total = 0;
  const int off = block_exclusive_scan(cnt, s_scan, total);
  const int flag = cnt > 0 ? 1 : 0;
  int U = 0;
  const int rank = block_exclusive_scan(flag, s_scan, U);
  if (tid < E) {
    a.counts[tid] = cnt;
    a.offsets[tid] = off;
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
  // the task table: all gate/up tasks (touched order, pass, stripe), then all down tasks; one
  // warp per pass (its touched expert found by binary search over the touched experts' first
  // passes) writes the pass's gate/up and down entries, one lane per stripe, so that each
  // store instruction covers consecutive entries
  __syncthreads();
  if (flag) {
    s_counts[rank] = tid;  // expert, row count and first position of touched index `rank`
    s_cnt[rank] = cnt;
    s_off[rank] = off;
  }
  if (tid < U) s_pass0[tid] = gu_start / a.S_gu;
  if (tid == 0) s_pass0[U] = gu_total / a.S_gu;
  __syncthreads();
  int4* tasks = reinterpret_cast<int4*>(a.tasks);
  const int passes = (U > 0 && write_table && !a.no_table) ? s_pass0[U] : 0;
  const int lane = tid & 31;
  for (int P = tid >> 5; P < passes; P += blockDim.x >> 5) {
    int lo = 0, hi = U - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pass0[mid] <= P) lo = mid;
      else hi = mid - 1;
    }
    const int e = s_counts[lo];
    const int p = P - s_pass0[lo];
    const int c = s_cnt[lo];
    const int rows = min(kRowsPerPass, c - p * kRowsPerPass);
    const int z = rows | (c > kRowsPerPass ? 1 << 17 : 0);
    const int x = e | (lo << 16), row0 = s_off[lo] + p * kRowsPerPass;
    for (int s2 = lane; s2 < a.S_gu; s2 += 32) tasks[P * a.S_gu + s2] = make_int4(x, row0, z, s2);
    for (int s2 = lane; s2 < a.S_dn; s2 += 32) tasks[gu_total + P * a.S_dn + s2] = make_int4(x, row0, z | (1 << 16), s2);
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
    // without a table the task counts read 0, so that an expert kernel that follows the table
    // finds no work rather than stale entries
    a.meta[META_NGU] = a.no_table ? 0 : gu_total;
    a.meta[META_NDN] = a.no_table ? 0 : dn_total;
    a.meta[META_MAXROWS] = m;
    a.meta[META_YFMT] = 0;
  }
  __syncthreads();
  return off;
}

// The plan for all T * k routes, computed by one 1024-thread CTA.  ids/weights are read past
// L1: in the fused front they were written by other CTAs of the same launch.
__device__ __forceinline__ void plan_block(const PlanArgs& a) {
  __shared__ int s_counts[1024];
  __shared__ int s_cursor[1025];
  __shared__ int s_cnt[1024];
  __shared__ int s_off[1024];
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
    } else if (local_expert(a, e)) {
      atomicAdd(&s_counts[e], 1);
    }
  }
  __syncthreads();
  const int cnt = tid < E ? s_counts[tid] : 0;
  const int off = plan_from_counts(a, cnt, s_counts, s_scan, s_cursor, s_cnt, s_off, true);
  if (tid < E) s_cursor[tid] = off;
  __syncthreads();
  // route positions in expert-major order
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = __ldcg(a.ids + r);
    if (e < 0 || e >= E || !local_expert(a, e)) {
      a.route_pos[r] = -1;
      continue;
    }
    const int pos = atomicAdd(&s_cursor[e], 1);
    a.route_pos[r] = pos;
    a.pos_tok[pos] = r / a.k;
  }
}

// The plan for up to kPlanCached * 1024 routes in one 1024-thread CTA, with one pass over
// the routes (each thread keeps NJ routes' experts and in-bucket ranks in registers) and one
// block scan of (count, touched flag, extra passes) packed in one word: 32 bits when every
// field fits (NJ = 1: at most 1024 routes), else 64 bits.  ids/weights come from shared
// memory (from_smem) or from global memory past L1 (written by other CTAs).  Route positions
// within a bucket follow shared-memory atomic order (outputs do not depend on it).
constexpr int kPlanCached = 16;
constexpr int kPlanMaxPasses = 1024 + kPlanCached * 1024 / kRowsPerPass;  // E + R / kRowsPerPass

struct PlanSmem {
  int off[1024];
  int num[1024];
  int expert[1024];  // touched index -> expert
  int pass0[1024];   // touched index -> its first pass
  int pass_rank[kPlanMaxPasses];  // pass -> touched index
  unsigned long long sum[33];
  int mx[33];
};

template <int NJ>
struct PlanPack;
template <>
struct PlanPack<1> {  // count <= 1024, touched <= 1024, extra passes <= 16
  using V = uint32_t;
  static constexpr int kF = 11, kX = 22;
};
template <>
struct PlanPack<4> {  // count <= 4096, touched <= 1024, extra passes <= 64
  using V = uint32_t;
  static constexpr int kF = 13, kX = 24;
};
template <>
struct PlanPack<kPlanCached> {
  using V = unsigned long long;
  static constexpr int kF = 22, kX = 34;
};

// Exclusive scan of one V per thread over a 1024-thread block, with the block total and the
// block maximum of `m` (warp reductions; two barriers).
template <typename V>
__device__ __forceinline__ V block_scan_max(V v, int m, PlanSmem& ps, V& total, int& mtotal) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  const int wm = __reduce_max_sync(kFull, m);
  if (lane == 31) ps.sum[warp] = incl;
  if (lane == 0) ps.mx[warp] = wm;
  __syncthreads();
  if (warp == 0) {
    const V w = static_cast<V>(ps.sum[lane]);
    V wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const V n = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += n;
    }
    ps.sum[lane] = wi - w;
    if (lane == 31) ps.sum[32] = wi;
    const int mm = __reduce_max_sync(kFull, ps.mx[lane]);
    if (lane == 0) ps.mx[32] = mm;
  }
  __syncthreads();
  total = static_cast<V>(ps.sum[32]);
  mtotal = ps.mx[32];
  return static_cast<V>(ps.sum[warp]) + incl - v;
}

template <int NJ>
__device__ __forceinline__ void plan_block_cached(const PlanArgs& a, const int* ids_src, const float* w_src,
                                                  bool from_smem, PlanSmem& ps) {
  using Pk = PlanPack<NJ>;
  using V = typename Pk::V;
  const int tid = threadIdx.x;
  const int E = a.E, R = a.T * a.k;
  if (tid < E) ps.num[tid] = 0;
  __syncthreads();
  int ev[NJ], rk[NJ];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int r = tid + j * 1024;
    ev[j] = -1;
    rk[j] = 0;
    if (r < R) {
      const int e = from_smem ? ids_src[r] : __ldcg(ids_src + r);
      a.route_w[r] = from_smem ? w_src[r] : __ldcg(w_src + r);
      if (e < 0 || e >= E) {
        bad = true;
        a.route_pos[r] = -1;
      } else if (!local_expert(a, e)) {
        a.route_pos[r] = -1;  // another shard's expert
      } else {
        ev[j] = e;
        rk[j] = atomicAdd(&ps.num[e], 1);
      }
    }
  }
  if (bad) atomicOr(a.status, static_cast<int>(MOE_DEV_BAD_EXPERT_ID));
  __syncthreads();
  const int cnt = tid < E ? ps.num[tid] : 0;
  const int flag = cnt > 0 ? 1 : 0;
  const int np = (cnt + kRowsPerPass - 1) / kRowsPerPass;
  V tot = 0;
  int mx = 0;
  const V pre = block_scan_max<V>(static_cast<V>(cnt) | (static_cast<V>(flag) << Pk::kF) |
                                      (static_cast<V>(np - flag) << Pk::kX),
                                  cnt, ps, tot, mx);
  constexpr V kMaskC = (V(1) << Pk::kF) - 1, kMaskF = (V(1) << (Pk::kX - Pk::kF)) - 1;
  const int off = static_cast<int>(pre & kMaskC);
  const int rank = static_cast<int>((pre >> Pk::kF) & kMaskF);
  const int pass0 = rank + static_cast<int>(pre >> Pk::kX);
  const int total = static_cast<int>(tot & kMaskC);
  const int U = static_cast<int>((tot >> Pk::kF) & kMaskF);
  const int passes = U + static_cast<int>(tot >> Pk::kX);
  if (tid < E) {
    a.counts[tid] = cnt;
    a.offsets[tid] = off;
    ps.off[tid] = off;
    if (flag) {
      ps.expert[rank] = tid;
      ps.pass0[rank] = pass0;
      for (int p = 0; p < np; ++p) ps.pass_rank[pass0 + p] = rank;
    }
  }
  if (tid == 0) {
    a.offsets[E] = total;
    a.gu_start[U] = passes * a.S_gu;
    a.dn_start[U] = passes * a.S_dn;
    a.meta[META_U] = U;
    a.meta[META_NGU] = a.no_table ? 0 : passes * a.S_gu;
    a.meta[META_NDN] = a.no_table ? 0 : passes * a.S_dn;
    a.meta[META_MAXROWS] = mx;
    a.meta[META_YFMT] = 0;
  }
  __syncthreads();
  // touched list in touched order (coalesced)
  for (int r = tid; r < U; r += blockDim.x) {
    a.touched[r] = ps.expert[r];
    a.gu_start[r] = ps.pass0[r] * a.S_gu;
    a.dn_start[r] = ps.pass0[r] * a.S_dn;
  }
  // route positions in expert-major order
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int r = tid + j * 1024;
    if (ev[j] >= 0) {
      const int pos = ps.off[ev[j]] + rk[j];
      a.route_pos[r] = pos;
      a.pos_tok[pos] = r / a.k;
    }
  }
  // the task table: all gate/up tasks (touched order, pass, stripe), then all down tasks;
  // consecutive threads write consecutive 16-byte entries
  const int ngu = passes * a.S_gu, ntask = a.no_table ? 0 : ngu + passes * a.S_dn;
  int4* tasks = reinterpret_cast<int4*>(a.tasks);
  for (int i = tid; i < ntask; i += blockDim.x) {
    const bool dn = i >= ngu;
    const int j = dn ? i - ngu : i;
    const int S = dn ? a.S_dn : a.S_gu;
    const int P = j / S, s2 = j - P * S;
    const int rk2 = ps.pass_rank[P];
    const int e = ps.expert[rk2];
    const int p = P - ps.pass0[rk2];
    const int c = ps.num[e];
    const int rows = min(kRowsPerPass, c - p * kRowsPerPass);
    const int z = rows | (dn ? 1 << 16 : 0) | (c > kRowsPerPass ? 1 << 17 : 0);
    tasks[i] = make_int4(e | (rk2 << 16), ps.off[e] + p * kRowsPerPass, z, s2);
  }
}

// plan of the routes in ids_src/w_src by the best-fitting variant (R <= kPlanCached * 1024)
__device__ __forceinline__ void plan_cached(const PlanArgs& a, const int* ids_src, const float* w_src,
                                            bool from_smem, PlanSmem& ps) {
  const int R = a.T * a.k;
  if (R <= 1024) plan_block_cached<1>(a, ids_src, w_src, from_smem, ps);
  else if (R <= 4096) plan_block_cached<4>(a, ids_src, w_src, from_smem, ps);
  else plan_block_cached<kPlanCached>(a, ids_src, w_src, from_smem, ps);
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanArgs a) {
  __shared__ PlanSmem ps;
  pdl_wait();
  pdl_launch_dependents();
  if (a.T * a.k <= kPlanCached * 1024) plan_cached(a, a.ids, a.weights, false, ps);
  else plan_block(a);
}

// ---------------------------------------------------------------------------------
// Fused front for moderate T * k: each 1024-thread CTA routes f.tpc tokens (one per warp;
// few per CTA, so that the latency-bound selection of different tokens runs on different
// SMs) and converts their hidden rows to FP16; CTA 0 zeroes the expert kernel's counters.  With one
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
  __shared__ PlanSmem ps;
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const PlanArgs& a = f.plan;
  const int t0 = blockIdx.x * f.tpc, nt = min(f.tpc, a.T - t0);
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
    for (int i = threadIdx.x; i < a.E + a.S_dn; i += blockDim.x) f.ready[i] = 0u;
    if (threadIdx.x == 0) *f.ticket = 0u;
  }
  if (single) {
    __syncthreads();
    plan_cached(a, s_ids, s_w, true, ps);
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
  if (a.T * a.k <= kPlanCached * 1024) plan_cached(a, a.ids, a.weights, false, ps);
  else plan_block(a);
  if (threadIdx.x == 0) *f.done = 0u;
}

cudaError_t launch_front(FrontArgs f, cudaStream_t stream) {
  const int npl = (f.plan.E + 31) / 32;
  // tokens per CTA: 4 while the CTAs fit the SMs in one wave, up to 32 beyond
  f.tpc = min(32, max(4, (f.plan.T + 147) / 148));
  const dim3 grid((f.plan.T + f.tpc - 1) / f.tpc), block(1024);
  void (*kern)(FrontArgs) = npl <= 1 ? front_kernel<1> : npl <= 2 ? front_kernel<2> : npl <= 4 ? front_kernel<4>
                           : npl <= 8 ? front_kernel<8> : npl <= 16 ? front_kernel<16> : front_kernel<32>;
  return launch_pdl(kern, grid, block, 0, stream, f);
}

// ---------------------------------------------------------------------------------
// The plan for many routes (prefill chunks) over several CTAs, in three launches:
//   1. per slice of kPlanSlice routes: route weights copied, expert histogram of the slice
//      (hist row = slice);
//   2. one CTA: per-expert counts summed over the slices, everything that follows from them
//      (plan_from_counts), and each slice's first position in every expert's bucket (written
//      over the histogram);
//   3. per slice: route positions from the slice's bucket bases (shared-memory cursors).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_hist_kernel(PlanArgs a, int* hist) {
  __shared__ int s_counts[1024];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, E = a.E, R = a.T * a.k;
  if (tid < E) s_counts[tid] = 0;
  __syncthreads();
  const int r1 = min(R, (blockIdx.x + 1) * kPlanSlice);
  for (int r = blockIdx.x * kPlanSlice + tid; r < r1; r += blockDim.x) {
    const int e = __ldcg(a.ids + r);
    a.route_w[r] = __ldcg(a.weights + r);
    if (e < 0 || e >= E) atomicOr(a.status, static_cast<int>(MOE_DEV_BAD_EXPERT_ID));
    else if (local_expert(a, e)) atomicAdd(&s_counts[e], 1);
  }
  __syncthreads();
  if (tid < E) hist[static_cast<size_t>(blockIdx.x) * E + tid] = s_counts[tid];
}

__global__ void __launch_bounds__(1024) plan_scan_kernel(PlanArgs a, int* hist, int slices) {
  __shared__ int s_counts[1024];
  __shared__ int s_scan[33];
  __shared__ int s_pass0[1025];
  __shared__ int s_cnt[1024];
  __shared__ int s_off[1024];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, E = a.E;
  // up to kScanCached slices: this expert's per-slice counts stay in registers between the
  // sum and the per-slice starts (independent loads instead of a dependent chain)
  constexpr int kScanCached = 32;
  int hv[kScanCached];
  int cnt = 0;
  if (slices <= kScanCached) {
#pragma unroll
    for (int g = 0; g < kScanCached; ++g) {
      hv[g] = (g < slices && tid < E) ? __ldcg(hist + static_cast<size_t>(g) * E + tid) : 0;
      cnt += hv[g];
    }
  } else if (tid < E) {
    for (int g = 0; g < slices; ++g) cnt += __ldcg(hist + static_cast<size_t>(g) * E + tid);
  }
  const int off = plan_from_counts(a, cnt, s_counts, s_scan, s_pass0, s_cnt, s_off, false);
  if (tid < E) {
    int run = off;
    if (slices <= kScanCached) {
#pragma unroll
      for (int g = 0; g < kScanCached; ++g) {
        if (g < slices) hist[static_cast<size_t>(g) * E + tid] = run;
        run += hv[g];
      }
    } else {
      for (int g = 0; g < slices; ++g) {
        int* h = hist + static_cast<size_t>(g) * E + tid;
        const int c = *h;
        *h = run;
        run += c;
      }
    }
  }
}

__global__ void __launch_bounds__(1024) plan_scatter_kernel(PlanArgs a, const int* hist) {
  __shared__ int s_cursor[1024];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, E = a.E, R = a.T * a.k;
  if (tid < E) s_cursor[tid] = __ldcg(hist + static_cast<size_t>(blockIdx.x) * E + tid);
  __syncthreads();
  const int r1 = min(R, (blockIdx.x + 1) * kPlanSlice);
  for (int r = blockIdx.x * kPlanSlice + tid; r < r1; r += blockDim.x) {
    const int e = __ldcg(a.ids + r);
    if (e < 0 || e >= E || !local_expert(a, e)) {
      a.route_pos[r] = -1;
      continue;
    }
    const int pos = atomicAdd(&s_cursor[e], 1);
    a.route_pos[r] = pos;
    a.pos_tok[pos] = r / a.k;
  }
  // the task table of plan_from_counts (written by plan_scan_kernel's arrays): warp w of CTA
  // b writes the passes of touched indices b * 32 + w, + 32 * gridDim.x, ..., one lane per
  // stripe, so that each store instruction covers consecutive entries
  const int lane = tid & 31;
  const int U = a.no_table ? 0 : __ldcg(a.meta + META_U), ngu = __ldcg(a.meta + META_NGU);
  int4* tasks = reinterpret_cast<int4*>(a.tasks);
  for (int u = blockIdx.x * 32 + (tid >> 5); u < U; u += 32 * gridDim.x) {
    const int e = __ldcg(a.touched + u);
    const int c = __ldcg(a.counts + e), base = __ldcg(a.offsets + e);
    const int P0 = __ldcg(a.gu_start + u) / a.S_gu;
    const int np = (c + kRowsPerPass - 1) / kRowsPerPass;
    for (int p = 0; p < np; ++p) {
      const int rows = min(kRowsPerPass, c - p * kRowsPerPass);
      const int z = rows | (c > kRowsPerPass ? 1 << 17 : 0);
      const int x = e | (u << 16), row0 = base + p * kRowsPerPass, P = P0 + p;
      for (int s2 = lane; s2 < a.S_gu; s2 += 32) tasks[P * a.S_gu + s2] = make_int4(x, row0, z, s2);
      for (int s2 = lane; s2 < a.S_dn; s2 += 32) tasks[ngu + P * a.S_dn + s2] = make_int4(x, row0, z | (1 << 16), s2);
    }
  }
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  const int R = a.T * a.k;
  if (R <= kPlanCached * 1024 || a.hist == nullptr) return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, a);
  const int slices = (R + kPlanSlice - 1) / kPlanSlice;
  cudaError_t e = launch_pdl(plan_hist_kernel, dim3(slices), dim3(1024), 0, stream, a, a.hist);
  if (e != cudaSuccess) return e;
  e = launch_pdl(plan_scan_kernel, dim3(1), dim3(1024), 0, stream, a, a.hist, slices);
  if (e != cudaSuccess) return e;
  return launch_pdl(plan_scatter_kernel, dim3(slices), dim3(1024), 0, stream, a, static_cast<const int*>(a.hist));
}

}  // namespace moe
