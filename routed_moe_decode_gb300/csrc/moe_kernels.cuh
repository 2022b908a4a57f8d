// Kernel argument blocks and host-side launchers of the routed-MoE CUDA path.
#pragma once

#include <cuda.h>

#include "moe_common.cuh"

namespace moe {

struct PlanArgs {
  int T, E, k, S_gu, S_dn;
  int e_lo, e_hi;  // experts this call plans: [e_lo, e_hi) (all: [0, E))
  const int32_t* ids;
  const float* weights;
  int* status;
  int* meta;
  int* counts;
  int* offsets;
  int* touched;
  int* gu_start;
  int* dn_start;
  int* route_pos;
  int* pos_tok;
  float* route_w;
  TaskEntry* tasks;
  int* hist;  // [ceil(T * k / kPlanSlice), E] scratch of the multi-CTA plan (many routes)
  // 1: leave the task table unwritten (a layer whose expert kernel derives its tasks itself)
  int no_table;
};

// The fused front (router + plan + FP16 hidden) for T * k up to kFrontMaxRoutes.
struct FrontArgs {
  PlanArgs plan;  // plan.ids / plan.weights receive the router's output
  int d;
  const float* logits;
  const __nv_bfloat16* hidden;
  __half* x16;
  uint32_t* ready;
  uint32_t* ticket;
  uint32_t* done;  // CTA arrival counter: zero between calls
  int tpc;         // tokens routed per CTA (one warp each), at most 32
};
constexpr int kFrontMaxRoutes = 16384;

struct PrepArgs {
  int T, d, E, S_dn;
  const __nv_bfloat16* hidden;
  __half* x16;
  uint32_t* ready;
  uint32_t* ticket;
  int* status;
};

// Everything the expert kernels read besides the two tensor maps.
struct ExpertArgs {
  int T, d, F, E, k, R, S_gu, S_dn, nck_gu, nck_dn;
  float w13_ts, w2_ts;
  // per-expert FP32 tensor scales (entry e - e_lo, like the weights), or null for the one
  // value above for every expert
  const float* w13_ts_e;
  const float* w2_ts_e;
  const uint8_t* w13_codes;
  const uint8_t* w13_scales;
  const uint8_t* w2_codes;
  const uint8_t* w2_scales;
  const int* meta;
  const int* counts;
  const int* offsets;
  const int* touched;
  const int* pos_tok;
  const int* route_pos;
  const float* route_w;
  const TaskEntry* tasks;
  const __half* x16;
  __half* hs16;
  float* y;
  uint32_t* ready;    // per touched expert: gate/up tasks published
  uint32_t* dn_done;  // per down stripe: down tasks published (ready + E)
  uint32_t* ticket;
  int* status;
  const __nv_bfloat16* residual;
  __nv_bfloat16* out;
  int e_lo;  // first expert of the weight tensors passed in (expert e's weights are entry e - e_lo)
  int ncb;  // un-route tasks appended to the task order (0: the un-route runs as its own kernel)
  int task_cap;  // entries the task table has room for
  // self test of the failure path: this down task (index among the down tasks of the
  // decode kernel's 8-row passes) waits for a readiness counter nothing publishes; -1: none
  int poison_dn;
  // every bounded wait of the expert kernels gives up after this many clock cycles
  // (kDefaultWaitLimit; the self tests shorten it to exercise the failure path)
  long long wait_limit;
  // optional timeline (diagnostics, off when null): per CTA kTraceRoles x kTracePerRole
  // uint64 events = event code << 56 | index << 40 | %globaltimer low 40 bits
  unsigned long long* trace;
};

// FP32 tensor scale of expert e's W13 / W2: the per-expert array when given, else the one
// value for every expert.
__device__ __forceinline__ float ts13_of(const ExpertArgs& a, int e) {
  return a.w13_ts_e ? __ldg(a.w13_ts_e + (e - a.e_lo)) : a.w13_ts;
}
__device__ __forceinline__ float ts2_of(const ExpertArgs& a, int e) {
  return a.w2_ts_e ? __ldg(a.w2_ts_e + (e - a.e_lo)) : a.w2_ts;
}

// Un-route of four consecutive columns [c, c + 4) of token t: out = residual + sum_j w_{t,j}
// y_{pos(t,j)}, FP32, slots in order, one BF16 rounding ("First implementation boundary",
// step 4: routes summed in a fixed order).  The loads of eight slots are in flight together.
// y is read past L1 (it may have been written by the calling kernel).  Shared by the un-route
// kernel and the expert kernel's fused un-route, so both give the same bits.
__device__ __forceinline__ void unroute4(const ExpertArgs& a, int t, int c) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int* rp = a.route_pos + static_cast<size_t>(t) * a.k;
  const float* rw = a.route_w + static_cast<size_t>(t) * a.k;
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    int pos[8];
    float w[8];
    float4 yv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      pos[jj] = j0 + jj < a.k ? __ldg(rp + j0 + jj) : -1;
      w[jj] = j0 + jj < a.k ? __ldg(rw + j0 + jj) : 0.f;
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      yv[jj] = pos[jj] >= 0 ? __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<size_t>(pos[jj]) * a.d + c))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (pos[jj] < 0) continue;
      acc.x += w[jj] * yv[jj].x;
      acc.y += w[jj] * yv[jj].y;
      acc.z += w[jj] * yv[jj].z;
      acc.w += w[jj] * yv[jj].w;
    }
  }
  const size_t o = static_cast<size_t>(t) * a.d + c;
  float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.residual) {
    const uint2 rb = *reinterpret_cast<const uint2*>(a.residual + o);
    const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.x));
    const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.y));
    res = make_float4(r0.x, r0.y, r1.x, r1.y);
  }
  __nv_bfloat162 o0 = __floats2bfloat162_rn(res.x + acc.x, res.y + acc.y);
  __nv_bfloat162 o1 = __floats2bfloat162_rn(res.z + acc.z, res.w + acc.w);
  uint2 ob;
  ob.x = *reinterpret_cast<uint32_t*>(&o0);
  ob.y = *reinterpret_cast<uint32_t*>(&o1);
  *reinterpret_cast<uint2*>(a.out + o) = ob;
}

// unroute4 for per-route outputs stored as FP16(y * 2^-4) (the wide kernel): the same slot
// order and FP32 accumulation, four slots' loads in flight at a time (at the prefill chunk
// the un-route kernel took 75 us so, against 95 us with eight and 124 us with two columns
// per thread).
__device__ __forceinline__ void unroute4_y16(const ExpertArgs& a, int t, int c) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int* rp = a.route_pos + static_cast<size_t>(t) * a.k;
  const float* rw = a.route_w + static_cast<size_t>(t) * a.k;
  const __half* y16 = reinterpret_cast<const __half*>(a.y);
  for (int j0 = 0; j0 < a.k; j0 += 4) {
    int pos[4];
    float w[4];
    uint2 yv[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      pos[jj] = j0 + jj < a.k ? __ldg(rp + j0 + jj) : -1;
      w[jj] = j0 + jj < a.k ? __ldg(rw + j0 + jj) * kYUnscale : 0.f;
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      yv[jj] = pos[jj] >= 0 ? __ldcg(reinterpret_cast<const uint2*>(y16 + static_cast<size_t>(pos[jj]) * a.d + c))
                            : make_uint2(0, 0);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (pos[jj] < 0) continue;
      const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&yv[jj].x));
      const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&yv[jj].y));
      acc.x += w[jj] * lo.x;
      acc.y += w[jj] * lo.y;
      acc.z += w[jj] * hi.x;
      acc.w += w[jj] * hi.y;
    }
  }
  const size_t o = static_cast<size_t>(t) * a.d + c;
  float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.residual) {
    const uint2 rb = *reinterpret_cast<const uint2*>(a.residual + o);
    const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.x));
    const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.y));
    res = make_float4(r0.x, r0.y, r1.x, r1.y);
  }
  __nv_bfloat162 o0 = __floats2bfloat162_rn(res.x + acc.x, res.y + acc.y);
  __nv_bfloat162 o1 = __floats2bfloat162_rn(res.z + acc.z, res.w + acc.w);
  uint2 ob;
  ob.x = *reinterpret_cast<uint32_t*>(&o0);
  ob.y = *reinterpret_cast<uint32_t*>(&o1);
  *reinterpret_cast<uint2*>(a.out + o) = ob;
}

// unroute4 in two halves for a caller that must wait for y: the slot positions and weights
// of the first 16 slots and the residual are loaded before the wait (they do not depend on
// y), the rest after it.  Same arithmetic in the same order as unroute4, so the same bits.
struct Unroute4Pre {
  int pos[16];
  float w[16];
  float4 res;
};

// kSmemPlan: the route positions and weights come from shared-memory arrays [T * k] (rp_all,
// rw_all: the decode kernel's own plan) instead of the workspace's.
template <bool kSmemPlan, typename V>
__device__ __forceinline__ V plan_load(const V* p) {
  if constexpr (kSmemPlan) return *p;
  else return __ldg(p);
}

template <bool kSmemPlan = false>
__device__ __forceinline__ void unroute4_pre(const ExpertArgs& a, int t, int c, Unroute4Pre& u,
                                             const int* rp_all = nullptr, const float* rw_all = nullptr) {
  const int* rp = (kSmemPlan ? rp_all : a.route_pos) + static_cast<size_t>(t) * a.k;
  const float* rw = (kSmemPlan ? rw_all : a.route_w) + static_cast<size_t>(t) * a.k;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    u.pos[j] = j < a.k ? plan_load<kSmemPlan>(rp + j) : -1;
    u.w[j] = j < a.k ? plan_load<kSmemPlan>(rw + j) : 0.f;
  }
  u.res = make_float4(0.f, 0.f, 0.f, 0.f);
  if (a.residual) {
    const uint2 rb = *reinterpret_cast<const uint2*>(a.residual + static_cast<size_t>(t) * a.d + c);
    const float2 r0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.x));
    const float2 r1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.y));
    u.res = make_float4(r0.x, r0.y, r1.x, r1.y);
  }
}

template <bool kSmemPlan = false>
__device__ __forceinline__ void unroute4_post(const ExpertArgs& a, int t, int c, const Unroute4Pre& u,
                                              const int* rp_all = nullptr, const float* rw_all = nullptr) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int* rp = (kSmemPlan ? rp_all : a.route_pos) + static_cast<size_t>(t) * a.k;
  const float* rw = (kSmemPlan ? rw_all : a.route_w) + static_cast<size_t>(t) * a.k;
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    int pos[8];
    float w[8];
    float4 yv[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (j0 == 0) {
        pos[jj] = u.pos[jj];
        w[jj] = u.w[jj];
      } else if (j0 == 8) {
        pos[jj] = u.pos[8 + jj];
        w[jj] = u.w[8 + jj];
      } else {
        pos[jj] = j0 + jj < a.k ? plan_load<kSmemPlan>(rp + j0 + jj) : -1;
        w[jj] = j0 + jj < a.k ? plan_load<kSmemPlan>(rw + j0 + jj) : 0.f;
      }
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      yv[jj] = pos[jj] >= 0 ? __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<size_t>(pos[jj]) * a.d + c))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (pos[jj] < 0) continue;
      acc.x += w[jj] * yv[jj].x;
      acc.y += w[jj] * yv[jj].y;
      acc.z += w[jj] * yv[jj].z;
      acc.w += w[jj] * yv[jj].w;
    }
  }
  __nv_bfloat162 o0 = __floats2bfloat162_rn(u.res.x + acc.x, u.res.y + acc.y);
  __nv_bfloat162 o1 = __floats2bfloat162_rn(u.res.z + acc.z, u.res.w + acc.w);
  uint2 ob;
  ob.x = *reinterpret_cast<uint32_t*>(&o0);
  ob.y = *reinterpret_cast<uint32_t*>(&o1);
  *reinterpret_cast<uint2*>(a.out + static_cast<size_t>(t) * a.d + c) = ob;
}

constexpr int kTraceRoles = 8;
constexpr int kTracePerRole = 1024;

// Launch `kernel` as a programmatic dependent of the preceding work in `stream` (it may
// begin while its predecessor finishes; the kernels order themselves with pdl_wait).
// Every kernel of the library asks for the largest shared-memory carveout, so that an SM
// need not be reconfigured between the small front kernels and the expert kernels (which
// use ~200 KB): a reconfiguration waits for the SM to drain and defeats the early start.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaError_t ce = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* weights,
                              cudaStream_t stream);
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
cudaError_t launch_front(FrontArgs f, cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream);
cudaError_t launch_expert_tc(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                             int num_sms, cudaStream_t stream);
cudaError_t launch_expert_mma(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_s13, const CUtensorMap& tm_s2, int num_sms,
                              cudaStream_t stream);
cudaError_t launch_expert_simt(const ExpertArgs& a, cudaStream_t stream);
// The many-rows kernel: its task table (passes of kWideRows rows) is built from the plan's
// per-expert arrays by launch_wide_plan, then launch_expert_wide runs with a.tasks = that table.
cudaError_t launch_wide_plan(const ExpertArgs& a, TaskEntry* tasks_w, cudaStream_t stream);
// launch_wide_gather writes the FP16 hidden rows in route order (xs[pos] = x16[pos_tok[pos]])
// for the wide kernel's gate/up passes.  The wide kernel reads those rows [R, d] and the FP16 h
// rows [R, ffn] through tensor maps of 64-element (128-byte) wide boxes with the 128-byte
// swizzle, entry j of each array with boxes of 64 (j + 1) rows.
struct WideActMaps {
  CUtensorMap xs[3];
  CUtensorMap h[3];
};
cudaError_t launch_wide_gather(const ExpertArgs& a, __half* xs, int num_sms, cudaStream_t stream);
cudaError_t launch_expert_wide(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                               const WideActMaps& am, int num_sms, cudaStream_t stream);
int encode_f16_rows_map(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);
size_t expert_wide_smem_bytes();
cudaError_t launch_combine(const ExpertArgs& a, cudaStream_t stream);
size_t expert_tc_smem_bytes();
size_t expert_mma_smem_bytes();
// The decode kernel for at most eight tokens (expert_dec.cu): hidden rows resident in shared
// memory, h rows copied once per down task; same task table, counters and outputs as
// launch_expert_mma, which it replaces where expert_dec_supports holds.
cudaError_t launch_expert_dec(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_s13, const CUtensorMap& tm_s2, int num_sms,
                              cudaStream_t stream);
bool expert_dec_supports(int T, int d, int F);
size_t expert_dec_smem_bytes(int T, int d, int F);

// The decode kernel with its own front, for a whole layer of at most eight tokens: every CTA
// routes the T tokens (one warp each, the router of route_select.cuh), converts their hidden
// rows to FP16 straight into shared memory and builds the plan there (the same buckets,
// touched list and task order as the plan kernel, route positions in route order within a
// bucket), so the weight stream starts without a separate front launch.  The CTAs also write
// the routing (ids, weights), the plan and the FP16 hidden rows into the workspace, split
// between them, for later calls that reuse them.  Its counters alternate between two zeroed
// sets: the set in use is read at start (after the wait on the preceding kernel), CTA 0
// zeroes the other one, and the last CTA to finish flips the parity.
struct DecFront {
  const float* logits;          // [T, E]
  const __nv_bfloat16* hidden;  // [T, d]
  int32_t* ids;                 // [T, k] out
  float* weights;               // [T, k] out
  int* meta;
  int* counts;
  int* offsets;
  int* touched;
  int* gu_start;
  int* dn_start;
  int* route_pos;
  int* pos_tok;
  float* route_w;
  TaskEntry* tasks;
  __half* x16;
  uint32_t* sets;    // 2 x kDecSetWords
  uint32_t* parity;  // set of the next launch
  uint32_t* done;    // CTA arrivals of the current launch
};
bool expert_dec_front_supports(int T, int d, int F, int E, int k);
cudaError_t launch_expert_dec_front(const ExpertArgs& a, const DecFront& f, const CUtensorMap& tm_w13,
                                    const CUtensorMap& tm_w2, const CUtensorMap& tm_s13, const CUtensorMap& tm_s2,
                                    int num_sms, cudaStream_t stream);
// true when the decode kernel gathers each task's hidden rows (T > 8): its tasks are then
// 8-row passes, which every CTA derives from the plan's per-expert arrays
bool expert_dec_gathers(int T);
// un-route tasks the decode kernel appends when it runs the un-route itself (one per down
// stripe; T <= 8), or 0
int expert_dec_unroute_tasks(int T, int d, int F);
// number of un-route tasks the decode kernel appends when it runs the un-route itself
int expert_mma_unroute_tasks(int T, int S_dn);
int encode_codes_map(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes);
// Tensor map of a [rows, row_bytes] uint8 matrix (row_bytes a multiple of 16) loaded in
// unswizzled boxes of 16 bytes x box_rows rows.
int encode_scales_map(CUtensorMap* tm, const void* base, uint32_t row_bytes, uint64_t rows, uint32_t box_rows);
// Shapes the decode (warp-MMA) kernel handles: d and ffn powers of two from 256 to 2048.
bool expert_mma_supports(int d, int F);
// Router projection logits = hidden x Wr^T (BF16 in, FP32 out) with the weight tile copied
// before the wait for the preceding kernel (router_norm.cu); E a multiple of 16, d of 64.
bool router_gemv_supports(int T, int d, int E);
size_t router_smem_bytes(int d);
cudaError_t launch_router_gemv(const __nv_bfloat16* hidden, const __nv_bfloat16* wr, float* logits, int T, int d,
                               int E, cudaStream_t stream);
// Gated un-route: R'[g] = BF16(R[g] + 2 sigmoid(a[g]) O), N[g] = GemmaRMSNorm(R'[g], w[g]) for
// G residual branches, O the token's weighted routes (router_norm.cu); d <= 4096, G <= 8.
bool gated_unroute_supports(int d, int G);
cudaError_t launch_gated_unroute(const ExpertArgs& a, int G, const __nv_bfloat16* residual, const float* inject,
                                 const __nv_bfloat16* norm_w, float eps, __nv_bfloat16* residual_out,
                                 __nv_bfloat16* normed, cudaStream_t stream);
// Record a message for moe_last_cuda_error on the calling host thread.
void set_last_error_message(const char* msg);

}  // namespace moe
