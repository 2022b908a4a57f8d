// The two steps next to the routed-MoE layer on the Qwen3.8-Flash-Next path:
//
//   router projection  logits[t][e] = sum_c x[t][c] * Wr[e][c] (BF16 inputs, FP32 sums), the
//                      producer of the router's input ("Router: selection and expert-task
//                      production" in "Persistent execution for Flash-Next GGUF on SM70"),
//                      written as the weight-prefetch GEMV of "How I forked vLLM and made
//                      Qwen3.8-Flash-Next decode 1.6x faster on one GPU" (section 5, "PDL
//                      weight-prefetch GEMV"): every CTA copies its whole weight tile into
//                      shared memory before the wait for the preceding kernel and lets the
//                      next kernel launch at once, so that under programmatic dependent
//                      launch the router weights stream while the previous layer finishes;
//   gated un-route     for G residual branches, R'[g] = BF16(R[g] + 2 sigmoid(a[g]) O) and
//                      N[g] = GemmaRMSNorm(R'[g], w[g]) with O the token's weighted sum of its
//                      routes ("TokenSpeed: Qwen3.8-Flash-Next optimisations", section "Residual
//                      update and normalization fusion"): one CTA per token computes O, rounds
//                      each branch's updated residual to BF16, keeps it on chip for the
//                      normalisation and stores both.
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kRouterRows = 16;    // experts per CTA: one m16n8k16 A tile
constexpr int kRouterTokens = 8;   // tokens per CTA: one B tile
constexpr int kRouterWarps = 4;    // K is split over the warps, partial sums added in a fixed order

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Row pitch of the shared-memory tiles: 2d bytes plus 16, so the 8 rows one quarter-warp
// reads fall on different banks.
__host__ __device__ inline int router_pitch(int d) { return 2 * d + 16; }

// grid (E / 16, ceil(T / 8)); 128 threads.  Shared memory: the CTA's 16 weight rows, then its
// 8 hidden rows, then the warps' partial sums.
__global__ void __launch_bounds__(32 * kRouterWarps) router_gemv_kernel(const __nv_bfloat16* __restrict__ hidden,
                                                                        const __nv_bfloat16* __restrict__ wr,
                                                                        float* __restrict__ logits, int T, int d,
                                                                        int E) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int pitch = router_pitch(d);
  uint8_t* ws = smem;                                  // [16][pitch]
  uint8_t* xs = smem + kRouterRows * pitch;            // [8][pitch]
  float* part = reinterpret_cast<float*>(xs + kRouterTokens * pitch);  // [warps][16][8]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kRouterRows, t0 = blockIdx.y * kRouterTokens;
  const int n16 = d / 8;  // 16-byte pieces per row
  // the weight tile does not depend on the preceding kernel: copy it first
  for (int i = tid; i < kRouterRows * n16; i += blockDim.x) {
    const int r = i / n16, p = i - r * n16;
    cp_async_16(smem_addr(ws + r * pitch + 16 * p), wr + static_cast<size_t>(e0 + r) * d + 8 * p);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  pdl_launch_dependents();
  pdl_wait();  // the hidden rows come from the preceding kernel
  const int nt = min(kRouterTokens, T - t0);
  for (int i = tid; i < kRouterTokens * n16; i += blockDim.x) {
    const int r = i / n16, p = i - r * n16;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < nt) v = *reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(t0 + r) * d + 8 * p);
    *reinterpret_cast<uint4*>(xs + r * pitch + 16 * p) = v;
  }
  cp_async_wait_all();
  __syncthreads();
  // warp w: k-steps [w * d / 64, (w + 1) * d / 64) of 16 elements
  const int g = lane >> 2, q = lane & 3;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int ksteps = d / 16 / kRouterWarps;
  const uint8_t* a_lo = ws + g * pitch;
  const uint8_t* a_hi = ws + (g + 8) * pitch;
  const uint8_t* b_row = xs + g * pitch;
  for (int s = 0; s < ksteps; ++s) {
    const int kb = 2 * (16 * (warp * ksteps + s) + 2 * q);  // byte offset of elements (2q, 2q+1)
    const uint32_t a0 = *reinterpret_cast<const uint32_t*>(a_lo + kb);
    const uint32_t a1 = *reinterpret_cast<const uint32_t*>(a_hi + kb);
    const uint32_t a2 = *reinterpret_cast<const uint32_t*>(a_lo + kb + 16);
    const uint32_t a3 = *reinterpret_cast<const uint32_t*>(a_hi + kb + 16);
    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(b_row + kb);
    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(b_row + kb + 16);
    mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
  }
  // D fragment: rows g / g + 8 (experts), columns 2q, 2q + 1 (tokens)
  float* pw = part + warp * (kRouterRows * kRouterTokens);
  pw[g * kRouterTokens + 2 * q] = acc[0];
  pw[g * kRouterTokens + 2 * q + 1] = acc[1];
  pw[(g + 8) * kRouterTokens + 2 * q] = acc[2];
  pw[(g + 8) * kRouterTokens + 2 * q + 1] = acc[3];
  __syncthreads();
  for (int i = tid; i < kRouterRows * kRouterTokens; i += blockDim.x) {
    const int r = i / kRouterTokens, c = i - r * kRouterTokens;
    const int stride = kRouterRows * kRouterTokens;
    const float v = (part[i] + part[stride + i]) + (part[2 * stride + i] + part[3 * stride + i]);
    if (c < nt) logits[static_cast<size_t>(t0 + c) * E + e0 + r] = v;
  }
}

// One CTA per token: O = sum_j w_j y_{pos(t, j)} in slot order (FP32), then per branch the
// gated update, its BF16 rounding, the sum of squares of the rounded values and GemmaRMSNorm.
// Each thread owns groups of 4 consecutive columns (at most kGatedGroups per thread).
constexpr int kGatedThreads = 256;
constexpr int kGatedGroups = 4;  // d <= 4 * 4 * 256 = 4096

struct GatedArgs {
  ExpertArgs a;  // plan, per-route outputs, T, d, k
  int G;
  const __nv_bfloat16* residual;  // [G][T][d]
  const float* inject;            // [T][G]
  const __nv_bfloat16* norm_w;    // [G][d]
  float eps;
  __nv_bfloat16* residual_out;    // [G][T][d], may alias residual
  __nv_bfloat16* normed;          // [G][T][d]
};

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] free from the previous use
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  if (warp == 0) {
    s = lane < kGatedThreads / 32 ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[32] = s;
  }
  __syncthreads();
  return red[32];
}

__global__ void __launch_bounds__(kGatedThreads) gated_unroute_kernel(GatedArgs ga) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[33];
  const ExpertArgs& a = ga.a;
  const int t = blockIdx.x;
  const bool y16 = __ldcg(a.meta + META_YFMT) != 0;
  const int ngroups = a.d / 4;
  float4 o[kGatedGroups];
#pragma unroll
  for (int i = 0; i < kGatedGroups; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // the token's routes, slots in order
  const int* rp = a.route_pos + static_cast<size_t>(t) * a.k;
  const float* rw = a.route_w + static_cast<size_t>(t) * a.k;
  for (int j = 0; j < a.k; ++j) {
    const int pos = __ldg(rp + j);
    if (pos < 0) continue;  // a route to another shard's expert
    const float w = __ldg(rw + j) * (y16 ? kYUnscale : 1.f);
#pragma unroll
    for (int i = 0; i < kGatedGroups; ++i) {
      const int grp = threadIdx.x + i * kGatedThreads;
      if (grp >= ngroups) continue;
      float4 yv;
      if (y16) {
        const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(a.y) +
                                                                static_cast<size_t>(pos) * a.d + 4 * grp));
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        yv = make_float4(lo.x, lo.y, hi.x, hi.y);
      } else {
        yv = __ldcg(reinterpret_cast<const float4*>(a.y + static_cast<size_t>(pos) * a.d + 4 * grp));
      }
      o[i].x += w * yv.x;
      o[i].y += w * yv.y;
      o[i].z += w * yv.z;
      o[i].w += w * yv.w;
    }
  }
  for (int g = 0; g < ga.G; ++g) {
    const float z = ga.inject[static_cast<size_t>(t) * ga.G + g];
    const float gate = 2.f * (1.f / (1.f + expf(-z)));
    const size_t row = (static_cast<size_t>(g) * a.T + t) * a.d;
    float r[kGatedGroups][4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kGatedGroups; ++i) {
      const int grp = threadIdx.x + i * kGatedThreads;
      if (grp >= ngroups) continue;
      const uint2 rb = *reinterpret_cast<const uint2*>(ga.residual + row + 4 * grp);
      const float2 r01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.x));
      const float2 r23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rb.y));
      const float ov[4] = {o[i].x, o[i].y, o[i].z, o[i].w};
      const float rv[4] = {r01.x, r01.y, r23.x, r23.y};
      __nv_bfloat16 nb[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // R + gate * O as the definition writes it (a product, then a sum: no fused multiply-add)
        nb[c] = __float2bfloat16_rn(__fadd_rn(rv[c], __fmul_rn(gate, ov[c])));
        r[i][c] = __bfloat162float(nb[c]);
        ss += r[i][c] * r[i][c];
      }
      uint2 ob;
      ob.x = (static_cast<uint32_t>(__bfloat16_as_ushort(nb[1])) << 16) | __bfloat16_as_ushort(nb[0]);
      ob.y = (static_cast<uint32_t>(__bfloat16_as_ushort(nb[3])) << 16) | __bfloat16_as_ushort(nb[2]);
      *reinterpret_cast<uint2*>(ga.residual_out + row + 4 * grp) = ob;
    }
    const float mean = block_sum(ss, red) / static_cast<float>(a.d);
    const float inv = 1.f / sqrtf(mean + ga.eps);
#pragma unroll
    for (int i = 0; i < kGatedGroups; ++i) {
      const int grp = threadIdx.x + i * kGatedThreads;
      if (grp >= ngroups) continue;
      const uint2 wb = *reinterpret_cast<const uint2*>(ga.norm_w + static_cast<size_t>(g) * a.d + 4 * grp);
      const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb.x));
      const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb.y));
      const float wv[4] = {w01.x, w01.y, w23.x, w23.y};
      float nv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) nv[c] = __fmul_rn(__fmul_rn(r[i][c], inv), 1.f + wv[c]);
      const __nv_bfloat162 n01 = __floats2bfloat162_rn(nv[0], nv[1]);
      const __nv_bfloat162 n23 = __floats2bfloat162_rn(nv[2], nv[3]);
      uint2 ob;
      ob.x = *reinterpret_cast<const uint32_t*>(&n01);
      ob.y = *reinterpret_cast<const uint32_t*>(&n23);
      *reinterpret_cast<uint2*>(ga.normed + row + 4 * grp) = ob;
    }
  }
}

}  // namespace

bool router_gemv_supports(int T, int d, int E) {
  return T >= 1 && E % kRouterRows == 0 && d % (16 * kRouterWarps) == 0 && router_smem_bytes(d) <= 227 * 1024;
}

size_t router_smem_bytes(int d) {
  return static_cast<size_t>(kRouterRows + kRouterTokens) * router_pitch(d) +
         sizeof(float) * kRouterWarps * kRouterRows * kRouterTokens;
}

cudaError_t launch_router_gemv(const __nv_bfloat16* hidden, const __nv_bfloat16* wr, float* logits, int T, int d,
                               int E, cudaStream_t stream) {
  const size_t smem = router_smem_bytes(d);
  cudaError_t e = cudaFuncSetAttribute(router_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(E / kRouterRows, (T + kRouterTokens - 1) / kRouterTokens);
  return launch_pdl(router_gemv_kernel, grid, dim3(32 * kRouterWarps), smem, stream, hidden, wr, logits, T, d, E);
}

bool gated_unroute_supports(int d, int G) { return G >= 1 && G <= 8 && d % 4 == 0 && d <= 4 * kGatedGroups * kGatedThreads; }

cudaError_t launch_gated_unroute(const ExpertArgs& a, int G, const __nv_bfloat16* residual, const float* inject,
                                 const __nv_bfloat16* norm_w, float eps, __nv_bfloat16* residual_out,
                                 __nv_bfloat16* normed, cudaStream_t stream) {
  GatedArgs ga;
  ga.a = a;
  ga.G = G;
  ga.residual = residual;
  ga.inject = inject;
  ga.norm_w = norm_w;
  ga.eps = eps;
  ga.residual_out = residual_out;
  ga.normed = normed;
  return launch_pdl(gated_unroute_kernel, dim3(a.T), dim3(kGatedThreads), 0, stream, ga);
}

}  // namespace moe
