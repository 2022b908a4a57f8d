// CUDA-core expert path: one launch per stage (gate/up, down; the shared un-route kernel
// follows), one warp per weight row, FP32 FMA on weights dequantised through a
// shared-memory E2M1 table.
//
// Kept as the ablation baseline of the tensor-core kernel: it reads each touched
// expert's weights once per group of 8 routed rows (unique-expert reuse without the
// persistent schedule), and it serves as an independent GPU cross-check of the plan,
// the h format and the fixed-order un-route ("Measurements that can accept or reject
// the design" in "Persistent execution for Flash-Next GGUF on SM70": separate reuse from
// persistent scheduling).
#include <cuda_fp8.h>

#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kTok = 8;  // routed rows per pass over a weight row

// E2M1 value of a nibble from its bit fields (sign, 2-bit exponent with bias 1, 1-bit
// mantissa; exponent 0 is subnormal).
__device__ float e2m1_from_bits(int nib) {
  const int e = (nib >> 1) & 3, m = nib & 1;
  const float mag = e == 0 ? 0.5f * m : ldexpf(1.0f + 0.5f * m, e - 1);
  return (nib & 8) ? -mag : mag;
}

__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Dot products of one NVFP4 weight row with up to kTok FP16 activation rows.
// The warp's lanes split K into 8-element words; `rows_ptr[j]` is row j's base.
__device__ void row_dot(const uint8_t* codes, const uint8_t* scales, int K, const float* lut,
                        const __half* const* rows, int nrows, float (&acc)[kTok]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kTok; ++j) acc[j] = 0.f;
  for (int k0 = lane * 8; k0 < K; k0 += 256) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + k0 / 2);
    const float s = e4m3_to_float(scales[k0 / 16]);
    float wv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) wv[q] = lut[(w >> (4 * q)) & 15u] * s;
#pragma unroll
    for (int j = 0; j < kTok; ++j) {
      if (j < nrows) {
        const uint4 xr = *reinterpret_cast<const uint4*>(rows[j] + k0);
        const __half2* xh = reinterpret_cast<const __half2*>(&xr);
        float a = acc[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(xh[q]);
          a = fmaf(wv[2 * q], f.x, a);
          a = fmaf(wv[2 * q + 1], f.y, a);
        }
        acc[j] = a;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kTok; ++j) acc[j] = warp_sum(acc[j]);
}

__global__ void __launch_bounds__(256) simt_gateup_kernel(ExpertArgs a) {
  __shared__ float lut[16];
  pdl_wait();
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_from_bits(threadIdx.x);
  __syncthreads();
  const int u = blockIdx.x;
  if (u >= __ldg(a.meta + META_U)) return;
  const int e = __ldg(a.touched + u);
  const int m = __ldg(a.counts + e), off = __ldg(a.offsets + e);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rowb = static_cast<size_t>(a.d) / 2, rows = static_cast<size_t>(a.d) / 16;
  for (int nn = 0; nn < 4; ++nn) {
    const int n = blockIdx.y * 32 + warp * 4 + nn;
    if (n >= a.F) break;
    const size_t rg = static_cast<size_t>(e - a.e_lo) * 2 * a.F + n, ru = rg + a.F;
    for (int r0 = 0; r0 < m; r0 += kTok) {
      const int nr = min(kTok, m - r0);
      const __half* xr[kTok];
#pragma unroll
      for (int j = 0; j < kTok; ++j)
        xr[j] = a.x16 + static_cast<size_t>(__ldg(a.pos_tok + off + r0 + min(j, nr - 1))) * a.d;
      float g[kTok], up[kTok];
      row_dot(a.w13_codes + rg * rowb, a.w13_scales + rg * rows, a.d, lut, xr, nr, g);
      row_dot(a.w13_codes + ru * rowb, a.w13_scales + ru * rows, a.d, lut, xr, nr, up);
      if (lane < kTok && lane < nr) {
        float gv = 0.f, uv = 0.f;
#pragma unroll
        for (int j = 0; j < kTok; ++j)
          if (j == lane) { gv = g[j]; uv = up[j]; }
        gv *= ts13_of(a, e);
        uv *= ts13_of(a, e);
        float h = gv / (1.0f + __expf(-gv)) * uv * kHScale;
        if (fabsf(h) > 65504.f) {
          atomicOr(a.status, static_cast<int>(MOE_DEV_H_SATURATED));
          h = copysignf(65504.f, h);
        }
        a.hs16[static_cast<size_t>(off + r0 + lane) * a.F + n] = __float2half_rn(h);
      }
    }
  }
}

__global__ void __launch_bounds__(256) simt_down_kernel(ExpertArgs a) {
  __shared__ float lut[16];
  pdl_wait();
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_from_bits(threadIdx.x);
  __syncthreads();
  const int u = blockIdx.x;
  if (u >= __ldg(a.meta + META_U)) return;
  const int e = __ldg(a.touched + u);
  const int m = __ldg(a.counts + e), off = __ldg(a.offsets + e);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rowb = static_cast<size_t>(a.F) / 2, rows = static_cast<size_t>(a.F) / 16;
  for (int rr = 0; rr < 4; ++rr) {
    const int r = blockIdx.y * 32 + warp * 4 + rr;
    if (r >= a.d) break;
    const size_t wr = static_cast<size_t>(e - a.e_lo) * a.d + r;
    for (int r0 = 0; r0 < m; r0 += kTok) {
      const int nr = min(kTok, m - r0);
      const __half* hr[kTok];
#pragma unroll
      for (int j = 0; j < kTok; ++j) hr[j] = a.hs16 + static_cast<size_t>(off + r0 + min(j, nr - 1)) * a.F;
      float y[kTok];
      row_dot(a.w2_codes + wr * rowb, a.w2_scales + wr * rows, a.F, lut, hr, nr, y);
      if (lane < nr) {
        float yv = 0.f;
#pragma unroll
        for (int j = 0; j < kTok; ++j)
          if (j == lane) yv = y[j];
        a.y[static_cast<size_t>(off + r0 + lane) * a.d + r] = yv * ts2_of(a, e) * kHUnscale;
      }
    }
  }
}

}  // namespace

cudaError_t launch_expert_simt(const ExpertArgs& a, cudaStream_t stream) {
  simt_gateup_kernel<<<dim3(a.E, (a.F + 31) / 32), 256, 0, stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  simt_down_kernel<<<dim3(a.E, (a.d + 31) / 32), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
