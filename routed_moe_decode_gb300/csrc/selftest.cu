// Self-test kernels: the expert kernel's building blocks run in isolation (declared in
// include/moe_selftest.h).  Every index is bounded by the sizes the entry points fix.
#include "../../include/moe_selftest.h"
#include "moe_kernels.cuh"

namespace moe {
namespace {

__global__ void selftest_decode_kernel(const uint32_t* words, int n, uint32_t* out, const uint32_t* pairs, int m,
                                       uint32_t* sout) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    uint32_t o0, o1, o2, o3;
    e2m1x8_to_f16x2x4(words[i], o0, o1, o2, o3);
    out[4 * i + 0] = o0;
    out[4 * i + 1] = o1;
    out[4 * i + 2] = o2;
    out[4 * i + 3] = o3;
  }
  if (i < m) sout[i] = e4m3x2_to_f16x2(pairs[i]);
}

__global__ void __launch_bounds__(128) selftest_tma_kernel(const __grid_constant__ CUtensorMap tm, int x, int y,
                                                           uint8_t* out) {
  __shared__ __align__(1024) uint8_t tile[4096];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_addr(&bar), 4096);
    tma_load_2d(smem_addr(tile), &tm, x, y, smem_addr(&bar), policy_evict_first());
  }
  const long long t0 = clock64();
  while (!mbar_try_wait(smem_addr(&bar), 0) && clock64() - t0 < (1ll << 32)) {}
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) out[i] = tile[i];
}

__global__ void __launch_bounds__(128) selftest_mma_kernel(const __half* A, const __half* B, float* D) {
  __shared__ __align__(1024) uint8_t btile[4096];  // 2 atoms x 16 rows x 128 B
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(smem_addr(&tmem_slot), 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  // B rows into the 128-byte-swizzled K-major layout the expert kernel's producer writes
  for (int gidx = tid; gidx < 16 * 16; gidx += 128) {
    const int r = gidx >> 4, g = gidx & 15;
    const int atom = g >> 3, ch = g & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(B + r * 128 + g * 8);
    *reinterpret_cast<uint4*>(btile + atom * 2048 + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // A row `tid` into tensor-memory lane `tid`, columns 0..63 (two FP16 per column)
  uint32_t v[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = reinterpret_cast<const uint32_t*>(A + tid * 128)[j];
  tmem_st_x64(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t idesc = idesc_f16_f32(128, 16);
    const uint32_t bbase = smem_addr(btile);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t bdesc = smem_desc_sw128(bbase + (kk >> 2) * 2048 + (kk & 3) * 32, 1024);
      tc_mma_f16_ts(tmem + 64, tmem + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
    }
    tc_commit(smem_addr(&bar));
  }
  const long long t0 = clock64();
  while (!mbar_try_wait(smem_addr(&bar), 0) && clock64() - t0 < (1ll << 32)) {}
  __syncwarp();
  tc_fence_after();
  uint32_t acc[16];
  tmem_ld_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 64, acc);
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < 16; ++j) D[tid * 16 + j] = __uint_as_float(acc[j]);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_selftest_decode(const uint32_t* words, int n, uint32_t* out, const uint32_t* pairs, int m, uint32_t* sout,
                        moe_stream_t stream) {
  if (n < 0 || m < 0 || (n && (!words || !out)) || (m && (!pairs || !sout))) return MOE_ERR_INVALID_ARG;
  const int total = n > m ? n : m;
  if (total == 0) return MOE_OK;
  moe::selftest_decode_kernel<<<(total + 127) / 128, 128, 0, stream>>>(words, n, out, pairs, m, sout);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_selftest_tma(const uint8_t* src, int rows, int row_bytes, int x, int y, uint8_t* out, moe_stream_t stream) {
  if (!src || !out || rows < 64 || row_bytes < 64 || row_bytes % 16 || x < 0 || y < 0 || x % 16 ||
      x + 64 > row_bytes || y + 64 > rows)
    return MOE_ERR_INVALID_ARG;
  CUtensorMap tm;
  int rc = moe::encode_codes_map(&tm, src, static_cast<uint64_t>(row_bytes), static_cast<uint64_t>(rows), 64);
  if (rc != MOE_OK) return rc;
  moe::selftest_tma_kernel<<<1, 128, 0, stream>>>(tm, x, y, out);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_selftest_mma(const void* A, const void* B, float* D, moe_stream_t stream) {
  if (!A || !B || !D) return MOE_ERR_INVALID_ARG;
  moe::selftest_mma_kernel<<<1, 128, 0, stream>>>(static_cast<const __half*>(A), static_cast<const __half*>(B), D);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
