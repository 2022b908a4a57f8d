// Building blocks shared by the two warp-MMA decode kernels (expert_mma.cu, expert_dec.cu):
// the weight-chunk geometry, bounded mbarrier waits, the m16n8k16 fragment layout, NVFP4
// dequantisation into A fragments and the task-entry helpers.
#pragma once

#include "moe_kernels.cuh"

namespace moe {
namespace mk {

constexpr int kChunk = 256;                     // K elements per chunk (128 B of codes per row)
constexpr int kCodeBytes = 16384;               // codes: 2 halves x 64 rows x 128 B (SWIZZLE_128B)
constexpr int kScaleBytes = 2048;               // block scales: 128 rows x 16 B (the chunk's 16 blocks)
constexpr int kStageA = kCodeBytes + kScaleBytes;
constexpr int kComputeWarps = 8;
constexpr int kFirstCompute = 3;
constexpr int kThreads = 32 * (kFirstCompute + kComputeWarps);
constexpr int kTaskSlots = 8;
// Bound of the drain waits at exit: copies already issued land within microseconds, but after
// an abort a stage's barrier may lack the arrival of a role that gave up, so the drain waits
// this long (~8 ms) at most per barrier rather than for a completion that may never come.
constexpr long long kDrainCycles = 1ll << 24;

// Wait for phase `parity` of mbarrier `bar`, giving up after `limit` cycles (sets *abort_flag
// and MOE_DEV_TIMEOUT) or as soon as another role of the CTA has raised *abort_flag.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, int* abort_flag, int* status,
                                             long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (clock64() - t0 > limit) {
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      atomicOr(status, static_cast<int>(MOE_DEV_TIMEOUT));
      return false;
    }
  }
  return true;
}

// bounded_wait by every lane of a warp, one decision for the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* abort_flag, int* status,
                                          long long limit) {
  const bool ok = bounded_wait(bar, parity, abort_flag, status, limit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool is_unroute(const TaskEntry& t) { return ((t.z >> 18) & 1) != 0; }

// Task i of the ticket order: entry i of the plan's table, or, past its ntask entries, one of
// the a.ncb un-route tasks: stripe c mod S_dn (128 output columns) of the tokens
// [8 (c / S_dn), +8), one token per compute warp (c = i - ntask).
__device__ __forceinline__ TaskEntry task_at(const ExpertArgs& a, int i, int ntask) {
  if (i < ntask) return a.tasks[i];
  const int c = i - ntask;
  return TaskEntry{0, kComputeWarps * (c / a.S_dn), 1 << 18, c % a.S_dn};
}

// Tile row (0..7 within an 8-row group) held by fragment row g: 0, 4, 1, 5, 2, 6, 3, 7.
__device__ __forceinline__ int frag_row(int g) { return ((g & 1) << 2) | (g >> 1); }

// D += A * B for one m16n8k16 step (FP16 inputs, FP32 accumulators).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One thread's share of a 256-K chunk: per sub-chunk h the 16 code bytes and the two block
// scales of its rows a (fragment row g) and b (fragment row g + 8).
struct ChunkCodes {
  uint4 ca[2], cb[2];
  uint32_t sa[2], sb[2];
};

// codes: sub-chunk h covers K [128h, 128h+128); thread q its elements [32q, 32q+32), i.e.
// 16-byte piece 4h + q of the 128-byte row, stored at (piece ^ (row & 7)); scales: the
// chunk's blocks 8h + 2q and 8h + 2q + 1, i.e. bytes 8h + 2q of the row's 16 scale bytes.
__device__ __forceinline__ void load_chunk_codes(const uint8_t* stage, int lra, int lrb, int q, ChunkCodes& o) {
  const int ra = lra & 63, rb = lrb & 63;
  const uint8_t* pa = stage + (lra >> 6) * (kCodeBytes / 2) + ra * 128;
  const uint8_t* pb = stage + (lrb >> 6) * (kCodeBytes / 2) + rb * 128;
  const uint8_t* qa = stage + kCodeBytes + lra * 16 + 2 * q;
  const uint8_t* qb = stage + kCodeBytes + lrb * 16 + 2 * q;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    o.ca[h] = *reinterpret_cast<const uint4*>(pa + (((4 * h + q) ^ (ra & 7)) << 4));
    o.cb[h] = *reinterpret_cast<const uint4*>(pb + (((4 * h + q) ^ (rb & 7)) << 4));
    o.sa[h] = *reinterpret_cast<const uint16_t*>(qa + 8 * h);
    o.sb[h] = *reinterpret_cast<const uint16_t*>(qb + 8 * h);
  }
}

// Dequantise 32 elements (16 bytes of codes, two 16-element scale blocks) of one row into
// 16 FP16x2 registers in fragment order: register 4j + i holds elements (8j + 2i, 8j + 2i + 1).
__device__ __forceinline__ void dequant32(const uint4 codes, uint32_t scale_pair_bytes, uint32_t (&o)[16]) {
  const uint32_t s2 = e4m3x2_to_f16x2(scale_pair_bytes);  // (block 0, block 1)
  const uint32_t sb0 = bcast_lo_half(s2), sb1 = bcast_hi_half(s2);
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t scale = j < 2 ? sb0 : sb1;
    uint32_t r0, r1, r2, r3;
    e2m1x8_to_f16x2x4(w[j], r0, r1, r2, r3);
    o[4 * j + 0] = hmul2_bits(r0, scale);
    o[4 * j + 1] = hmul2_bits(r1, scale);
    o[4 * j + 2] = hmul2_bits(r2, scale);
    o[4 * j + 3] = hmul2_bits(r3, scale);
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

__device__ __forceinline__ __half h_store_value(float h, int* status) {
  float v = h * kHScale;
  if (fabsf(v) > 65504.f) {
    atomicOr(status, static_cast<int>(MOE_DEV_H_SATURATED));
    v = copysignf(65504.f, v);
  }
  return __float2half_rn(v);
}

__device__ __forceinline__ void trace_ev(const ExpertArgs& a, int role, int& cnt, int code, int idx) {
  if (a.trace != nullptr && cnt < kTracePerRole) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    a.trace[(static_cast<size_t>(blockIdx.x) * kTraceRoles + role) * kTracePerRole + cnt] =
        (static_cast<unsigned long long>(code) << 56) | (static_cast<unsigned long long>(idx & 0xffff) << 40) |
        (t & 0xffffffffffull);
    ++cnt;
  }
}

}  // namespace mk
}  // namespace moe
