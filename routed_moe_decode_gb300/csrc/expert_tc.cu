// Persistent weight-stripe expert kernel (gate/up + SiLU*mul, down + weighted un-route)
// on the 5th-generation tensor core.
//
// Design (the pages' ideas re-derived for sm_103a; "Persistent execution for Flash-Next
// GGUF on SM70", sections "MonoMoE" and "First implementation boundary"):
//   * one resident CTA per SM walks a static list of tasks; every gate/up task id is
//     below every down task id, so a CTA that waits on a down task only waits for work
//     that resident CTAs already own (forward progress without a grid barrier);
//   * each task streams one stripe of one touched expert's NVFP4 weights exactly once,
//     whatever the number of routed rows (unique-expert reuse): TMA tiles of E2M1 codes
//     (64-byte swizzled rows) plus cp.async block scales into a multi-stage ring;
//   * four dequantisation warps turn each 128-row x 128-K chunk into exact FP16
//     (E2M1 x E4M3 has at most 6 significant bits) in registers and store it into
//     tensor memory, where it is the A operand of tcgen05.mma (kind::f16, FP32
//     accumulators in tensor memory); the routed token rows are the N = 16 operand in
//     shared memory (128-byte swizzle), so one weight pass serves up to 64 rows;
//   * gate/up tasks publish per-expert readiness counters after their FP16 h rows are
//     stored (release); down tasks wait on them (acquire) before loading h, while their
//     weights already stream;
//   * down tasks write per-route FP32 outputs; the CTA whose counter increment completes
//     a (token, 128-column stripe) sums the k routes in slot order, adds the residual
//     and writes BF16 (fixed-order reduction, no float atomics);
//   * every wait is bounded: on expiry the CTA records MOE_DEV_TIMEOUT, drains its own
//     copies and MMAs, frees tensor memory and returns.
//
// Warp roles (352 threads): 0-3 epilogue, 4-7 dequantisation, 8 weight producer (TMA +
// scales), 9 activation producer (cp.async), 10 MMA issuer and tensor-memory owner.
#include "moe_kernels.cuh"

namespace moe {

namespace tc {

constexpr int kStages = 7;
constexpr int kStageCodes = 8192;   // 2 halves x 64 rows x 64 B (SWIZZLE_64B)
constexpr int kStageScales = 1024;  // 128 rows x 8 B
constexpr int kStageB = 16384;      // 4 groups x 2 atoms x (16 rows x 128 B), SWIZZLE_128B
constexpr int kOffScales = kStageCodes;
constexpr int kOffB = kStageCodes + kStageScales;  // 9216, 1024-aligned
constexpr int kStageBytes = kStageCodes + kStageScales + kStageB;
constexpr int kNumA = 4;            // tensor-memory A buffers (64 columns each)
constexpr int kNumD = 2;            // tensor-memory accumulator buffers (64 columns each)
constexpr int kDCol0 = kNumA * 64;  // first accumulator column
constexpr int kTmemCols = 512;
constexpr int kThreads = 352;
constexpr long long kTimeoutCycles = 1ll << 33;  // ~4 s at 2 GHz

struct Smem {
  uint8_t ring[kStages][kStageBytes];
  float xch[kRowsPerPass * 64];  // up-projection values handed to the gate threads
  uint64_t full_a[kStages];
  uint64_t full_b[kStages];
  uint64_t empty[kStages];
  uint64_t a_full[kNumA];
  uint64_t a_empty[kNumA];
  uint64_t d_full[kNumD];
  uint64_t d_empty[kNumD];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
  int comb_tok[kRowsPerPass];
};

struct Task {
  int is_dn, u, e, pass, s, part, row0, rows, nck, gid;
};

__device__ __forceinline__ Task decode_task(const ExpertArgs& a, int t, int U, int ngu) {
  Task k{};
  const bool dn = t >= ngu;
  const int* start = dn ? a.dn_start : a.gu_start;
  int local = dn ? t - ngu : t;
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(start + mid) <= local) lo = mid;
    else hi = mid;
  }
  local -= __ldg(start + lo);
  k.is_dn = dn;
  k.u = lo;
  k.e = __ldg(a.touched + lo);
  k.gid = t;
  if (!dn) {
    const int per_pass = a.S_gu * a.KS;
    k.pass = local / per_pass;
    const int rem = local - k.pass * per_pass;
    k.s = rem / a.KS;
    k.part = rem - k.s * a.KS;
    k.nck = a.nck_gu;
  } else {
    k.pass = local / a.S_dn;
    k.s = local - k.pass * a.S_dn;
    k.part = 0;
    k.nck = a.nck_dn;
  }
  const int m = __ldg(a.counts + k.e);
  k.row0 = __ldg(a.offsets + k.e) + k.pass * kRowsPerPass;
  k.rows = min(kRowsPerPass, m - k.pass * kRowsPerPass);
  return k;
}

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, Smem& sm, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
      atomicOr(status, static_cast<int>(MOE_DEV_TIMEOUT));
      return false;
    }
  }
  return true;
}

// Every lane waits; the warp then agrees on the outcome, so that no lane runs a
// warp-collective (.sync.aligned) instruction that another lane has abandoned.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Smem& sm, int* status) {
  const bool ok = bounded_wait(bar, parity, sm, status);
  return __all_sync(0xffffffffu, ok);
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

}  // namespace tc

using namespace tc;

__global__ void __launch_bounds__(kThreads, 1)
    expert_tc_kernel(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                     const __grid_constant__ ExpertArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 10) {
    tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_addr(&sm.full_a[i]), 33);  // 32 cp.async arrivals + 1 expect_tx arrival
      mbar_init(smem_addr(&sm.full_b[i]), 32);
      mbar_init(smem_addr(&sm.empty[i]), 1);
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(smem_addr(&sm.a_full[i]), 4);
      mbar_init(smem_addr(&sm.a_empty[i]), 1);
    }
    for (int i = 0; i < kNumD; ++i) {
      mbar_init(smem_addr(&sm.d_full[i]), 1);
      mbar_init(smem_addr(&sm.d_empty[i]), 4);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_w13);
    prefetch_tmap(&tm_w2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  const int U = __ldg(a.meta + META_U);
  const int ngu = __ldg(a.meta + META_NGU);
  const int ntot = ngu + __ldg(a.meta + META_NDN);
  const uint32_t ring0 = smem_addr(&sm.ring[0][0]);

  if (warp == 8) {
    // ---------------- weight producer: TMA code tiles + cp.async block scales ----------------
    const uint64_t pol = policy_evict_first();
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < ntot; t += gridDim.x) {
      const Task tk = decode_task(a, t, U, ngu);
      int rA0, rA1, sstride;
      const CUtensorMap* tm;
      const uint8_t* sbase;
      if (!tk.is_dn) {
        rA0 = tk.e * 2 * a.F + tk.s * kGuRows;
        rA1 = rA0 + a.F;
        sstride = a.d / 16;
        tm = &tm_w13;
        sbase = a.w13_scales;
      } else {
        rA0 = tk.e * a.d + tk.s * kDnRows;
        rA1 = rA0 + 64;
        sstride = a.F / 16;
        tm = &tm_w2;
        sbase = a.w2_scales;
      }
      const int kpart = tk.is_dn ? 0 : tk.part * (a.d / a.KS);
      bool ok = true;
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, sm, a.status)) { ok = false; break; }
        const int kb = kpart + c * kChunkK;
        const uint32_t sbase_smem = ring0 + stage * kStageBytes;
        const uint32_t fa = smem_addr(&sm.full_a[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(fa, kStageCodes);
          tma_load_2d(sbase_smem, tm, kb / 2, rA0, fa, pol);
          tma_load_2d(sbase_smem + kStageCodes / 2, tm, kb / 2, rA1, fa, pol);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = lane + 32 * q;
          const int grow = i < 64 ? rA0 + i : rA1 + (i - 64);
          cp_async_8(sbase_smem + kOffScales + i * 8, sbase + static_cast<size_t>(grow) * sstride + kb / 16);
        }
        cp_async_arrive_noinc(fa);
        ++issued;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    cp_async_wait_all();
    // drain: the last phase issued on every stage must have landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int n = 0; n < min(issued, kStages); ++n) {
        if (--st < 0) { st = kStages - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_a[st]), ph) && clock64() - t0 < kTimeoutCycles) {}
      }
    }
  } else if (warp == 9) {
    // ---------------- activation producer: routed rows (FP16) via cp.async ----------------
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < ntot; t += gridDim.x) {
      const Task tk = decode_task(a, t, U, ngu);
      bool ok = true;
      if (tk.is_dn) {
        // all gate/up stripes of this expert (every pass) must have published h
        const int npass = (__ldg(a.counts + tk.e) + kRowsPerPass - 1) / kRowsPerPass;
        const uint32_t target = static_cast<uint32_t>(npass * a.S_gu);
        if (lane == 0) {
          const long long t0 = clock64();
          while (ld_acquire_u32(a.ready + tk.u) < target) {
            if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) { ok = false; break; }
            if (clock64() - t0 > kTimeoutCycles) {
              *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
              atomicOr(a.status, static_cast<int>(MOE_DEV_TIMEOUT));
              ok = false;
              break;
            }
            __nanosleep(64);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      const int kpart = tk.is_dn ? 0 : tk.part * (a.d / a.KS);
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, sm, a.status)) { ok = false; break; }
        const int kb = kpart + c * kChunkK;
        const uint32_t bbase = ring0 + stage * kStageBytes + kOffB;
        const int g = lane & 15;  // 16-byte granule of the 256-byte row chunk
        for (int r0 = 0; r0 < tk.rows; r0 += 2) {
          const int r = r0 + (lane >> 4);
          if (r < tk.rows) {
            const __half* src = tk.is_dn ? a.hs16 + static_cast<size_t>(tk.row0 + r) * a.F + kb + g * 8
                                         : a.x16 + static_cast<size_t>(__ldg(a.pos_tok + tk.row0 + r)) * a.d + kb + g * 8;
            const int atom = g >> 3, ch = g & 7, grp = r >> 4, rr = r & 15;
            const uint32_t dst = bbase + grp * 4096 + atom * 2048 + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                 ((ch ^ (rr & 7)) << 4);
            cp_async_16(dst, src);
          }
        }
        cp_async_arrive_noinc(smem_addr(&sm.full_b[stage]));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    cp_async_wait_all();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- dequantisation: NVFP4 -> FP16 A tile in tensor memory ----------------
    const int i = tid - 128;           // A row of this thread (= tensor-memory lane)
    const int half = i >> 6, r = i & 63;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int stage = 0, abuf = 0;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntot && ok; t += gridDim.x) {
      const Task tk = decode_task(a, t, U, ngu);
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.full_a[stage]), phase, sm, a.status)) { ok = false; break; }
        if (!warp_wait(smem_addr(&sm.a_empty[abuf]), aphase ^ 1u, sm, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* st = &sm.ring[stage][0];
        const uint8_t* crow = st + half * (kStageCodes / 2) + r * 64;
        uint4 q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) q[j] = *reinterpret_cast<const uint4*>(crow + ((j ^ ((r >> 1) & 3)) << 4));
        const uint2 sc = *reinterpret_cast<const uint2*>(st + kOffScales + i * 8);
        uint32_t v[64];
        const uint32_t s01 = e4m3x2_to_f16x2(sc.x), s23 = e4m3x2_to_f16x2(sc.x >> 16);
        const uint32_t s45 = e4m3x2_to_f16x2(sc.y), s67 = e4m3x2_to_f16x2(sc.y >> 16);
        const uint32_t sb[8] = {bcast_lo_half(s01), bcast_hi_half(s01), bcast_lo_half(s23), bcast_hi_half(s23),
                                bcast_lo_half(s45), bcast_hi_half(s45), bcast_lo_half(s67), bcast_hi_half(s67)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint32_t scale = sb[2 * j + (h >> 1)];  // 16 elements (2 words) per block
            uint32_t o0, o1, o2, o3;
            e2m1x8_to_f16x2x4(w[h], o0, o1, o2, o3);
            v[16 * j + 4 * h + 0] = hmul2_bits(o0, scale);
            v[16 * j + 4 * h + 1] = hmul2_bits(o1, scale);
            v[16 * j + 4 * h + 2] = hmul2_bits(o2, scale);
            v[16 * j + 4 * h + 3] = hmul2_bits(o3, scale);
          }
        }
        tmem_st_x64(tmem + lane_base + abuf * 64, v);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.a_full[abuf]));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
      }
    }
  } else if (warp == 10) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(128, kGroupRows);
      int stage = 0, abuf = 0, dbuf = 0;
      uint32_t phase = 0, aphase = 0, dphase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntot && ok; t += gridDim.x) {
        const Task tk = decode_task(a, t, U, ngu);
        const int G = (tk.rows + kGroupRows - 1) / kGroupRows;
        if (!bounded_wait(smem_addr(&sm.d_empty[dbuf]), dphase ^ 1u, sm, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dcol = tmem + kDCol0 + dbuf * 64;
        for (int c = 0; c < tk.nck; ++c) {
          if (!bounded_wait(smem_addr(&sm.full_b[stage]), phase, sm, a.status)) { ok = false; break; }
          if (!bounded_wait(smem_addr(&sm.a_full[abuf]), aphase, sm, a.status)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();
          const uint32_t bbase = ring0 + stage * kStageBytes + kOffB;
          for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int kk = 0; kk < kChunkK / 16; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(bbase + g * 4096 + (kk >> 2) * 2048 + (kk & 3) * 32, 1024);
              tc_mma_f16_ts(dcol + g * kGroupRows, tmem + abuf * 64 + kk * 8, bdesc, idesc,
                            (c > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(smem_addr(&sm.a_empty[abuf]));
          tc_commit(smem_addr(&sm.empty[stage]));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(smem_addr(&sm.d_full[dbuf]));
        if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }
      }
      // all issued MMAs complete before tensor memory is released
      tc_commit(smem_addr(&sm.drain));
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_addr(&sm.drain), 0) && clock64() - t0 < kTimeoutCycles) {}
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 0-3): thread i owns accumulator lane i ----------------
    const int i = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    int dbuf = 0;
    uint32_t dphase = 0;
    for (int t = blockIdx.x; t < ntot; t += gridDim.x) {
      const Task tk = decode_task(a, t, U, ngu);
      const int G = (tk.rows + kGroupRows - 1) / kGroupRows;
      const bool got = warp_wait(smem_addr(&sm.d_full[dbuf]), dphase, sm, a.status);
      if (!named_bar_and(2, 128, got)) break;
      tc_fence_after();
      uint32_t accb[kMaxGroups][16];
#pragma unroll
      for (int g = 0; g < kMaxGroups; ++g) {
        if (g < G) tmem_ld_x16(tmem + lane_base + kDCol0 + dbuf * 64 + g * kGroupRows, accb[g]);
      }
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.d_empty[dbuf]));
      if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }
      float acc[kRowsPerPass];
#pragma unroll
      for (int c = 0; c < kRowsPerPass; ++c) acc[c] = __uint_as_float(accb[c >> 4][c & 15]);

      if (!tk.is_dn) {
        bool have = true;
        if (a.KS > 1) {
          // split-K partial: store, then the last of the KS parts reduces in part order
          const int col = i < 64 ? tk.s * kGuRows + i : a.F + tk.s * kGuRows + (i - 64);
          float* base = a.gu_part + (static_cast<size_t>(tk.part) * a.R + tk.row0) * (2 * a.F) + col;
#pragma unroll
          for (int c = 0; c < kRowsPerPass; ++c)
            if (c < tk.rows) base[static_cast<size_t>(c) * 2 * a.F] = acc[c];
          __threadfence();
          named_bar_sync(1, 128);
          if (i == 0) {
            const uint32_t old = atom_add_acqrel_u32(a.cnt_gu + tk.gid / a.KS, 1u);
            sm.last_flag = (old == static_cast<uint32_t>(a.KS - 1)) ? 1 : 0;
          }
          named_bar_sync(1, 128);
          have = sm.last_flag != 0;
          if (have) {
            __threadfence();
            const float* pb = a.gu_part + static_cast<size_t>(tk.row0) * (2 * a.F) + col;
#pragma unroll
            for (int c = 0; c < kRowsPerPass; ++c) {
              if (c < tk.rows) {
                float v = 0.f;
                for (int p = 0; p < a.KS; ++p) v += __ldcg(pb + (static_cast<size_t>(p) * a.R + c) * 2 * a.F);
                acc[c] = v;
              }
            }
          }
        }
        if (have) {
          if (i >= 64) {
#pragma unroll
            for (int c = 0; c < kRowsPerPass; ++c)
              if (c < tk.rows) sm.xch[c * 64 + (i - 64)] = acc[c];
          }
          named_bar_sync(1, 128);
          if (i < 64) {
            const int n = tk.s * kGuRows + i;
#pragma unroll
            for (int c = 0; c < kRowsPerPass; ++c) {
              if (c < tk.rows) {
                const float g = acc[c] * a.w13_ts;
                const float u = sm.xch[c * 64 + i] * a.w13_ts;
                a.hs16[static_cast<size_t>(tk.row0 + c) * a.F + n] = h_store_value(silu_mul(g, u), a.status);
              }
            }
          }
          __threadfence();
          named_bar_sync(1, 128);
          if (i == 0) atom_add_acqrel_u32(a.ready + tk.u, 1u);
        }
      } else {
        // down stripe: per-route FP32 outputs, then fixed-order combine by the last arrival
        const int rcol = tk.s * kDnRows + i;
        const float scale = a.w2_ts * kHUnscale;
#pragma unroll
        for (int c = 0; c < kRowsPerPass; ++c)
          if (c < tk.rows) a.y[static_cast<size_t>(tk.row0 + c) * a.d + rcol] = acc[c] * scale;
        __threadfence();
        named_bar_sync(1, 128);
        if (i < tk.rows) {
          const int tok = __ldg(a.pos_tok + tk.row0 + i);
          const uint32_t old = atom_add_acqrel_u32(a.comb_cnt + static_cast<size_t>(tok) * a.S_dn + tk.s, 1u);
          sm.comb_tok[i] = (old == static_cast<uint32_t>(a.k - 1)) ? tok : -1;
        }
        named_bar_sync(1, 128);
        __threadfence();
        for (int c = 0; c < tk.rows; ++c) {
          const int tok = sm.comb_tok[c];
          if (tok < 0) continue;
          float accum = 0.f;
          for (int j = 0; j < a.k; ++j) {
            const int pos = __ldg(a.route_pos + tok * a.k + j);
            const float w = __ldg(a.route_w + tok * a.k + j);
            accum += w * __ldcg(a.y + static_cast<size_t>(pos) * a.d + rcol);
          }
          const size_t o = static_cast<size_t>(tok) * a.d + rcol;
          const float res = a.residual ? __bfloat162float(a.residual[o]) : 0.f;
          a.out[o] = __float2bfloat16_rn(res + accum);
        }
        named_bar_sync(1, 128);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t expert_tc_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_expert_tc(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                             int num_sms, cudaStream_t stream) {
  const size_t smem = expert_tc_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  expert_tc_kernel<<<num_sms, kThreads, smem, stream>>>(tm_w13, tm_w2, a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// Per-call preparation: zero the counters this call uses and convert the hidden rows to
// FP16 (the tensor-core operand type), flagging values outside the FP16 range.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs p) {
  const size_t gtid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = gtid; i < static_cast<size_t>(p.E); i += nthreads) p.ready[i] = 0u;
  for (size_t i = gtid; i < static_cast<size_t>(p.max_units); i += nthreads) p.cnt_gu[i] = 0u;
  for (size_t i = gtid; i < static_cast<size_t>(p.T) * p.S_dn; i += nthreads) p.comb_cnt[i] = 0u;
  const size_t n8 = static_cast<size_t>(p.T) * p.d / 8;
  bool bad = false;
  for (size_t i = gtid; i < n8; i += nthreads) {
    const uint4 raw = reinterpret_cast<const uint4*>(p.hidden)[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      bad |= !(fabsf(f.x) <= 65504.f) || !(fabsf(f.y) <= 65504.f);
      h[j] = __floats2half2_rn(f.x, f.y);
    }
    reinterpret_cast<uint4*>(p.x16)[i] = o;
  }
  if (bad) atomicOr(p.status, static_cast<int>(MOE_DEV_HIDDEN_RANGE));
}

cudaError_t launch_prep(const PrepArgs& p, cudaStream_t stream) {
  const size_t n8 = static_cast<size_t>(p.T) * p.d / 8;
  size_t work = n8;
  if (static_cast<size_t>(p.T) * p.S_dn > work) work = static_cast<size_t>(p.T) * p.S_dn;
  if (static_cast<size_t>(p.max_units) > work) work = p.max_units;
  int blocks = static_cast<int>((work + 255) / 256);
  if (blocks > 1184) blocks = 1184;
  if (blocks < 1) blocks = 1;
  prep_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
