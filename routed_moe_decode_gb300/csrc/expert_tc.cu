// Persistent weight-stripe expert kernel (gate/up + SiLU*mul, down projection) on the
// 5th-generation tensor core, followed by the fixed-order un-route kernel.
//
// Design (the pages' ideas re-derived for sm_103a; "Persistent execution for Flash-Next
// GGUF on SM70", sections "MonoMoE" and "First implementation boundary"):
//   * one resident CTA per SM takes tasks from the plan's task table through a ticket
//     counter (first ticket = CTA index); every gate/up task precedes every down task in
//     the table, so a CTA waiting on a down task only waits for tasks that resident CTAs
//     already hold (forward progress without a grid barrier);
//   * one warp fetches tickets ahead and publishes the decoded task to the other roles
//     through a shared-memory task ring, so no role decodes tasks from global memory;
//   * each task streams one stripe of one touched expert's NVFP4 weights exactly once,
//     whatever the number of routed rows (unique-expert reuse): TMA tiles of E2M1 codes
//     (64-byte swizzled rows) plus cp.async block scales into a multi-stage ring;
//   * four dequantisation warps turn each 128-row x 128-K chunk into exact FP16
//     (E2M1 x E4M3 has at most 6 significant bits) in registers and store it into
//     tensor memory, where it is the A operand of tcgen05.mma (kind::f16, FP32
//     accumulators in tensor memory); the routed token rows are the N = 16 operand in
//     shared memory (128-byte swizzle), so one weight pass serves up to 64 rows;
//   * gate/up tasks publish a per-expert readiness counter after their FP16 h rows are
//     stored (release); down tasks wait on it (acquire) before loading h, while their
//     weights already stream;
//   * down tasks store per-route FP32 outputs; the un-route kernel then sums the k
//     routes of each token in slot order and adds the residual (fixed-order reduction,
//     no float atomics);
//   * every wait is bounded: on expiry the CTA records MOE_DEV_TIMEOUT, every role stops
//     (warp-uniform decisions), the producer drains its copies, the MMA warp its MMAs,
//     and tensor memory is freed.
//
// Warp roles (352 threads): 0-3 epilogue, 4-7 dequantisation, 8 weight producer and task
// fetcher, 9 activation producer, 10 MMA issuer and tensor-memory owner.
#include "moe_kernels.cuh"

namespace moe {

namespace tc {

constexpr int kStagesA = 14;        // weight ring (codes + scales), released by the dequant warps
constexpr int kStagesB = 16;        // activation ring (one 16-row group per stage), released by the MMA
constexpr int kStageCodes = 8192;   // 2 halves x 64 rows x 64 B (SWIZZLE_64B)
constexpr int kStageScales = 1024;  // 128 rows x 8 B
constexpr int kStageA = kStageCodes + kStageScales;  // 9216, a multiple of 1024
constexpr int kOffScales = kStageCodes;
constexpr int kStageB = 4096;       // one group: 2 atoms x (16 rows x 128 B), SWIZZLE_128B
constexpr int kNumA = 4;            // tensor-memory A buffers (64 columns each)
constexpr int kNumD = 4;            // tensor-memory accumulator buffers (64 columns each)
constexpr int kDCol0 = kNumA * 64;  // first accumulator column
constexpr int kTmemCols = 512;
constexpr int kTaskSlots = 8;
constexpr int kTaskConsumers = 10;  // activation producer, 4 dequant warps, MMA, 4 epilogue warps
constexpr int kThreads = 352;
// Bound of the drain waits at exit (copies and MMAs already issued complete within
// microseconds; after an abort a barrier may lack the arrival of a role that gave up).
constexpr long long kDrainCycles = 1ll << 24;

struct Smem {
  uint8_t ring_b[kStagesB][kStageB];
  uint8_t ring_a[kStagesA][kStageA];
  float xch[kRowsPerPass * 64];  // up-projection values handed to the gate threads
  TaskEntry task[kTaskSlots];
  uint64_t full_a[kStagesA];
  uint64_t empty_a[kStagesA];
  uint64_t full_b[kStagesB];
  uint64_t empty_b[kStagesB];
  uint64_t a_full[kNumA];
  uint64_t a_empty[kNumA];
  uint64_t d_full[kNumD];
  uint64_t d_empty[kNumD];
  uint64_t task_full[kTaskSlots];
  uint64_t task_empty[kTaskSlots];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Decoded task (from a TaskEntry); `valid` is false for the end-of-work sentinel.
struct Task {
  bool valid;
  bool is_dn;
  int e, u, row0, rows, s, nck;
};

__device__ __forceinline__ Task unpack(const TaskEntry& t, const ExpertArgs& a) {
  Task k;
  k.valid = t.x >= 0;
  k.e = t.x & 0xffff;
  k.u = (t.x >> 16) & 0xffff;
  k.row0 = t.y;
  k.rows = t.z & 0xffff;
  k.is_dn = ((t.z >> 16) & 1) != 0;
  k.s = t.w;
  k.nck = k.is_dn ? a.nck_dn : a.nck_gu;
  return k;
}

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, Smem& sm, int* status,
                                             long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
    if (clock64() - t0 > limit) {
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
      atomicOr(status, static_cast<int>(MOE_DEV_TIMEOUT));
      return false;
    }
  }
  return true;
}

// Every lane waits; the warp then agrees on the outcome, so that no lane runs a
// warp-collective (.sync.aligned) instruction that another lane has abandoned.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Smem& sm, int* status, long long limit) {
  const bool ok = bounded_wait(bar, parity, sm, status, limit);
  return __all_sync(0xffffffffu, ok);
}

// Task-ring consumer: wait for slot n, copy the entry, release the slot (one arrival per
// consuming warp, made by lane 0 after the warp has the entry).
__device__ __forceinline__ bool take_task(Smem& sm, int n, TaskEntry& out, int* status, long long limit) {
  const int q = n % kTaskSlots;
  const uint32_t ph = static_cast<uint32_t>((n / kTaskSlots) & 1);
  if (!warp_wait(smem_addr(&sm.task_full[q]), ph, sm, status, limit)) return false;
  out = sm.task[q];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&sm.task_empty[q]));
  return true;
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

// Optional timeline event (lane 0 of a role; no-op unless a trace buffer is given).
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
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(smem_addr(&sm.full_a[i]), 33);  // 32 cp.async arrivals + 1 expect_tx arrival
      mbar_init(smem_addr(&sm.empty_a[i]), 4);  // the four dequantisation warps
    }
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(smem_addr(&sm.full_b[i]), 32);
      mbar_init(smem_addr(&sm.empty_b[i]), 1);  // MMA commit
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(smem_addr(&sm.a_full[i]), 4);
      mbar_init(smem_addr(&sm.a_empty[i]), 1);
    }
    for (int i = 0; i < kNumD; ++i) {
      mbar_init(smem_addr(&sm.d_full[i]), 1);
      mbar_init(smem_addr(&sm.d_empty[i]), 4);
    }
    for (int i = 0; i < kTaskSlots; ++i) {
      mbar_init(smem_addr(&sm.task_full[i]), 1);
      mbar_init(smem_addr(&sm.task_empty[i]), kTaskConsumers);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tm_w13);
    prefetch_tmap(&tm_w2);
  }
  // everything above is local to the CTA; the plan and the counters come from the
  // preceding kernel
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t ringa0 = smem_addr(&sm.ring_a[0][0]);
  const uint32_t ringb0 = smem_addr(&sm.ring_b[0][0]);
  int tcnt = 0;  // trace events of this thread's role
  if (tid == 0) trace_ev(a, 5, tcnt, 10, 0);

  if (warp == 8) {
    // ------------- task fetcher + weight producer: TMA code tiles, cp.async scales -------------
    // Tickets run two tasks ahead: the ticket of task i+2 is taken when task i starts and its
    // table entry is loaded when task i ends, so neither latency stalls the copies.
    const uint64_t pol = policy_evict_first();
    const int ntot = __ldg(a.meta + META_NGU) + __ldg(a.meta + META_NDN);
    const TaskEntry kEnd = TaskEntry{-1, 0, 0, 0};
    int stage = 0, issued = 0, n = 0, chunk_seq = 0;
    uint32_t phase = 0;
    int cur = blockIdx.x, nxt = ntot;  // second ticket: the first dynamic one
    TaskEntry entry = kEnd, entry_nxt = kEnd;
    if (lane == 0) {
      if (cur < ntot) entry = a.tasks[cur];
      if (cur < ntot) {
        nxt = static_cast<int>(atomicAdd(a.ticket, 1u)) + static_cast<int>(gridDim.x);
        if (nxt < ntot) entry_nxt = a.tasks[nxt];
      }
    }
    bool ok = true;
    while (ok) {
      // publish the current task (or the end-of-work sentinel) to the consumers
      const int q = n % kTaskSlots;
      if (!warp_wait(smem_addr(&sm.task_empty[q]), static_cast<uint32_t>(((n / kTaskSlots) & 1) ^ 1), sm,
                     a.status, a.wait_limit)) {
        ok = false;
        break;
      }
      const bool live = __shfl_sync(0xffffffffu, cur, 0) < ntot;
      if (lane == 0) {
        sm.task[q] = live ? entry : kEnd;
        mbar_arrive(smem_addr(&sm.task_full[q]));
        trace_ev(a, 0, tcnt, 1, cur);
      }
      ++n;
      if (!live) break;
      const int x = __shfl_sync(0xffffffffu, entry.x, 0);
      const int z = __shfl_sync(0xffffffffu, entry.z, 0);
      const int s = __shfl_sync(0xffffffffu, entry.w, 0);
      int nxt2 = ntot;
      if (lane == 0 && nxt < ntot) nxt2 = static_cast<int>(atomicAdd(a.ticket, 1u)) + static_cast<int>(gridDim.x);
      const int e = x & 0xffff;
      const bool is_dn = ((z >> 16) & 1) != 0;
      int rA0, rA1, sstride, nck;
      const CUtensorMap* tm;
      const uint8_t* sbase;
      if (!is_dn) {
        rA0 = (e - a.e_lo) * 2 * a.F + s * kGuRows;
        rA1 = rA0 + a.F;
        sstride = a.d / 16;
        tm = &tm_w13;
        sbase = a.w13_scales;
        nck = a.nck_gu;
      } else {
        rA0 = (e - a.e_lo) * a.d + s * kDnRows;
        rA1 = rA0 + 64;
        sstride = a.F / 16;
        tm = &tm_w2;
        sbase = a.w2_scales;
        nck = a.nck_dn;
      }
      for (int c = 0; c < nck; ++c) {
        if (!warp_wait(smem_addr(&sm.empty_a[stage]), phase ^ 1u, sm, a.status, a.wait_limit)) { ok = false; break; }
        const int kb = c * kChunkK;
        const uint32_t sb = ringa0 + stage * kStageA;
        const uint32_t fa = smem_addr(&sm.full_a[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(fa, kStageCodes);
          tma_load_2d(sb, tm, kb / 2, rA0, fa, pol);
          tma_load_2d(sb + kStageCodes / 2, tm, kb / 2, rA1, fa, pol);
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int i = lane + 32 * qq;
          const int grow = i < 64 ? rA0 + i : rA1 + (i - 64);
          cp_async_8(sb + kOffScales + i * 8, sbase + static_cast<size_t>(grow) * sstride + kb / 16);
        }
        cp_async_arrive_noinc(fa);
        if (lane == 0) trace_ev(a, 0, tcnt, 2, chunk_seq);
        ++chunk_seq;
        ++issued;
        if (++stage == kStagesA) { stage = 0; phase ^= 1u; }
      }
      // advance: task i+1 becomes current, task i+2's entry is loaded now
      if (lane == 0) {
        cur = nxt;
        entry = entry_nxt;
        nxt = nxt2;
        entry_nxt = nxt < ntot ? a.tasks[nxt] : kEnd;
      }
    }
    cp_async_wait_all();
    // drain: the last phase issued on every stage must have landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int i = 0; i < min(issued, kStagesA); ++i) {
        if (--st < 0) { st = kStagesA - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_a[st]), ph) && clock64() - t0 < kDrainCycles) {}
      }
    }
  } else if (warp == 9) {
    // ---------------- activation producer: routed rows (FP16) via cp.async ----------------
    int stage = 0, n = 0, chunk_seq = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      if (tk.is_dn) {
        // every gate/up stripe of this expert (all passes) must have published its h rows
        const int npass = (__ldg(a.counts + tk.e) + kRowsPerPass - 1) / kRowsPerPass;
        const uint32_t target = static_cast<uint32_t>(npass * a.S_gu);
        const bool good = warp_wait_counter(a.ready + tk.u, target, &sm.abort_flag, a.status, a.wait_limit);
        if (lane == 0) trace_ev(a, 1, tcnt, 3, n);
        if (!good) break;
      }
      // source row of each routed row of this pass: lanes hold rows lane and lane + 32
      const __half* src0 = nullptr;
      const __half* src1 = nullptr;
      if (tk.is_dn) {
        src0 = a.hs16 + static_cast<size_t>(tk.row0 + lane) * a.F;
        src1 = a.hs16 + static_cast<size_t>(tk.row0 + lane + 32) * a.F;
      } else {
        const int t0 = lane < tk.rows ? __ldg(a.pos_tok + tk.row0 + lane) : 0;
        const int t1 = lane + 32 < tk.rows ? __ldg(a.pos_tok + tk.row0 + lane + 32) : 0;
        src0 = a.x16 + static_cast<size_t>(t0) * a.d;
        src1 = a.x16 + static_cast<size_t>(t1) * a.d;
      }
      const int g = lane & 15;  // 16-byte granule of the 256-byte row chunk
      const int atom = g >> 3, ch = g & 7;
      const int G = (tk.rows + kGroupRows - 1) / kGroupRows;
      for (int c = 0; ok && c < tk.nck; ++c) {
        const int kb = c * kChunkK;
        for (int grp = 0; grp < G; ++grp) {
          if (!warp_wait(smem_addr(&sm.empty_b[stage]), phase ^ 1u, sm, a.status, a.wait_limit)) { ok = false; break; }
          const uint32_t bbase = ringb0 + stage * kStageB;
          const int rend = min(tk.rows, (grp + 1) * kGroupRows);
          for (int r0 = grp * kGroupRows; r0 < rend; r0 += 2) {
            const int r = r0 + (lane >> 4);
            // row r's base pointer lives in lane (r & 31), register src0 (r < 32) or src1
            const __half* p0 = reinterpret_cast<const __half*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src0), r & 31));
            const __half* p1 = reinterpret_cast<const __half*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src1), r & 31));
            if (r < rend) {
              const __half* src = (r < 32 ? p0 : p1) + kb + g * 8;
              const int rr = r & 15;
              const uint32_t dst = bbase + atom * 2048 + (rr >> 3) * 1024 + (rr & 7) * 128 + ((ch ^ (rr & 7)) << 4);
              cp_async_16(dst, src);
            }
          }
          cp_async_arrive_noinc(smem_addr(&sm.full_b[stage]));
          if (++stage == kStagesB) { stage = 0; phase ^= 1u; }
        }
        if (lane == 0) trace_ev(a, 1, tcnt, 4, chunk_seq);
        ++chunk_seq;
      }
    }
    cp_async_wait_all();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- dequantisation: NVFP4 -> FP16 A tile in tensor memory ----------------
    const int i = tid - 128;  // A row of this thread (= tensor-memory lane)
    const int half = i >> 6, r = i & 63;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int stage = 0, abuf = 0, n = 0, chunk_seq = 0, tcnt2 = 0;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.full_a[stage]), phase, sm, a.status, a.wait_limit)) { ok = false; break; }
        if (warp == 4 && lane == 0) trace_ev(a, 2, tcnt, 5, chunk_seq);
        const uint8_t* st = &sm.ring_a[stage][0];
        const uint8_t* crow = st + half * (kStageCodes / 2) + r * 64;
        uint4 q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) q[j] = *reinterpret_cast<const uint4*>(crow + ((j ^ ((r >> 1) & 3)) << 4));
        const uint2 sc = *reinterpret_cast<const uint2*>(st + kOffScales + i * 8);
        uint32_t v[64];
        // block scales s (one per 16 elements) as FP16x2 pairs
        const uint32_t s01 = e4m3x2_to_f16x2(sc.x), s23 = e4m3x2_to_f16x2(sc.x >> 16);
        const uint32_t s45 = e4m3x2_to_f16x2(sc.y), s67 = e4m3x2_to_f16x2(sc.y >> 16);
        const uint32_t sp[4] = {s01, s23, s45, s67};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int wi = 4 * j + h;   // word index in the row chunk (8 elements each)
            const int blk = wi >> 1;    // 16-element scale block
            const uint32_t pair = sp[blk >> 1];
            const uint32_t sraw = (blk & 1) ? bcast_hi_half(pair) : bcast_lo_half(pair);
            uint32_t o0, o1, o2, o3;
            e2m1x8_to_f16x2x4(w[h], o0, o1, o2, o3);
            v[4 * wi + 0] = hmul2_bits(o0, sraw);
            v[4 * wi + 1] = hmul2_bits(o1, sraw);
            v[4 * wi + 2] = hmul2_bits(o2, sraw);
            v[4 * wi + 3] = hmul2_bits(o3, sraw);
          }
        }
        // the weight stage is consumed (its bytes are in registers): hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty_a[stage]));
        if (!warp_wait(smem_addr(&sm.a_empty[abuf]), aphase ^ 1u, sm, a.status, a.wait_limit)) { ok = false; break; }
        if (warp == 4 && lane == 0) trace_ev(a, 7, tcnt2, 15, chunk_seq);
        tc_fence_after();
        tmem_st_x64(tmem + lane_base + abuf * 64, v);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.a_full[abuf]));
        if (warp == 4 && lane == 0) trace_ev(a, 2, tcnt, 6, chunk_seq);
        ++chunk_seq;
        if (++stage == kStagesA) { stage = 0; phase ^= 1u; }
        if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
      }
    }
  } else if (warp == 10) {
    // ---------------- MMA issuer (one lane; the whole warp takes the tasks) ----------------
    const uint32_t idesc = idesc_f16_f32(128, kGroupRows);
    int stage = 0, abuf = 0, dbuf = 0, n = 0, chunk_seq = 0;
    uint32_t phase = 0, aphase = 0, dphase = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      if (lane == 0) {
        const int G = (tk.rows + kGroupRows - 1) / kGroupRows;
        if (!bounded_wait(smem_addr(&sm.d_empty[dbuf]), dphase ^ 1u, sm, a.status, a.wait_limit)) ok = false;
        tc_fence_after();
        const uint32_t dcol = tmem + kDCol0 + dbuf * 64;
        for (int c = 0; ok && c < tk.nck; ++c) {
          if (!bounded_wait(smem_addr(&sm.a_full[abuf]), aphase, sm, a.status, a.wait_limit)) { ok = false; break; }
          trace_ev(a, 6, tcnt, 12, chunk_seq);
          tc_fence_after();
          for (int g = 0; ok && g < G; ++g) {
            const int bst = (stage + g) % kStagesB;
            const uint32_t bph = phase ^ static_cast<uint32_t>((stage + g) >= kStagesB ? 1 : 0);
            if (!bounded_wait(smem_addr(&sm.full_b[bst]), bph, sm, a.status, a.wait_limit)) { ok = false; break; }
            tc_fence_after();
            fence_proxy_async_smem();
            if (g == 0) trace_ev(a, 6, tcnt, 13, chunk_seq);
            const uint32_t bbase = ringb0 + bst * kStageB;
#pragma unroll
            for (int kk = 0; kk < kChunkK / 16; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(bbase + (kk >> 2) * 2048 + (kk & 3) * 32, 1024);
              tc_mma_f16_ts(dcol + g * kGroupRows, tmem + abuf * 64 + kk * 8, bdesc, idesc,
                            (c > 0 || kk > 0) ? 1u : 0u);
            }
            if (g == G - 1) trace_ev(a, 6, tcnt, 14, chunk_seq);
            tc_commit(smem_addr(&sm.empty_b[bst]));
          }
          if (!ok) break;
          tc_commit(smem_addr(&sm.a_empty[abuf]));
          trace_ev(a, 3, tcnt, 7, chunk_seq);
          ++chunk_seq;
          stage += G;
          if (stage >= kStagesB) { stage -= kStagesB; phase ^= 1u; }
          if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
        }
        if (ok) tc_commit(smem_addr(&sm.d_full[dbuf]));
        if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) {
      // every issued MMA completes before tensor memory is released
      tc_commit(smem_addr(&sm.drain));
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_addr(&sm.drain), 0) && clock64() - t0 < kDrainCycles) {}
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 0-3): thread i owns accumulator lane i ----------------
    const int i = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    int dbuf = 0, n = 0;
    uint32_t dphase = 0;
    while (true) {
      TaskEntry te;
      const bool got_task = take_task(sm, n++, te, a.status, a.wait_limit);
      if (!named_bar_and(2, 128, got_task)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      const int G = (tk.rows + kGroupRows - 1) / kGroupRows;
      const bool got = warp_wait(smem_addr(&sm.d_full[dbuf]), dphase, sm, a.status, a.wait_limit);
      if (!named_bar_and(2, 128, got)) break;
      if (tid == 0) trace_ev(a, 4, tcnt, 8, n);
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
      if (tid == 0) trace_ev(a, 4, tcnt, 16, n);
      if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }

      if (!tk.is_dn) {
        // gate/up stripe: up values to the gate threads, h = silu(g) * u stored as FP16
        if (i >= 64) {
#pragma unroll
          for (int c = 0; c < kRowsPerPass; ++c)
            if (c < tk.rows) sm.xch[c * 64 + (i - 64)] = __uint_as_float(accb[c >> 4][c & 15]);
        }
        named_bar_sync(1, 128);
        if (i < 64) {
          const int nidx = tk.s * kGuRows + i;  // element n of h
          const float sc13 = ts13_of(a, tk.e);
#pragma unroll
          for (int c = 0; c < kRowsPerPass; ++c) {
            if (c < tk.rows) {
              const float gv = __uint_as_float(accb[c >> 4][c & 15]) * sc13;
              const float uv = sm.xch[c * 64 + i] * sc13;
              a.hs16[static_cast<size_t>(tk.row0 + c) * a.F + nidx] = h_store_value(silu_mul(gv, uv), a.status);
            }
          }
          __threadfence();
        }
        named_bar_sync(1, 128);
        if (i == 0) atom_add_acqrel_u32(a.ready + tk.u, 1u);
      } else {
        // down stripe: per-route FP32 outputs (summed over routes by the un-route kernel)
        const int rcol = tk.s * kDnRows + i;
        const float scale = ts2_of(a, tk.e) * kHUnscale;
#pragma unroll
        for (int c = 0; c < kRowsPerPass; ++c)
          if (c < tk.rows)
            a.y[static_cast<size_t>(tk.row0 + c) * a.d + rcol] = __uint_as_float(accb[c >> 4][c & 15]) * scale;
      }
      if (tid == 0) trace_ev(a, 4, tcnt, 9, n);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    int c2 = 1;
    trace_ev(a, 5, c2, 11, 0);
  }
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
  return launch_pdl(expert_tc_kernel, dim3(num_sms), dim3(kThreads), smem, stream, tm_w13, tm_w2, a);
}

// ---------------------------------------------------------------------------------
// Un-route: out[t] = residual[t] + sum_{j<k} w_{t,j} y_{pos(t,j)}, slots in order, FP32,
// one BF16 rounding ("First implementation boundary", step 4: routes summed in a fixed
// order).  Each thread owns 4 consecutive columns of one token.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(ExpertArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (c >= a.d) return;
  // the expert kernel that ran records the format of its per-route outputs in the plan meta
  if (__ldcg(a.meta + META_YFMT) != 0) unroute4_y16(a, t, c);
  else unroute4(a, t, c);
}

cudaError_t launch_combine(const ExpertArgs& a, cudaStream_t stream) {
  const dim3 grid(a.T, (a.d / 4 + 255) / 256);
  return launch_pdl(combine_kernel, grid, dim3(256), 0, stream, a);
}

// ---------------------------------------------------------------------------------
// Per-call preparation: zero the counters this call uses and convert the hidden rows to
// FP16 (the tensor-core operand type), flagging values outside the FP16 range.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs p) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t gtid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = gtid; i < static_cast<size_t>(p.E + p.S_dn); i += nthreads) p.ready[i] = 0u;
  if (gtid == 0) *p.ticket = 0u;
  const size_t n8 = static_cast<size_t>(p.T) * p.d / 8;
  bool bad = false;
  for (size_t i = gtid; i < n8; i += nthreads) {
    const uint4 raw = reinterpret_cast<const uint4*>(p.hidden)[i];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 t = __bfloat1622float2(b[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
    uint4 o;
    __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      bad |= !(fabsf(f[2 * q]) <= 65504.f) || !(fabsf(f[2 * q + 1]) <= 65504.f);
      h[q] = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
    }
    reinterpret_cast<uint4*>(p.x16)[i] = o;
  }
  if (bad) atomicOr(p.status, static_cast<int>(MOE_DEV_HIDDEN_RANGE));
}

cudaError_t launch_prep(const PrepArgs& p, cudaStream_t stream) {
  const size_t n8 = static_cast<size_t>(p.T) * p.d / 8;
  const size_t nr = static_cast<size_t>(p.E + p.S_dn);
  size_t work = n8 > nr ? n8 : nr;
  int blocks = static_cast<int>((work + 255) / 256);
  if (blocks > 1184) blocks = 1184;
  if (blocks < 1) blocks = 1;
  return launch_pdl(prep_kernel, dim3(blocks), dim3(256), 0, stream, p);
}

}  // namespace moe
