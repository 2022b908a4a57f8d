// Expert kernel for many routed rows per expert (prefill chunks): the weight-stripe task of
// the persistent tcgen05 kernel, with up to kWideRows (192) routed rows per weight pass in
// ONE tcgen05.mma per 16-element K step (N = the pass's rows rounded up to 16).
//
// "Persistent execution for Flash-Next GGUF on SM70", sections "MonoMoE" and "First
// implementation boundary", restated for sm_103a: one resident CTA per SM takes tasks through
// a ticket counter; every gate/up task precedes every down task, so a CTA that waits on a down
// task only waits for work resident CTAs already hold.  A task streams one 128-row stripe of
// one touched expert's NVFP4 weights once per pass, whatever the pass's row count.
//
// Warp roles (480 threads):
//   0-7   epilogue, two groups of four warps taking alternate 32-column slices of an
//         accumulator; thread t owns accumulator lane t % 128.  Gate/up tasks exchange half of
//         the gate and up values between the lane halves through shared memory, so that all
//         128 threads of a group form h = silu(g) * u (FP16); down tasks store per-route
//         outputs as FP16(y * 2^-4) (summed by the un-route kernel in slot order, in FP32);
//         both leave through shared-memory staging in 16-byte stores;
//   8-11  dequantisation: thread i owns A row i; each 128-K chunk of E2M1 codes (TMA tile,
//         64-byte swizzle) and its E4M3 block scales become exact FP16 in registers and are
//         stored into tensor memory, where they are the A operand (M = 128);
//   12    task fetcher + weight producer (TMA codes, cp.async scales);
//   13    activation producer: the pass's routed rows as 128-byte swizzled K-major tiles, the
//         B operand (N up to 192), by TMA: one box of 64, 128 or 192 rows per 64-K atom.  The
//         rows of a pass are contiguous: for gate/up the FP16 hidden rows in route order
//         (wide_gather_kernel writes them before this kernel), for down the expert's h rows;
//   14    MMA issuer and tensor-memory owner: 8 kind::f16 MMAs per chunk into one of two
//         accumulator buffers, so the epilogue of a task overlaps the next task's MMAs; the
//         warp waits and forms the descriptors, one elected lane issues.
// Tensor memory (512 columns): two A buffers of 64 columns, two accumulators of 192 columns.
#include "moe_kernels.cuh"

namespace moe {

namespace wd {

constexpr int kStagesA = 6;                          // weight ring (codes + scales)
constexpr int kStagesB = 3;                          // activation ring (one chunk each)
constexpr int kStageCodes = 8192;                    // 2 halves x 64 rows x 64 B (SWIZZLE_64B)
constexpr int kStageScales = 1024;                   // 128 rows x 8 B
constexpr int kStageA = kStageCodes + kStageScales;  // 9216, a multiple of 1024
constexpr int kAtomB = kWideRows * 128;              // one 64-K atom of a B tile (24576 B)
constexpr int kStageB = 2 * kAtomB;                  // a 128-K chunk of up to 192 rows
constexpr int kNumA = 2;                             // A buffers (64 columns each)
constexpr int kNumD = 2;                             // accumulators (kWideRows columns each)
constexpr int kDCol0 = kNumA * 64;
constexpr int kTmemCols = 512;
constexpr int kTaskSlots = 8;
constexpr int kActWarps = 1;
constexpr int kEpiWarps = 8;   // two groups of four: alternate 32-column slices of an accumulator
constexpr int kWarpDeq0 = kEpiWarps;                           // 8-11
constexpr int kWarpFetch = kWarpDeq0 + 4;                      // 12
constexpr int kWarpAct0 = kWarpFetch + 1;                      // 13
constexpr int kWarpMma = kWarpAct0 + kActWarps;                // 14
constexpr int kThreads = 32 * (kWarpMma + 1);                  // 480
constexpr int kBoxRows = 64;                                   // activation box heights: 64, 128, 192 rows
constexpr int kBoxMaps = kWideRows / kBoxRows;                 // tensor maps per activation operand
static_assert(kBoxMaps == 3, "WideActMaps holds three box heights");
constexpr int kTaskConsumers = kActWarps + 4 + 1 + kEpiWarps;  // activation, dequant, MMA, epilogue warps
// Bound of the drain waits at exit (copies and MMAs already issued complete within
// microseconds; after an abort a barrier may lack the arrival of a role that gave up).
constexpr long long kDrainCycles = 1ll << 24;

static_assert(kDCol0 + kNumD * kWideRows <= kTmemCols, "tensor memory budget");
static_assert(kWideRows % 16 == 0 && kWideRows <= 256, "MMA N limit");

struct Smem {
  uint8_t ring_b[kStagesB][kStageB];
  uint8_t ring_a[kStagesA][kStageA];
  // per epilogue group: gate/up values exchanged between lane halves; the FP16 down outputs
  // of a 32-column slice staged for row-contiguous stores
  float xch[2][32 * 64];
  // per epilogue group: the FP16 h values of a slice, two routed rows per word
  uint32_t hstage[2][16 * 64];
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

struct Task {
  bool valid, is_dn;
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

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Smem& sm, int* status, long long limit) {
  const bool ok = bounded_wait(bar, parity, sm, status, limit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool take_task(Smem& sm, int n, TaskEntry& out, int* status, long long limit) {
  const int q = n % kTaskSlots;
  const uint32_t ph = static_cast<uint32_t>((n / kTaskSlots) & 1);
  if (!warp_wait(smem_addr(&sm.task_full[q]), ph, sm, status, limit)) return false;
  out = sm.task[q];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&sm.task_empty[q]));
  return true;
}

// Two FP32 values to FP16 (round to nearest), magnitudes past the FP16 range clamped to
// +-65504 (NaN stays NaN); lo in the low half.
__device__ __forceinline__ uint32_t f16x2_satfinite(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// MMA N for a pass of `rows` routed rows: a multiple of 16 (kind::f16 with M = 128).
__device__ __forceinline__ int mma_n(int rows) { return (rows + 15) & ~15; }

}  // namespace wd

using namespace wd;

// ---------------------------------------------------------------------------------
// Task table of the wide kernel, built from the plan's per-expert arrays (touched list,
// counts, offsets): per touched expert, passes of kWideRows rows; all gate/up tasks
// (touched order, pass, stripe) first, then all down tasks.  Each 1024-thread CTA scans the
// pass counts of all touched experts (one thread each, U <= E <= 1024) and writes the entries
// of its share of them: one CTA alone writes a few hundred KB slowly.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) wide_plan_kernel(const int* meta_in, int* meta, const int* touched,
                                                         const int* counts, const int* offsets, TaskEntry* tasks,
                                                         int S_gu, int S_dn) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int U = __ldcg(meta_in + META_U);
  int e = 0, m = 0, np = 0;
  if (tid < U) {
    e = __ldcg(touched + tid);
    m = __ldcg(counts + e);
    np = (m + kWideRows - 1) / kWideRows;
  }
  // exclusive scan of the pass counts over the block
  int incl = np;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    s_warp[lane] = wi - w;  // exclusive prefix of the warp totals
    if (lane == 31) s_total = wi;
  }
  __syncthreads();
  const int before = s_warp[warp] + incl - np;
  const int total = s_total;
  // one warp per touched expert writes its passes' entries, one lane per stripe, so that each
  // store instruction covers consecutive entries
  __shared__ int s_e[1024], s_m[1024], s_before[1024], s_base[1024];
  if (tid < U) {
    s_e[tid] = e;
    s_m[tid] = m;
    s_before[tid] = before;
    s_base[tid] = __ldcg(offsets + e);
  }
  __syncthreads();
  int4* tasks4 = reinterpret_cast<int4*>(tasks);
  for (int u = blockIdx.x * 32 + warp; u < U; u += 32 * gridDim.x) {
    const int eu = s_e[u], mu = s_m[u], npu = (mu + kWideRows - 1) / kWideRows;
    for (int p = 0; p < npu; ++p) {
      const int rows = min(kWideRows, mu - p * kWideRows);
      const int z = rows | (npu > 1 ? 1 << 17 : 0);
      const int row0 = s_base[u] + p * kWideRows;
      const int P = s_before[u] + p;
      for (int s2 = lane; s2 < S_gu; s2 += 32) tasks4[P * S_gu + s2] = make_int4(eu | (u << 16), row0, z, s2);
      for (int s2 = lane; s2 < S_dn; s2 += 32)
        tasks4[total * S_gu + P * S_dn + s2] = make_int4(eu | (u << 16), row0, z | (1 << 16), s2);
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    meta[META_WGU] = total * S_gu;
    meta[META_WDN] = total * S_dn;
    meta[META_YFMT] = 1;  // this kernel's down tasks store FP16(y * 2^-4)
  }
}

// ---------------------------------------------------------------------------------
// The FP16 hidden rows in route order, xs[pos] = x16[pos_tok[pos]] for the plan's routed rows,
// so that the rows of every gate/up pass are contiguous (TMA boxes instead of row gathers).
// One warp per row at a time, 16-byte pieces, last positions first: the rows written last,
// still in L2 when the wide kernel starts, are those of the first experts, which it reads first.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) wide_gather_kernel(const __half* __restrict__ x16, const int* __restrict__ pos_tok,
                                                          const int* __restrict__ offsets, int E, int R, int d,
                                                          __half* __restrict__ xs) {
  pdl_wait();
  pdl_launch_dependents();
  const int n = min(__ldcg(offsets + E), R);
  const int lane = threadIdx.x & 31;
  const int w0 = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  const int q = d / 8;  // 16-byte pieces per row
  for (int i = w0; i < n; i += nw) {
    const int pos = n - 1 - i;
    const int t = __ldcg(pos_tok + pos);
    const uint4* src = reinterpret_cast<const uint4*>(x16 + static_cast<size_t>(t) * d);
    uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(pos) * d);
    for (int j0 = 0; j0 < q; j0 += 32 * 4) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 32 * u + lane;
        if (j < q) v[u] = src[j];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + 32 * u + lane;
        if (j < q) dst[j] = v[u];
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    expert_wide_kernel(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                       const __grid_constant__ WideActMaps am, const __grid_constant__ ExpertArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(smem_addr(&sm.full_a[i]), 33);  // 32 cp.async arrivals + 1 expect_tx arrival
      mbar_init(smem_addr(&sm.empty_a[i]), 4);  // the four dequantisation warps
    }
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(smem_addr(&sm.full_b[i]), 1);  // expect_tx arrival of the activation producer
      mbar_init(smem_addr(&sm.empty_b[i]), 1);  // MMA commit
    }
    for (int i = 0; i < kNumA; ++i) {
      mbar_init(smem_addr(&sm.a_full[i]), 4);
      mbar_init(smem_addr(&sm.a_empty[i]), 1);
    }
    for (int i = 0; i < kNumD; ++i) {
      mbar_init(smem_addr(&sm.d_full[i]), 1);
      mbar_init(smem_addr(&sm.d_empty[i]), kEpiWarps);
    }
    for (int i = 0; i < kTaskSlots; ++i) {
      mbar_init(smem_addr(&sm.task_full[i]), 1);
      mbar_init(smem_addr(&sm.task_empty[i]), kTaskConsumers);
    }
    mbar_init(smem_addr(&sm.drain), 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpFetch && lane == 0) {
    prefetch_tmap(&tm_w13);
    prefetch_tmap(&tm_w2);
  }
  if (warp == kWarpAct0 && lane < 2 * kBoxMaps) prefetch_tmap(lane < kBoxMaps ? &am.xs[lane] : &am.h[lane - kBoxMaps]);
  // everything above is local to the CTA; the task table and the counters come from the
  // preceding kernels
  pdl_wait();
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t ringa0 = smem_addr(&sm.ring_a[0][0]);
  const uint32_t ringb0 = smem_addr(&sm.ring_b[0][0]);

  if (warp == kWarpFetch) {
    // ------------- task fetcher + weight producer: TMA code tiles, cp.async scales -------------
    // The ticket of task i+2 is taken when task i starts and its entry loaded when task i
    // ends, so neither latency stalls the copies.
    const uint64_t pol = policy_evict_first();
    const int ntot = __ldcg(a.meta + META_WGU) + __ldcg(a.meta + META_WDN);
    const TaskEntry kEnd = TaskEntry{-1, 0, 0, 0};
    int stage = 0, issued = 0, n = 0;
    uint32_t phase = 0;
    int cur = blockIdx.x, nxt = ntot;
    TaskEntry entry = kEnd, entry_nxt = kEnd;
    if (lane == 0 && cur < ntot) {
      entry = a.tasks[cur];
      nxt = static_cast<int>(atomicAdd(a.ticket, 1u)) + static_cast<int>(gridDim.x);
      if (nxt < ntot) entry_nxt = a.tasks[nxt];
    }
    bool ok = true;
    while (ok) {
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
      const int rA0 = is_dn ? (e - a.e_lo) * a.d + s * kDnRows : (e - a.e_lo) * 2 * a.F + s * kGuRows;
      const int rA1 = is_dn ? rA0 + 64 : rA0 + a.F;
      const int sstride = is_dn ? a.F / 16 : a.d / 16;
      const CUtensorMap* tm = is_dn ? &tm_w2 : &tm_w13;
      const uint8_t* sbase = is_dn ? a.w2_scales : a.w13_scales;
      const int nck = is_dn ? a.nck_dn : a.nck_gu;
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
          cp_async_8(sb + kStageCodes + i * 8, sbase + static_cast<size_t>(grow) * sstride + kb / 16);
        }
        cp_async_arrive_noinc(fa);
        ++issued;
        if (++stage == kStagesA) { stage = 0; phase ^= 1u; }
      }
      if (lane == 0) {
        cur = nxt;
        entry = entry_nxt;
        nxt = nxt2;
        entry_nxt = nxt < ntot ? a.tasks[nxt] : kEnd;
      }
    }
    cp_async_wait_all();
    // drain: the last phase issued on every stage has landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int i = 0; i < min(issued, kStagesA); ++i) {
        if (--st < 0) { st = kStagesA - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_a[st]), ph) && clock64() - t0 < kDrainCycles) {}
      }
    }
  } else if (warp == kWarpAct0) {
    // ------------- activation producer: the pass's routed rows by TMA -------------
    // Lanes 0 and 1 load atoms 0 and 1 of a chunk (64 K elements each), one box of the
    // smallest height (64, 128 or 192 rows) that covers the pass.  Rows past the pass (other
    // passes' rows, or zeros past the tensor) feed accumulator columns the epilogue never reads.
    int stage = 0, n = 0, issued = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      if (tk.is_dn) {
        // every gate/up stripe of this expert (all passes) has published its h rows
        const int npass = (__ldg(a.counts + tk.e) + kWideRows - 1) / kWideRows;
        const uint32_t target = static_cast<uint32_t>(npass * a.S_gu);
        if (!warp_wait_counter(a.ready + tk.u, target, &sm.abort_flag, a.status, a.wait_limit)) break;
      }
      const int nbox = (tk.rows + kBoxRows - 1) / kBoxRows;
      const CUtensorMap* tm = tk.is_dn ? &am.h[nbox - 1] : &am.xs[nbox - 1];
      const uint32_t bytes = static_cast<uint32_t>(nbox * 2 * kBoxRows * 128);
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.empty_b[stage]), phase ^ 1u, sm, a.status, a.wait_limit)) { ok = false; break; }
        const uint32_t fb = smem_addr(&sm.full_b[stage]);
        if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
        __syncwarp();
        if (lane < 2) tma_load_2d_plain(ringb0 + stage * kStageB + lane * kAtomB, tm, c * kChunkK + 64 * lane, tk.row0, fb);
        ++issued;
        if (++stage == kStagesB) { stage = 0; phase ^= 1u; }
      }
    }
    // drain: the last phase issued on every stage has landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int i = 0; i < min(issued, kStagesB); ++i) {
        if (--st < 0) { st = kStagesB - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_b[st]), ph) && clock64() - t0 < kDrainCycles) {}
      }
    }
    __syncwarp();
  } else if (warp >= kWarpDeq0 && warp < kWarpDeq0 + 4) {
    // ---------------- dequantisation: NVFP4 -> FP16 A tile in tensor memory ----------------
    const int i = tid - 32 * kWarpDeq0;  // A row of this thread (= tensor-memory lane)
    const int half = i >> 6, r = i & 63;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int stage = 0, abuf = 0, n = 0;
    uint32_t phase = 0, aphase = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.full_a[stage]), phase, sm, a.status, a.wait_limit)) { ok = false; break; }
        const uint8_t* st = &sm.ring_a[stage][0];
        const uint8_t* crow = st + half * (kStageCodes / 2) + r * 64;
        uint4 q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) q[j] = *reinterpret_cast<const uint4*>(crow + ((j ^ ((r >> 1) & 3)) << 4));
        const uint2 sc = *reinterpret_cast<const uint2*>(st + kStageCodes + i * 8);
        uint32_t v[64];
        const uint32_t sp[4] = {e4m3x2_to_f16x2(sc.x), e4m3x2_to_f16x2(sc.x >> 16), e4m3x2_to_f16x2(sc.y),
                                e4m3x2_to_f16x2(sc.y >> 16)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int wi = 4 * j + h;  // word of the row chunk (8 elements)
            const int blk = wi >> 1;   // 16-element scale block
            const uint32_t sraw = (blk & 1) ? bcast_hi_half(sp[blk >> 1]) : bcast_lo_half(sp[blk >> 1]);
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
        tc_fence_after();
        tmem_st_x64(tmem + lane_base + abuf * 64, v);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.a_full[abuf]));
        if (++stage == kStagesA) { stage = 0; phase ^= 1u; }
        if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer: the warp waits, one elected lane issues ----------------
    // Descriptors and tensor-memory addresses are computed by the whole warp in converged
    // code; only the tcgen05 instructions run on the elected lane.  Both operands are written
    // by the async proxy (TMA; tcgen05.st ordered by the tensor-core fences and barriers), so
    // no proxy fence precedes the MMAs.
    int stage = 0, abuf = 0, dbuf = 0, n = 0;
    uint32_t phase = 0, aphase = 0, dphase = 0;
    bool ok = true;
    const uint64_t bdesc0 = smem_desc_sw128(ringb0, 1024);
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      const uint32_t idesc = idesc_f16_f32(128, mma_n(tk.rows));
      if (!warp_wait(smem_addr(&sm.d_empty[dbuf]), dphase ^ 1u, sm, a.status, a.wait_limit)) break;
      tc_fence_after();
      const uint32_t dcol = tmem + kDCol0 + dbuf * kWideRows;
      for (int c = 0; c < tk.nck; ++c) {
        if (!warp_wait(smem_addr(&sm.a_full[abuf]), aphase, sm, a.status, a.wait_limit)) { ok = false; break; }
        if (!warp_wait(smem_addr(&sm.full_b[stage]), phase, sm, a.status, a.wait_limit)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bd = bdesc0 + static_cast<uint64_t>((stage * kStageB) >> 4);
        const uint32_t acol = tmem + abuf * 64;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            tc_mma_f16_ts(dcol, acol + kk * 8, bd + static_cast<uint64_t>(((kk >> 2) * kAtomB + (kk & 3) * 32) >> 4),
                          idesc, (c > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_addr(&sm.empty_b[stage]));
          tc_commit(smem_addr(&sm.a_empty[abuf]));
        }
        __syncwarp();
        if (++stage == kStagesB) { stage = 0; phase ^= 1u; }
        if (++abuf == kNumA) { abuf = 0; aphase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(smem_addr(&sm.d_full[dbuf]));
      __syncwarp();
      if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }
    }
    if (lane == 0) {
      // every issued MMA completes before tensor memory is released
      tc_commit(smem_addr(&sm.drain));
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_addr(&sm.drain), 0) && clock64() - t0 < kDrainCycles) {}
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 0-7): thread t owns accumulator lane t % 128 ----------------
    const int i = tid & 127;   // accumulator lane
    const int grp = tid >> 7;  // slices 2k + grp of 32 columns
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* xch = sm.xch[grp];
    int dbuf = 0, n = 0;
    uint32_t dphase = 0;
    while (true) {
      TaskEntry te;
      const bool got_task = take_task(sm, n++, te, a.status, a.wait_limit);
      if (!named_bar_and(2, 32 * kEpiWarps, got_task)) break;
      const Task tk = unpack(te, a);
      if (!tk.valid) break;
      const bool got = warp_wait(smem_addr(&sm.d_full[dbuf]), dphase, sm, a.status, a.wait_limit);
      if (!named_bar_and(2, 32 * kEpiWarps, got)) break;
      tc_fence_after();
      const uint32_t dcol = tmem + lane_base + kDCol0 + dbuf * kWideRows;
      const float sc13 = ts13_of(a, tk.e), sc2 = ts2_of(a, tk.e) * kHUnscale;
      for (int c0 = 32 * grp; c0 < tk.rows; c0 += 64) {
        uint32_t v[32];
        tmem_ld_x32(dcol + c0, v);
        tc_wait_ld();
        if (!tk.is_dn) {
          // Lanes n < 64 hold the gate row of F index n, lanes n + 64 the up row.  Lane n
          // forms h for columns 0-15 of the slice, lane n + 64 for columns 16-31: the up
          // values of columns 0-15 and the gate values of columns 16-31 cross over.
          const int nF = i & 63;
          const bool up = i >= 64;
#pragma unroll
          for (int j = 0; j < 16; ++j) xch[(up ? j : 16 + j) * 64 + nF] = __uint_as_float(up ? v[j] : v[16 + j]);
          named_bar_sync(4 + grp, 128);
          uint32_t* hst = sm.hstage[grp];
          const int j0 = up ? 16 : 0;
          // branch-free, so that the independent SiLU chains interleave; the largest magnitude
          // of the valid columns decides the one status update.  Word (r / 2) * 64 + nF holds
          // rows r (low half) and r + 1 (high half) of column nF.
          const int nv = tk.rows - c0 - j0;  // valid columns among this thread's 16
          float hv[16];
          float mx = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float own = __uint_as_float(up ? v[16 + j] : v[j]) * sc13;
            const float other = xch[(j0 + j) * 64 + nF] * sc13;
            const float g = up ? other : own, u = up ? own : other;
            const float h = __fdividef(g, 1.0f + __expf(-g)) * u * kHScale;
            mx = j < nv ? fmaxf(mx, fabsf(h)) : mx;
            hv[j] = j < nv ? h : 0.f;
          }
#pragma unroll
          for (int j = 0; j < 16; j += 2) hst[((j0 + j) >> 1) * 64 + nF] = f16x2_satfinite(hv[j], hv[j + 1]);
          if (mx > 65504.f) atomicOr(a.status, static_cast<int>(MOE_DEV_H_SATURATED));
          named_bar_sync(4 + grp, 128);
          // rows 2p and 2p + 1, 8 F values each, from 8 words: one thread per (p, piece)
          {
            const int pp = i >> 3, part = i & 7;
            const uint4 w0 = *reinterpret_cast<const uint4*>(hst + pp * 64 + part * 8);
            const uint4 w1 = *reinterpret_cast<const uint4*>(hst + pp * 64 + part * 8 + 4);
            const uint4 lo = make_uint4(__byte_perm(w0.x, w0.y, 0x5410), __byte_perm(w0.z, w0.w, 0x5410),
                                        __byte_perm(w1.x, w1.y, 0x5410), __byte_perm(w1.z, w1.w, 0x5410));
            const uint4 hi = make_uint4(__byte_perm(w0.x, w0.y, 0x7632), __byte_perm(w0.z, w0.w, 0x7632),
                                        __byte_perm(w1.x, w1.y, 0x7632), __byte_perm(w1.z, w1.w, 0x7632));
            __half* hrow = a.hs16 + static_cast<size_t>(tk.row0 + c0 + 2 * pp) * a.F + tk.s * kGuRows + part * 8;
            if (c0 + 2 * pp < tk.rows) *reinterpret_cast<uint4*>(hrow) = lo;
            if (c0 + 2 * pp + 1 < tk.rows) *reinterpret_cast<uint4*>(hrow + a.F) = hi;
          }
        } else {
          // per-route outputs as FP16(y * 2^-4), staged so that each routed row's 128 values
          // leave in 16-byte pieces; word (r / 2) * 128 + i holds rows r and r + 1 of d-row i
          uint32_t* yst = reinterpret_cast<uint32_t*>(xch);
          const float ys = sc2 * kYScale;
          const int nv = tk.rows - c0;  // valid columns of the slice
          float mx = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float y0 = __uint_as_float(v[j]) * ys, y1 = __uint_as_float(v[j + 1]) * ys;
            mx = j < nv ? fmaxf(mx, fabsf(y0)) : mx;
            mx = j + 1 < nv ? fmaxf(mx, fabsf(y1)) : mx;
            yst[(j >> 1) * kDnRows + i] = f16x2_satfinite(y0, y1);
          }
          if (mx > 65504.f) atomicOr(a.status, static_cast<int>(MOE_DEV_Y_SATURATED));
          named_bar_sync(4 + grp, 128);
          __half* y16 = reinterpret_cast<__half*>(a.y);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int q = i + 128 * t, pp = q >> 4, part = q & 15;
            const uint4 w0 = *reinterpret_cast<const uint4*>(yst + pp * kDnRows + part * 8);
            const uint4 w1 = *reinterpret_cast<const uint4*>(yst + pp * kDnRows + part * 8 + 4);
            const uint4 lo = make_uint4(__byte_perm(w0.x, w0.y, 0x5410), __byte_perm(w0.z, w0.w, 0x5410),
                                        __byte_perm(w1.x, w1.y, 0x5410), __byte_perm(w1.z, w1.w, 0x5410));
            const uint4 hi = make_uint4(__byte_perm(w0.x, w0.y, 0x7632), __byte_perm(w0.z, w0.w, 0x7632),
                                        __byte_perm(w1.x, w1.y, 0x7632), __byte_perm(w1.z, w1.w, 0x7632));
            __half* yrow = y16 + static_cast<size_t>(tk.row0 + c0 + 2 * pp) * a.d + tk.s * kDnRows + part * 8;
            if (c0 + 2 * pp < tk.rows) *reinterpret_cast<uint4*>(yrow) = lo;
            if (c0 + 2 * pp + 1 < tk.rows) *reinterpret_cast<uint4*>(yrow + a.d) = hi;
          }
          named_bar_sync(4 + grp, 128);
        }
      }
      // the accumulator is read: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sm.d_empty[dbuf]));
      if (++dbuf == kNumD) { dbuf = 0; dphase ^= 1u; }
      if (!tk.is_dn) {
        // publish this stripe's h rows (release) for the down tasks of the expert
        __threadfence();
        named_bar_sync(3, 32 * kEpiWarps);
        if (tid == 0) atom_add_acqrel_u32(a.ready + tk.u, 1u);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per CTA (227 KB)");

size_t expert_wide_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_wide_gather(const ExpertArgs& a, __half* xs, int num_sms, cudaStream_t stream) {
  return launch_pdl(wide_gather_kernel, dim3(num_sms * 8), dim3(256), 0, stream, a.x16, a.pos_tok, a.offsets, a.E, a.R,
                    a.d, xs);
}

cudaError_t launch_expert_wide(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                               const WideActMaps& am, int num_sms, cudaStream_t stream) {
  const size_t smem = expert_wide_smem_bytes();
  cudaError_t err = cudaFuncSetAttribute(expert_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(expert_wide_kernel, dim3(num_sms), dim3(kThreads), smem, stream, tm_w13, tm_w2, am, a);
}

cudaError_t launch_wide_plan(const ExpertArgs& a, TaskEntry* tasks_w, cudaStream_t stream) {
  return launch_pdl(wide_plan_kernel, dim3(16), dim3(1024), 0, stream, a.meta, const_cast<int*>(a.meta), a.touched,
                    a.counts, a.offsets, tasks_w, a.S_gu, a.S_dn);
}

}  // namespace moe
