// Decode-shaped expert kernel: weight-stationary GEMV on the warp-level tensor-core MMA.
//
// For the few routed rows of a verify step (1-64 per expert) a tcgen05 MMA is bound by
// its fixed per-instruction time (~94 ns whatever N <= 128, measured on GB300), so a
// 128x16 FP16 A tile per instruction cannot keep up with the weight stream.  Here the
// dequantised weights stay in registers as the 16-row A fragment of mma.sync m16n8k16 and
// the routed rows are its 8-column B operand: one weight fragment serves every row (the
// multi-row weight-stationary GEMV described in the b12x tensor-core GEMV notes of the
// pages).
//
// Structure (one resident CTA per SM, tasks from the plan's task table via tickets):
//   warp 0      task fetcher + weight producer: per 256-K chunk two TMA tiles of E2M1 codes
//               (64 rows x 128 B each, 128-byte swizzle) and two of the chunk's block scales
//               (64 rows x 16 B) into one stage of a ring, so short tasks never starve it;
//   warp 1      activation producer: per chunk and 8-row tile, one bulk copy per routed row
//               (512 B of FP16 hidden for gate/up, of h for down) into a padded tile;
//   warp 2      publisher: after the compute warps have written a gate/up task's h rows it
//               releases them to other CTAs (one fence and one reduction per task), so the
//               compute warps never wait on the fence; with the un-route fused it releases
//               each down task's y rows the same way, counted per 128-column stripe;
//   warps 3-10  compute: each owns 16 weight rows of the 128-row tile.  Gate/up tasks give
//               warp w gate rows of one 8-row group as fragment rows 0-7 and the up rows of
//               the same F indices as fragment rows 8-15, so h = silu(g) * u is formed in
//               registers.  With the un-route fused (few tokens), trailing un-route tasks
//               give each compute warp one token's 128 columns of one stripe, once every
//               down task of that stripe has been released.
// Fragment row g holds tile row 8w + frag_row(g): the permutation puts the two rows that
// one 8-lane shared-memory phase reads on different halves of the 128-byte swizzle, so the
// code reads are free of bank conflicts (the scale reads, 8 rows x 16 B, are too).
// Each thread dequantises 2 rows x 64 elements per chunk (exact FP16: E2M1 x E4M3 has at
// most 6 significant bits), feeds 16 MMAs per 8-row tile with FP32 accumulation, and
// writes h (FP16) or per-route down outputs (FP32) at the end of the task.  Only the TMA
// and bulk-copy engines write shared memory, so the consumers need no proxy fences.
#include "mma_parts.cuh"

namespace moe {

namespace mk {

constexpr int kStagesA = 9;
constexpr int kStagesB = 12;
constexpr int kTileRows = 8;
constexpr int kRowPitchB = 2 * kChunk + 16;     // padded FP16 row of one chunk (528 B)
constexpr int kStageB = kTileRows * kRowPitchB;  // 4224
constexpr int kMaxTiles = kRowsPerPass / kTileRows;  // 8
constexpr int kTaskConsumers = 2 + kComputeWarps;  // activation producer, publisher, compute
// Compute warps run at most kTaskSlots tasks ahead of the publisher (it frees each task
// slot before waiting on that task), so twice as many publication slots never wrap early.
constexpr int kPubSlots = 2 * kTaskSlots;
// The producer claims its next task (ticket) only once at most kReserve of its chunks are
// in flight: late enough that the last tasks go to whichever CTA frees up first, early
// enough that the ticket and table round trips are hidden behind the chunks still queued.
constexpr int kReserve = 4;

struct Smem {
  uint8_t ring_a[kStagesA][kStageA];
  uint8_t ring_b[kStagesB][kStageB];
  TaskEntry task[kTaskSlots];
  uint64_t full_a[kStagesA];
  uint64_t empty_a[kStagesA];
  uint64_t empty_b[kStagesB];
  uint64_t task_full[kTaskSlots];
  uint64_t task_empty[kTaskSlots];
  uint64_t pub_full[kPubSlots];
  int abort_flag;
};

__device__ __forceinline__ bool take_task(Smem& sm, int n, TaskEntry& out, int* status, long long limit) {
  const int q = n % kTaskSlots;
  const uint32_t ph = static_cast<uint32_t>((n / kTaskSlots) & 1);
  if (!warp_wait(smem_addr(&sm.task_full[q]), ph, &sm.abort_flag, status, limit)) return false;
  out = sm.task[q];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&sm.task_empty[q]));
  return true;
}

// B fragments of one 8-row activation tile for sub-chunk h: tile row g, elements
// [128h + 32q, +32) as four 16-byte pieces (piece j feeds k-steps (h, j, 0) and (h, j, 1)).
// Rows past the task's routed rows were not copied and enter as zeros.
__device__ __forceinline__ void load_b_frag(const uint8_t* tile, int g, int q, int h, bool live, uint4 (&x)[4]) {
  const uint8_t* row = tile + g * kRowPitchB + 64 * q + 256 * h;
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = live ? *reinterpret_cast<const uint4*>(row + 16 * j) : make_uint4(0, 0, 0, 0);
}

// Per-warp pipeline position of the compute warps.
struct ComputeState {
  int stage_a, stage_b;
  uint32_t phase_a;
};

// The chunk loop of one task for one compute warp, one instantiation per accumulation
// layout so that a task runs one tight loop.  acc receives, per 8-row tile t, the FP32
// partial products of fragment rows g / g + 8 with the task's routed rows.
//   MODE 1 (one tile):  the 16 k-steps of a chunk go to 8 independent accumulators;
//   MODE 2 (two tiles): 4 accumulators per tile;
//   MODE 0 (otherwise, and every pass of a multi-pass expert): one accumulator per tile,
//                       tiles in pairs (the second of an odd last pair multiplies zeros
//                       into an accumulator that is never stored).
// The independent sets are summed (fixed order) before returning.  Returns false when a
// bounded wait gave up.
template <int MODE>
__device__ __forceinline__ bool run_chunks(Smem& sm, const ExpertArgs& a, ComputeState& cs, float (&acc)[kMaxTiles][4],
                                           int lra, int lrb, int nck, int nt, int rows, int g, int q) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kMaxTiles; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  // codes and scales of chunk c are loaded into registers during chunk c - 1, so their
  // shared-memory latency overlaps the previous chunk's MMAs.  A chunk's stage is full only
  // once its activation tiles have landed too; if two chunks' tiles do not fit in the tile
  // ring together, they land only after this chunk releases its tiles, so the next chunk is
  // then loaded after the release.
  const bool early = MODE != 0 || 2 * nt <= kStagesB;
  ChunkCodes next;
  if (!warp_wait(smem_addr(&sm.full_a[cs.stage_a]), cs.phase_a, &sm.abort_flag, a.status, a.wait_limit)) return false;
  load_chunk_codes(&sm.ring_a[cs.stage_a][0], lra, lrb, q, next);
  for (int c = 0; c < nck; ++c) {
    const ChunkCodes cur = next;
    // the stage's bytes are in registers: hand it back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&sm.empty_a[cs.stage_a]));
    if (++cs.stage_a == kStagesA) { cs.stage_a = 0; cs.phase_a ^= 1u; }
    if (early && c + 1 < nck) {
      if (!warp_wait(smem_addr(&sm.full_a[cs.stage_a]), cs.phase_a, &sm.abort_flag, a.status, a.wait_limit)) return false;
      load_chunk_codes(&sm.ring_a[cs.stage_a][0], lra, lrb, q, next);
    }
    // Per sub-chunk h: activation fragments first (their latency overlaps the
    // dequantisation), then the 32 weights per row of this thread, then the MMAs.
    // MMA k-step (h, j, x): A registers 4j + 2x, 4j + 2x + 1, B word pair x of piece j.
    const uint8_t* b0 = &sm.ring_b[cs.stage_b][0];
    if constexpr (MODE == 1) {
      const bool live = g < rows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 xb[4];
        load_b_frag(b0, g, q, h, live, xb);
        uint32_t fa[16], fb[16];
        dequant32(cur.ca[h], cur.sa[h], fa);
        dequant32(cur.cb[h], cur.sb[h], fb);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mma_16816(acc[2 * j], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], xb[j].x, xb[j].y);
          mma_16816(acc[2 * j + 1], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], xb[j].z, xb[j].w);
        }
      }
    } else if constexpr (MODE == 2) {
      const uint8_t* b1 = &sm.ring_b[cs.stage_b + 1 == kStagesB ? 0 : cs.stage_b + 1][0];
      const bool live0 = g < rows, live1 = g < rows - kTileRows;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 x0[4], x1[4];
        load_b_frag(b0, g, q, h, live0, x0);
        load_b_frag(b1, g, q, h, live1, x1);
        uint32_t fa[16], fb[16];
        dequant32(cur.ca[h], cur.sa[h], fa);
        dequant32(cur.cb[h], cur.sb[h], fb);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = (2 * j) & 3;
          mma_16816(acc[ch], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], x0[j].x, x0[j].y);
          mma_16816(acc[4 + ch], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], x1[j].x, x1[j].y);
          mma_16816(acc[ch + 1], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], x0[j].z, x0[j].w);
          mma_16816(acc[5 + ch], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], x1[j].z, x1[j].w);
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t fa[16], fb[16];
        dequant32(cur.ca[h], cur.sa[h], fa);
        dequant32(cur.cb[h], cur.sb[h], fb);
#pragma unroll
        for (int tp = 0; tp < kMaxTiles / 2; ++tp) {
          if (2 * tp < nt) {
            const int t0 = 2 * tp, t1 = 2 * tp + 1;
            const uint8_t* s0 = &sm.ring_b[(cs.stage_b + t0) % kStagesB][0];
            const uint8_t* s1 = &sm.ring_b[(cs.stage_b + t1) % kStagesB][0];
            const bool live0 = g < rows - t0 * kTileRows;
            const bool live1 = t1 < nt && g < rows - t1 * kTileRows;
            uint4 x0[4], x1[4];
            load_b_frag(s0, g, q, h, live0, x0);
            load_b_frag(s1, g, q, h, live1, x1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              mma_16816(acc[t0], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], x0[j].x, x0[j].y);
              mma_16816(acc[t1], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], x1[j].x, x1[j].y);
              mma_16816(acc[t0], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], x0[j].z, x0[j].w);
              mma_16816(acc[t1], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], x1[j].z, x1[j].w);
            }
          }
        }
      }
    }
    // the chunk's activation tiles are consumed
    __syncwarp();
    if (lane == 0) {
      int sbt = cs.stage_b;
      for (int t = 0; t < nt; ++t) {
        mbar_arrive(smem_addr(&sm.empty_b[sbt]));
        if (++sbt == kStagesB) sbt = 0;
      }
    }
    cs.stage_b += nt;
    if (cs.stage_b >= kStagesB) cs.stage_b -= kStagesB;
    if (!early && c + 1 < nck) {
      if (!warp_wait(smem_addr(&sm.full_a[cs.stage_a]), cs.phase_a, &sm.abort_flag, a.status, a.wait_limit)) return false;
      load_chunk_codes(&sm.ring_a[cs.stage_a][0], lra, lrb, q, next);
    }
  }
  // fold the independent accumulator sets into one per tile
  if constexpr (MODE == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      acc[0][i] = ((acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i])) + ((acc[4][i] + acc[5][i]) + (acc[6][i] + acc[7][i]));
  } else if constexpr (MODE == 2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[0][i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
      acc[1][i] = (acc[4][i] + acc[5][i]) + (acc[6][i] + acc[7][i]);
    }
  }
  return true;
}

}  // namespace mk

using namespace mk;

// kFused: the kernel also runs the un-route, as a.ncb tasks after every expert task (each
// waits for the down tasks of its stripe); otherwise the un-route is a kernel of its own and
// none of that code is compiled in.
template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    expert_mma_kernel(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                      const __grid_constant__ CUtensorMap tm_s13, const __grid_constant__ CUtensorMap tm_s2,
                      const __grid_constant__ ExpertArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    // a chunk's stage is full once both producers have arrived and all its bytes (codes
    // and activation tiles) have landed
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(smem_addr(&sm.full_a[i]), 2);
      mbar_init(smem_addr(&sm.empty_a[i]), kComputeWarps);
    }
    for (int i = 0; i < kStagesB; ++i) mbar_init(smem_addr(&sm.empty_b[i]), kComputeWarps);
    for (int i = 0; i < kTaskSlots; ++i) {
      mbar_init(smem_addr(&sm.task_full[i]), 1);
      mbar_init(smem_addr(&sm.task_empty[i]), kTaskConsumers);
    }
    for (int i = 0; i < kPubSlots; ++i) mbar_init(smem_addr(&sm.pub_full[i]), kComputeWarps);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w13);
    prefetch_tmap(&tm_w2);
    prefetch_tmap(&tm_s13);
    prefetch_tmap(&tm_s2);
  }
  // everything above is local to the CTA; the plan and the counters come from the
  // preceding kernel
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  const uint32_t ringa0 = smem_addr(&sm.ring_a[0][0]);
  const uint32_t ringb0 = smem_addr(&sm.ring_b[0][0]);
  int tcnt = 0;
  if (tid == 0) trace_ev(a, 5, tcnt, 10, 0);

  if (warp == 0) {
    // ------------- task fetcher + weight producer (next ticket taken late: kReserve) -------------
    const uint64_t pol = policy_evict_first();
    const int ntask = __ldg(a.meta + META_NGU) + __ldg(a.meta + META_NDN);
    const int ntot = ntask + (kFused ? a.ncb : 0);
    const TaskEntry kEnd = TaskEntry{-1, 0, 0, 0};
    int stage = 0, issued = 0, n = 0, chunk_seq = 0;
    uint32_t phase = 0;
    int cur = blockIdx.x;
    TaskEntry entry = kEnd;
    if (lane == 0) {
      // the first entry is loaded alongside the task counts (the table has room for it)
      const TaskEntry raw = a.tasks[min(cur, a.task_cap - 1)];
      entry = cur < ntask ? raw : (cur < ntot ? task_at(a, cur, ntask) : kEnd);
    }
    bool ok = true;
    while (ok) {
      const int q = n % kTaskSlots;
      if (!warp_wait(smem_addr(&sm.task_empty[q]), static_cast<uint32_t>(((n / kTaskSlots) & 1) ^ 1), &sm.abort_flag,
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
      if (!live) break;
      const int x = __shfl_sync(0xffffffffu, entry.x, 0);
      const int z = __shfl_sync(0xffffffffu, entry.z, 0);
      const int s = __shfl_sync(0xffffffffu, entry.w, 0);
      const int e = x & 0xffff;
      const bool is_dn = ((z >> 16) & 1) != 0;
      int rA0, rA1, nck;
      const CUtensorMap* tm;
      if (!is_dn) {
        rA0 = (e - a.e_lo) * 2 * a.F + s * kGuRows;
        rA1 = rA0 + a.F;
        tm = &tm_w13;
        nck = a.d / kChunk;
      } else {
        rA0 = (e - a.e_lo) * a.d + s * kDnRows;
        rA1 = rA0 + 64;
        tm = &tm_w2;
        nck = a.F / kChunk;
      }
      if (kFused && ((z >> 18) & 1)) nck = 0;  // un-route task: no weights
      const CUtensorMap* tms = is_dn ? &tm_s2 : &tm_s13;
      ++n;
      for (int c = 0; c < nck; ++c) {
        if (!warp_wait(smem_addr(&sm.empty_a[stage]), phase ^ 1u, &sm.abort_flag, a.status, a.wait_limit)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t sb = ringa0 + stage * kStageA;
          const uint32_t fa = smem_addr(&sm.full_a[stage]);
          mbar_arrive_expect_tx(fa, kStageA);
          tma_load_2d(sb, tm, c * (kChunk / 2), rA0, fa, pol);
          tma_load_2d(sb + kCodeBytes / 2, tm, c * (kChunk / 2), rA1, fa, pol);
          // the chunk's 16 block scales of each row (16 bytes at column 16c)
          tma_load_2d(sb + kCodeBytes, tms, c * (kChunk / 16), rA0, fa, pol);
          tma_load_2d(sb + kCodeBytes + kScaleBytes / 2, tms, c * (kChunk / 16), rA1, fa, pol);
          trace_ev(a, 0, tcnt, 2, chunk_seq);
        }
        ++chunk_seq;
        ++issued;
        if (++stage == kStagesA) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      // take the next ticket once at most kReserve chunks are in flight, so that a task is
      // claimed shortly before this CTA can start it
      if (issued > kReserve) {
        const int sq = issued - 1 - kReserve + kStagesA;  // the issue that reuses that chunk's stage
        if (!warp_wait(smem_addr(&sm.empty_a[sq % kStagesA]), static_cast<uint32_t>(((sq / kStagesA) & 1) ^ 1),
                       &sm.abort_flag, a.status, a.wait_limit)) {
          ok = false;
          break;
        }
      }
      if (lane == 0) {
        cur = static_cast<int>(atomicAdd(a.ticket, 1u)) + static_cast<int>(gridDim.x);
        entry = cur < ntot ? (kFused ? task_at(a, cur, ntask) : a.tasks[cur]) : kEnd;
      }
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int i = 0; i < min(issued, kStagesA); ++i) {
        if (--st < 0) { st = kStagesA - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_a[st]), ph) && clock64() - t0 < kDrainCycles) {}
      }
    }
  } else if (warp == 1) {
    // ------------- activation producer: 8-row tiles, one bulk copy per routed row -------------
    // The copies complete on the weight stage's barrier of the same chunk (the chunk order
    // is the task order in both producers), so compute warps wait on one barrier per chunk.
    int stage = 0, n = 0, issued = 0, chunk_seq = 0, stage_a = 0;
    uint32_t phase = 0, phase_a = 0;
    bool ok = true;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if (kFused && is_unroute(te)) continue;
      const int e = te.x & 0xffff, u = (te.x >> 16) & 0xffff, row0 = te.y, rows = te.z & 0xffff;
      const bool is_dn = ((te.z >> 16) & 1) != 0;
      if (is_dn) {
        // every gate/up task of every stripe (all passes) of this expert must have published
        const int npass = (__ldg(a.counts + e) + kRowsPerPass - 1) / kRowsPerPass;
        const uint32_t target = static_cast<uint32_t>(npass * a.S_gu);
        const bool good = warp_wait_counter(a.ready + u, target, &sm.abort_flag, a.status, a.wait_limit);
        if (lane == 0) trace_ev(a, 1, tcnt, 3, n);
        if (!good) break;
      }
      const int nck = is_dn ? a.F / kChunk : a.d / kChunk;
      // lane l owns routed rows l and l + 32 of the pass
      const __half* src0;
      const __half* src1;
      if (is_dn) {
        src0 = a.hs16 + static_cast<size_t>(row0 + lane) * a.F;
        src1 = a.hs16 + static_cast<size_t>(row0 + lane + 32) * a.F;
      } else {
        const int t0 = lane < rows ? __ldg(a.pos_tok + row0 + lane) : 0;
        const int t1 = lane + 32 < rows ? __ldg(a.pos_tok + row0 + lane + 32) : 0;
        src0 = a.x16 + static_cast<size_t>(t0) * a.d;
        src1 = a.x16 + static_cast<size_t>(t1) * a.d;
      }
      const int nt = (rows + kTileRows - 1) / kTileRows;
      for (int c = 0; ok && c < nck; ++c) {
        // the chunk's weight stage must be free before this chunk's bytes are announced on it
        if (!warp_wait(smem_addr(&sm.empty_a[stage_a]), phase_a ^ 1u, &sm.abort_flag, a.status, a.wait_limit)) { ok = false; break; }
        const uint32_t fa = smem_addr(&sm.full_a[stage_a]);
        if (lane == 0) mbar_arrive_expect_tx(fa, static_cast<uint32_t>(rows) * (2 * kChunk));
        for (int t = 0; t < nt; ++t) {
          if (!warp_wait(smem_addr(&sm.empty_b[stage]), phase ^ 1u, &sm.abort_flag, a.status, a.wait_limit)) { ok = false; break; }
          const int trows = min(kTileRows, rows - t * kTileRows);
          // lanes 0..trows-1 copy their tile row: routed row r = 8t + lane
          const int r = t * kTileRows + lane;
          const __half* p0 = reinterpret_cast<const __half*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src0), r & 31));
          const __half* p1 = reinterpret_cast<const __half*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src1), r & 31));
          if (lane < trows) {
            const __half* src = (r < 32 ? p0 : p1) + c * kChunk;
            bulk_copy_g2s(ringb0 + stage * kStageB + lane * kRowPitchB, src, 2 * kChunk, fa);
          }
          ++issued;
          if (++stage == kStagesB) { stage = 0; phase ^= 1u; }
        }
        if (lane == 0) trace_ev(a, 1, tcnt, 4, chunk_seq);
        ++chunk_seq;
        if (++stage_a == kStagesA) { stage_a = 0; phase_a ^= 1u; }
      }
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      int st = stage_a;
      uint32_t ph = phase_a;
      for (int i = 0; i < min(chunk_seq, kStagesA); ++i) {
        if (--st < 0) { st = kStagesA - 1; ph ^= 1u; }
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_addr(&sm.full_a[st]), ph) && clock64() - t0 < kDrainCycles) {}
      }
    }
    (void)issued;
  } else if (warp == 2) {
    // ------------- publisher: release each finished gate/up task's h rows (fused: and each
    // finished down task's y rows, counted per stripe) -------------
    int n = 0, gu_n = 0;
    while (true) {
      TaskEntry te;
      if (!take_task(sm, n++, te, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if (kFused && is_unroute(te)) continue;
      const bool dn = ((te.z >> 16) & 1) != 0;
      if (dn && !kFused) continue;  // down task, un-route in its own kernel: nothing to publish
      uint32_t* ctr = dn ? a.dn_done + te.w : a.ready + ((te.x >> 16) & 0xffff);
      const int slot = gu_n % kPubSlots;
      const uint32_t ph = static_cast<uint32_t>((gu_n / kPubSlots) & 1);
      ++gu_n;
      // the compute warps' h stores are ordered before their arrivals (warp barrier, then a
      // release arrive); this acquire wait plus a GPU-scope fence makes the reduction below
      // release all of them
      if (!warp_wait(smem_addr(&sm.pub_full[slot]), ph, &sm.abort_flag, a.status, a.wait_limit)) break;
      if (lane == 0) {
        fence_acq_rel_gpu();
        red_add_relaxed_gpu_u32(ctr, 1u);
        trace_ev(a, 4, tcnt, 9, gu_n);
      }
      __syncwarp();
    }
  } else {
    // ------------- compute warps: dequantise into A fragments, mma.sync, epilogue -------------
    const int cw = warp - kFirstCompute;  // 0..7
    const int g = lane >> 2, q = lane & 3;
    const int fr = frag_row(g);
    ComputeState cs{0, 0, 0u};
    int n = 0, gu_n = 0;
    bool ok = true;
    // timeline (diagnostics only): the first and the last compute warp record task boundaries
    const bool tr = a.trace != nullptr && lane == 0 && (cw == 0 || cw == kComputeWarps - 1);
    const int trole = cw == 0 ? 2 : 3;
    while (ok) {
      TaskEntry te;
      if (!take_task(sm, n, te, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if constexpr (kFused) {
        if (is_unroute(te)) {
          ++n;
          const int t = min(te.y + cw, a.T - 1), c = te.w * kDnRows + 4 * lane;
          Unroute4Pre u;
          unroute4_pre(a, t, c, u);
          // every down task of the stripe (one per pass) has published its y columns
          const uint32_t dn_per_stripe = static_cast<uint32_t>(__ldg(a.meta + META_NDN) / a.S_dn);
          if (tr) trace_ev(a, trole, tcnt, 12, n);
          if (!warp_wait_counter(a.dn_done + te.w, dn_per_stripe, &sm.abort_flag, a.status, a.wait_limit)) break;
          if (tr) trace_ev(a, trole, tcnt, 13, n);
          if (te.y + cw < a.T) unroute4_post(a, t, c, u);
          continue;
        }
      }
      if (tr) trace_ev(a, trole, tcnt, 5, (((te.z >> 16) & 1) << 15) | (n & 0x7fff));
      const int row0 = te.y, rows = te.z & 0xffff, s = te.w;
      const bool is_dn = ((te.z >> 16) & 1) != 0;
      const int K = is_dn ? a.F : a.d;
      const int nck = K / kChunk;
      const int nt = (rows + kTileRows - 1) / kTileRows;
      // Accumulation layout: one- and two-tile passes spread their k-steps over independent
      // accumulator sets; an expert with several passes keeps one set per tile in every pass,
      // so a route's result does not depend on which pass the plan put it in.
      const bool multi = ((te.z >> 17) & 1) != 0;
      const int mode = multi ? 0 : (nt == 1 ? 1 : (nt == 2 ? 2 : 0));
      // tile rows (0..127) of fragment rows g and g + 8
      const int lra = is_dn ? 16 * cw + fr : 8 * cw + fr;
      const int lrb = is_dn ? 16 * cw + 8 + fr : 64 + 8 * cw + fr;
      float acc[kMaxTiles][4];
      if (mode == 1) ok = run_chunks<1>(sm, a, cs, acc, lra, lrb, nck, nt, rows, g, q);
      else if (mode == 2) ok = run_chunks<2>(sm, a, cs, acc, lra, lrb, nck, nt, rows, g, q);
      else ok = run_chunks<0>(sm, a, cs, acc, lra, lrb, nck, nt, rows, g, q);
      if (!ok) break;
      if (tr) trace_ev(a, trole, tcnt, 6, n);
      ++n;
      // ---- epilogue: fragment rows g / g+8, routed rows 8t + 2q, 8t + 2q + 1 ----
      if (!is_dn) {
        const int nidx = s * kGuRows + 8 * cw + fr;  // element n of h
        const float sc = ts13_of(a, te.x & 0xffff);
#pragma unroll
        for (int t = 0; t < kMaxTiles; ++t) {
          if (t < nt) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int r = t * kTileRows + 2 * q + cc;
              if (r < rows)
                a.hs16[static_cast<size_t>(row0 + r) * a.F + nidx] =
                    h_store_value(silu_mul(acc[t][cc] * sc, acc[t][2 + cc] * sc), a.status);
            }
          }
        }
        // hand the task to the publisher
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.pub_full[gu_n % kPubSlots]));
        ++gu_n;
      } else {
        const float sc = ts2_of(a, te.x & 0xffff) * kHUnscale;
        const int ra = s * kDnRows + lra, rb = s * kDnRows + lrb;
#pragma unroll
        for (int t = 0; t < kMaxTiles; ++t) {
          if (t < nt) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int r = t * kTileRows + 2 * q + cc;
              if (r < rows) {
                float* yrow = a.y + static_cast<size_t>(row0 + r) * a.d;
                yrow[ra] = acc[t][cc] * sc;
                yrow[rb] = acc[t][2 + cc] * sc;
              }
            }
          }
        }
        if constexpr (kFused) {
          // hand the task to the publisher: the un-route waits for its stripe
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.pub_full[gu_n % kPubSlots]));
          ++gu_n;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    int c2 = 1;
    trace_ev(a, 5, c2, 11, 0);
  }
}

size_t expert_mma_smem_bytes() { return sizeof(Smem) + 1024; }

// The un-route runs inside the kernel for at most this many tokens (measured: for more, the
// separate un-route kernel after the expert kernel is faster).
constexpr int kFuseMaxTokens = 8;

int expert_mma_unroute_tasks(int T, int S_dn) {
  return T <= kFuseMaxTokens ? S_dn * ((T + kComputeWarps - 1) / kComputeWarps) : 0;
}

bool expert_mma_supports(int d, int F) {
  const auto pow2_in_range = [](int v) { return v >= kChunk && v <= 2048 && (v & (v - 1)) == 0; };
  return pow2_in_range(d) && pow2_in_range(F);
}

cudaError_t launch_expert_mma(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_s13, const CUtensorMap& tm_s2, int num_sms,
                              cudaStream_t stream) {
  const size_t smem = expert_mma_smem_bytes();
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const ExpertArgs) =
      a.ncb > 0 ? expert_mma_kernel<true> : expert_mma_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, stream, tm_w13, tm_w2, tm_s13, tm_s2, a);
}

}  // namespace moe
