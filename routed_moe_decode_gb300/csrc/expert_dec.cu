// Decode expert kernel: every task is one expert pass of at most eight routed rows, so one
// 8-column MMA tile.
//
// Same weight stream and MMA core as the warp-MMA kernel of expert_mma.cu (one resident CTA
// per SM, tasks through tickets, 256-K chunks of E2M1 codes and block scales by TMA into a
// ring, in-register dequantisation into the A fragments of mma.sync m16n8k16), but the
// activations never travel with the chunks:
//   - T <= 8 (rows resident): the FP16 hidden rows of all T tokens (at most 8 x 2d bytes)
//     are copied into shared memory once, and every gate/up task reads its routed rows
//     there (the token of each routed row comes with the task entry); the plan's own task
//     table serves, or, for a whole layer, the kernel routes and plans for itself;
//   - 8 < T <= 256 (rows gathered): the kernel's own table of 8-row passes; each gate/up
//     task's rows are copied into one of two slots when the task is published;
//   - each down task's h rows (at most 8 x 2F bytes, published by the gate/up tasks of its
//     expert) are copied once per task into one of two to four slots, as soon as the expert's
//     readiness counter allows, while the compute warps still work on earlier tasks.
// So a chunk's stage is full once its weight bytes have landed; compute warps wait on one
// barrier per chunk and the weight producer is the only per-chunk issuer.
//
// Warps: 0 task fetcher + weight producer, 1 activation producer (hidden rows, h rows per
// down task), 2 publisher (one GPU-scope release per finished gate/up task or down stripe),
// 3-10 compute (16 weight rows each of the 128-row chunk, as in expert_mma.cu), and with the
// un-route fused, trailing un-route tasks (one token's 128 columns of a stripe per compute
// warp) once the stripe's down tasks have been released.
#include "mma_parts.cuh"
#include "route_select.cuh"

namespace moe {

namespace dk {

using namespace mk;

constexpr int kStagesResident = 9;  // weight ring with all hidden rows resident (T <= 8)
constexpr int kStagesGathered = 7;  // weight ring beside the gathered-row slots (8 < T <= 256)
constexpr int kMaxRows = 8;         // routed rows per task (T <= 8, or 8-row passes)
constexpr int kXSlots = 2;          // gathered hidden-row slots
// The fetcher claims its next ticket once at most kReserve of its chunks are in flight: a
// claim (ticket atomic, then the entry, then a gate/up task's tokens) takes about three L2
// round trips, which this many chunks cover.
constexpr int kReserve = 6;
constexpr int kTaskConsumers = 2 + kComputeWarps;  // activation producer, publisher, compute
constexpr int kPubSlots = 2 * kTaskSlots;
constexpr int kMaxHSlots = 4;

template <int S>
struct SmemT {
  uint8_t ring[S][kStageA];
  TaskEntry task[kTaskSlots];
  int task_tok[kTaskSlots][kMaxRows];  // token of each routed row of a gate/up task
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t task_full[kTaskSlots];
  uint64_t task_empty[kTaskSlots];
  uint64_t pub_full[kPubSlots];
  uint64_t x_full[kXSlots];   // resident mode: [0] once; gathered mode: per slot
  uint64_t x_empty[kXSlots];
  uint64_t h_full[kMaxHSlots];
  uint64_t h_empty[kMaxHSlots];
  int abort_flag;
};

constexpr int kSmemLimit = 227 * 1024;

template <bool kGather>
__host__ __device__ inline size_t fixed_smem_bytes() {
  return 1024 + ((sizeof(SmemT<kGather ? kStagesGathered : kStagesResident>) + 127) & ~size_t(127));
}

// Activation arena after the fixed part: the FP16 hidden rows -- all T rows [T][xpitch]
// (resident mode), or kXSlots slots of one task's rows [8][xpitch] (gathered mode) -- then
// `hslots` (2 to 4, as many as fit) slots of one down task's h rows [rows][hpitch]; the 16-byte
// pad per row keeps consecutive rows off the same banks.
struct Arena {
  int xpitch, hpitch, x_bytes, xslot_bytes, slot_bytes, hslots;
};

constexpr int kDnGroupGathered = 4, kDnGroupResident = 2;
constexpr int kNpassShift = 20, kGroupShift = 28;
__device__ __forceinline__ int task_npass(int z) { return max(1, (z >> kNpassShift) & 0xff); }
__device__ __forceinline__ int task_group(int z) { return max(1, (z >> kGroupShift) & 0x7); }

// The plan of the kernel's own front (T <= 8 tokens, at most 256 routes), after the h slots.
constexpr int kFrontRoutes = 256;
struct FrontSmem {
  int ids[kFrontRoutes];      // route t * k + j -> expert
  float w[kFrontRoutes];      // route -> renormalised weight
  int pos[kFrontRoutes];      // route -> position in expert-major order
  int pos_tok[kFrontRoutes];  // position -> token
  int first[kFrontRoutes];    // route -> its expert if it is the expert's first route, else a sentinel
  int touched[kFrontRoutes];  // touched index -> expert (ascending)
  int ucnt[kFrontRoutes];     // touched index -> routes of the expert
  int uoff[kFrontRoutes];     // touched index -> first position of its bucket
  int U;
  uint32_t parity;
};

// The gathered mode's passes, derived by every CTA from the plan's per-expert arrays: per
// touched index u, a[u] = expert | rows << 16 and b[u] = bucket start | first pass << 16
// (8-row passes numbered across the touched experts in order), and per pass its touched
// index (at most E + T k / 8 <= 2048 passes for T <= 256); total = passes.
struct GatherPlan {
  uint32_t a[1024];
  uint32_t b[1024];
  uint16_t pass_u[2048];
  int U, total;
  int wsum[16];  // scratch of the prefix over the pass counts (one per warp)
};

// Entry i (gate/up tasks by pass and stripe, then down tasks) of the gathered mode: its
// pass, that pass's touched index, rows, first routed row and the pass count of its expert
// (S_gu and S_dn are powers of two).  Down task `poison` (self test) waits for touched index
// U instead.
__device__ __forceinline__ TaskEntry gather_entry(const GatherPlan& gp, int i, int ngu, int S_gu, int S_dn,
                                                  int poison) {
  const bool dn = i >= ngu;
  const int j = dn ? i - ngu : i;
  const int S = dn ? S_dn : S_gu;
  const int P = j >> (__ffs(S) - 1), s2 = j & (S - 1);
  const int lo = gp.pass_u[P];
  const int e = static_cast<int>(gp.a[lo] & 0xffffu), c = static_cast<int>(gp.a[lo] >> 16);
  const int p = P - static_cast<int>(gp.b[lo] >> 16);
  const int np = (c + kMaxRows - 1) / kMaxRows;
  const int rows = min(kMaxRows, c - p * kMaxRows);
  const int z = rows | (dn ? 1 << 16 : 0) | (np > 1 ? 1 << 17 : 0) | (np << kNpassShift);
  const int u = (dn && j == poison) ? gp.U : lo;
  return TaskEntry{e | (u << 16), static_cast<int>(gp.b[lo] & 0xffffu) + p * kMaxRows, z, s2};
}

template <bool kGather>
__host__ __device__ inline Arena arena_of(int T, int d, int F, int extra = 0) {
  Arena r;
  const int rows = T < kMaxRows ? T : kMaxRows;
  r.xpitch = 2 * d + 16;
  r.hpitch = 2 * F + 16;
  r.xslot_bytes = rows * r.xpitch;
  r.x_bytes = kGather ? kXSlots * r.xslot_bytes : T * r.xpitch;
  r.slot_bytes = rows * r.hpitch;
  const long long room =
      static_cast<long long>(kSmemLimit) - static_cast<long long>(fixed_smem_bytes<kGather>()) - r.x_bytes - extra;
  const long long fit = r.slot_bytes > 0 ? room / r.slot_bytes : 0;
  r.hslots = static_cast<int>(fit < kMaxHSlots ? fit : kMaxHSlots);
  return r;
}

// Ticket order of this kernel: the plan's gate/up tasks, one per ticket; then its down tasks
// in table order (expert-major, so the down tasks of the experts whose gate/up tasks were
// claimed first come first) -- G = min(group, S_dn) stripes of one expert pass per ticket,
// run as one task (the table holds a pass's S_dn stripes consecutively and S_dn is a multiple
// of G), except the last `nsingle` (at least one per CTA of the grid), one stripe per ticket,
// so that the final claims are short; then, with the un-route fused, one un-route task per
// down stripe and group of eight tokens (one token per compute warp).  A group task copies
// its h rows once and pays one claim and one hand-off for G stripes.  The task entry carries
// G in bits 28-30 of z (the expert's pass count of gathered passes sits in bits 20-27).
// Group size (constants above): 4 when
// the rows are gathered (many short down tasks: T > 8), 2 with the rows resident (T <= 8,
// few tasks per CTA, where larger groups cost more in balance than they save).
struct TicketMap {
  int ngu, G, ngroup, nsingle, ndn_tickets;
};

__device__ __forceinline__ TicketMap ticket_map(int ngu, int ndn, int grid, int S_dn, int group) {
  TicketMap m;
  m.ngu = ngu;
  m.G = min(group, S_dn);
  m.ngroup = (ndn - min(ndn, grid)) / m.G;
  m.nsingle = ndn - m.ngroup * m.G;
  m.ndn_tickets = m.ngroup + m.nsingle;
  return m;
}

// entry index in the table and stripe count of ticket i (gate/up or down; i < ngu + ndn_tickets)
__device__ __forceinline__ int ticket_entry(int i, const TicketMap& m, int& G) {
  G = 1;
  if (i < m.ngu) return i;
  const int j = i - m.ngu;
  if (j < m.ngroup) {
    G = m.G;
    return m.ngu + j * m.G;
  }
  return m.ngu + m.ngroup * m.G + (j - m.ngroup);
}

// Un-route task c: the 128 columns of down stripe c mod S_dn for the tokens
// [8 (c / S_dn), +8), one token per compute warp.
__device__ __forceinline__ TaskEntry unroute_entry(int c, int S_dn) {
  return TaskEntry{0, kComputeWarps * (c / S_dn), 1 << 18, c % S_dn};
}

__device__ __forceinline__ void task_of(const ExpertArgs& a, int i, const TicketMap& m, TaskEntry& e0) {
  if (i < m.ngu + m.ndn_tickets) {
    int G;
    e0 = a.tasks[ticket_entry(i, m, G)];
    e0.z |= G << kGroupShift;
  } else {
    e0 = unroute_entry(i - m.ngu - m.ndn_tickets, a.S_dn);
  }
}

// Entry i of the plan's task order from the kernel's own plan: gate/up tasks (touched order,
// stripe), then down tasks (touched order, stripe); one pass per expert (at most 8 rows).
__device__ __forceinline__ TaskEntry front_entry(const FrontSmem& fs, int i, int ngu, int S_gu, int S_dn) {
  const bool dn = i >= ngu;
  const int j = dn ? i - ngu : i;
  const int S = dn ? S_dn : S_gu;
  const int u = j / S;
  return TaskEntry{fs.touched[u] | (u << 16), fs.uoff[u], fs.ucnt[u] | (dn ? 1 << 16 : 0), j - u * S};
}

__device__ __forceinline__ void front_task_of(const FrontSmem& fs, int i, const TicketMap& m, int S_gu, int S_dn,
                                              TaskEntry& e0) {
  if (i < m.ngu + m.ndn_tickets) {
    int G;
    e0 = front_entry(fs, ticket_entry(i, m, G), m.ngu, S_gu, S_dn);
    e0.z |= G << kGroupShift;
  } else {
    e0 = unroute_entry(i - m.ngu - m.ndn_tickets, S_dn);
  }
}

__device__ __forceinline__ void gather_task_of(const GatherPlan& gp, int i, const TicketMap& m, int S_gu, int S_dn,
                                               int poison, TaskEntry& e0) {
  if (i < m.ngu + m.ndn_tickets) {
    int G;
    e0 = gather_entry(gp, ticket_entry(i, m, G), m.ngu, S_gu, S_dn, poison);
    e0.z |= G << kGroupShift;
  } else {
    e0 = unroute_entry(i - m.ngu - m.ndn_tickets, S_dn);
  }
}

template <typename Smem>
__device__ __forceinline__ bool take_task(Smem& sm, int n, TaskEntry& out, int g, int& tok, int* status, long long limit) {
  const int q = n % kTaskSlots;
  const uint32_t ph = static_cast<uint32_t>((n / kTaskSlots) & 1);
  if (!warp_wait(smem_addr(&sm.task_full[q]), ph, &sm.abort_flag, status, limit)) return false;
  out = sm.task[q];
  tok = sm.task_tok[q][g & (kMaxRows - 1)];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&sm.task_empty[q]));
  return true;
}

// One chunk of a task for one compute warp: per sub-chunk h, the B fragments (elements
// [256c + 128h + 32q, +32) of the routed row as four 16-byte pieces), the dequantised A
// fragments of rows g and g + 8, and 8 MMAs into 8 independent accumulators.
__device__ __forceinline__ void chunk_mma(const ChunkCodes& cc, const uint8_t* bc, bool live, float (&acc)[8][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 xb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      xb[j] = live ? *reinterpret_cast<const uint4*>(bc + 256 * h + 16 * j) : make_uint4(0, 0, 0, 0);
    uint32_t fa[16], fb[16];
    dequant32(cc.ca[h], cc.sa[h], fa);
    dequant32(cc.cb[h], cc.sb[h], fb);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mma_16816(acc[2 * j], fa[4 * j + 0], fb[4 * j + 0], fa[4 * j + 1], fb[4 * j + 1], xb[j].x, xb[j].y);
      mma_16816(acc[2 * j + 1], fa[4 * j + 2], fb[4 * j + 2], fa[4 * j + 3], fb[4 * j + 3], xb[j].z, xb[j].w);
    }
  }
}

// The chunk loop of one task for one compute warp, two chunks per barrier round: wait for
// both stages, copy their codes and scales into registers, hand both stages back, then run
// the MMAs.  Each lane waits on its own (no warp vote per chunk); a wait that gives up leaves
// the lane computing on stale data until the task ends, where the warp decides together
// (every later wait returns at once because the CTA's abort flag is raised).  The 16
// k-steps of a chunk go to 8 independent accumulators, summed in a fixed order at the end.
// `brow` is the thread's activation row (routed row g) in shared memory.
template <int kStages, typename Smem>
__device__ __forceinline__ bool run_task_chunks(Smem& sm, const ExpertArgs& a, int& stage, uint32_t& phase,
                                                float (&acc)[8][4], int lra, int lrb, int nck, const uint8_t* brow,
                                                bool live, int q, bool tr, int& tcnt) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  bool ok = true;
  for (int c = 0; c < nck; c += 2) {
    const bool two = c + 1 < nck;
    ChunkCodes c0, c1;
    if (tr) trace_ev(a, 2, tcnt, 7, c);
    ok &= bounded_wait(smem_addr(&sm.full[stage]), phase, &sm.abort_flag, a.status, a.wait_limit);
    if (tr) trace_ev(a, 2, tcnt, 8, c);
    load_chunk_codes(&sm.ring[stage][0], lra, lrb, q, c0);
    const int st0 = stage;
    if (++stage == kStages) { stage = 0; phase ^= 1u; }
    int st1 = st0;
    if (two) {
      ok &= bounded_wait(smem_addr(&sm.full[stage]), phase, &sm.abort_flag, a.status, a.wait_limit);
      load_chunk_codes(&sm.ring[stage][0], lra, lrb, q, c1);
      st1 = stage;
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
    // the stages' bytes are in registers: hand them back to the producer
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(smem_addr(&sm.empty[st0]));
      if (two) mbar_arrive(smem_addr(&sm.empty[st1]));
    }
    const uint8_t* bc = brow + 2 * kChunk * c + 64 * q;
    chunk_mma(c0, bc, live, acc);
    if (two) chunk_mma(c1, bc + 2 * kChunk, live, acc);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    acc[0][i] = ((acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i])) + ((acc[4][i] + acc[5][i]) + (acc[6][i] + acc[7][i]));
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait for the last phase of a barrier this warp's copies complete on (drain).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kDrainCycles) {}
}

}  // namespace dk

using namespace dk;

// This CTA's share (grid-strided by warp lanes) of the workspace copy of the kernel's own
// plan: the arrays the plan kernel writes, in its layout, for at most 8 rows per expert (one
// pass each), so that later calls on the same workspace find the plan of this layer.
__device__ __forceinline__ void write_front_plan(const ExpertArgs& a, const DecFront& f, const FrontSmem& fs, int U) {
  const int lane = threadIdx.x & 31;
  const int stride = static_cast<int>(gridDim.x) * 32, first = static_cast<int>(blockIdx.x) * 32 + lane;
  const int E = a.E, R = a.T * a.k;
  const int ngu = U * a.S_gu, ntask = U * (a.S_gu + a.S_dn);
  for (int e = first; e <= E; e += stride) {
    // bucket start: the routes to lower experts; count: the routes to e
    int off = 0, cnt = 0;
    for (int u = 0; u < U; ++u) {
      const int x = fs.touched[u];
      off += x < e ? fs.ucnt[u] : 0;
      cnt += x == e ? fs.ucnt[u] : 0;
    }
    f.offsets[e] = off;
    if (e < E) f.counts[e] = cnt;
  }
  for (int u = first; u <= U; u += stride) {
    if (u < U) f.touched[u] = fs.touched[u];
    f.gu_start[u] = u * a.S_gu;
    f.dn_start[u] = u * a.S_dn;
  }
  for (int r = first; r < R; r += stride) {
    f.route_pos[r] = fs.pos[r];
    f.pos_tok[r] = fs.pos_tok[r];
    f.route_w[r] = fs.w[r];
  }
  for (int i = first; i < ntask; i += stride) f.tasks[i] = front_entry(fs, i, ngu, a.S_gu, a.S_dn);
  if (blockIdx.x == 0 && lane == 0) {
    int mx = 0;
    for (int u = 0; u < U; ++u) mx = max(mx, fs.ucnt[u]);
    f.meta[META_U] = U;
    f.meta[META_NGU] = ngu;
    f.meta[META_NDN] = U * a.S_dn;
    f.meta[META_MAXROWS] = mx;
    f.meta[META_YFMT] = 0;
  }
}

// kGather false: T <= 8, every token's hidden row resident (plan's task table, one pass per
// expert, optionally the fused un-route); kGather true: 8 < T <= 256, each gate/up task's rows
// gathered into one of kXSlots slots, task table of 8-row passes (written by the plan).
// kNpl > 0 (T <= 8, un-route fused): the kernel's own front, with kNpl logits per lane in
// the router (E <= 32 kNpl); the plan comes from shared memory, the counters from the set
// `f.parity` selects.
template <bool kFused, bool kGather, int kNpl>
__global__ void __launch_bounds__(kThreads, 1)
    expert_dec_kernel(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_w2,
                      const __grid_constant__ CUtensorMap tm_s13, const __grid_constant__ CUtensorMap tm_s2,
                      const __grid_constant__ ExpertArgs a, const __grid_constant__ DecFront f) {
  constexpr bool kFront = kNpl > 0;
  static_assert(!kFront || (kFused && !kGather), "the own front is for the resident, fused variant");
  constexpr int kStages = kGather ? kStagesGathered : kStagesResident;
  using Smem = SmemT<kStages>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* arena = reinterpret_cast<uint8_t*>(&sm) + ((sizeof(Smem) + 127) & ~size_t(127));
  const Arena ar = arena_of<kGather>(
      a.T, a.d, a.F, kFront ? static_cast<int>(sizeof(FrontSmem)) : kGather ? static_cast<int>(sizeof(GatherPlan)) : 0);
  uint8_t* xs = arena;                 // hidden rows (resident) or the gathered-row slots
  uint8_t* hs = arena + ar.x_bytes;    // h slots
  FrontSmem& fs = *reinterpret_cast<FrontSmem*>(hs + ar.hslots * ar.slot_bytes);   // kFront only
  GatherPlan& gp = *reinterpret_cast<GatherPlan*>(hs + ar.hslots * ar.slot_bytes);  // kGather only
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int tcnt0 = 2;
  if (tid == 0) trace_ev(a, 5, tcnt0, 14, 0);  // kernel entry, before the dependency wait

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_addr(&sm.full[i]), 1);
      mbar_init(smem_addr(&sm.empty[i]), kComputeWarps);
    }
    for (int i = 0; i < kTaskSlots; ++i) {
      mbar_init(smem_addr(&sm.task_full[i]), 1);
      mbar_init(smem_addr(&sm.task_empty[i]), kTaskConsumers);
    }
    for (int i = 0; i < kPubSlots; ++i) mbar_init(smem_addr(&sm.pub_full[i]), kComputeWarps);
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(smem_addr(&sm.x_full[i]), 1);
      mbar_init(smem_addr(&sm.x_empty[i]), kComputeWarps);
    }
    for (int i = 0; i < kMaxHSlots; ++i) {
      mbar_init(smem_addr(&sm.h_full[i]), 1);
      mbar_init(smem_addr(&sm.h_empty[i]), kComputeWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w13);
    prefetch_tmap(&tm_w2);
    prefetch_tmap(&tm_s13);
    prefetch_tmap(&tm_s2);
  }
  // everything above is local to the CTA; the plan, the counters and the FP16 hidden rows
  // come from the preceding kernel (kFront: the logits, the hidden rows and the counter set)
  pdl_wait();
  pdl_launch_dependents();
  uint32_t* ctr_ready = a.ready;
  uint32_t* ctr_dn = a.dn_done;
  uint32_t* ctr_ticket = a.ticket;
  int front_U = 0;
  if constexpr (kFront) {
    // ---- the kernel's own front: route, FP16 hidden rows, plan (every CTA the same) ----
    const int T = a.T, k = a.k, R = T * k;
    if (tid == 0) fs.parity = __ldcg(f.parity) & 1u;
    int pcnt = 0;
    if (warp < T) {
      route_token<kNpl>(f.logits, warp, a.E, k, blockIdx.x == 0 ? f.ids : nullptr, f.weights, fs.ids, fs.w, warp);
      if (tid == 0) trace_ev(a, 6, pcnt, 16, 0);  // token 0 routed
    } else {
      // hidden rows -> FP16 into the resident rows (CTA 0: also the workspace copy)
      const int n8 = T * a.d / 8, per_row = a.d / 8;
      bool bad = false;
      for (int i = tid - 32 * T; i < n8; i += kThreads - 32 * T) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(f.hidden) + i);
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
        uint4 o;
        __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 v = __bfloat1622float2(b[q]);
          bad |= !(fabsf(v.x) <= 65504.f) || !(fabsf(v.y) <= 65504.f);
          h[q] = __floats2half2_rn(v.x, v.y);
        }
        const int t = i / per_row, c8 = i - t * per_row;
        *reinterpret_cast<uint4*>(xs + t * ar.xpitch + 16 * c8) = o;
        if (blockIdx.x == 0) reinterpret_cast<uint4*>(f.x16)[i] = o;
      }
      if (bad && blockIdx.x == 0) atomicOr(a.status, static_cast<int>(MOE_DEV_HIDDEN_RANGE));
      if (tid == 32 * T) trace_ev(a, 7, pcnt, 17, 0);  // first converter's rows done
    }
    // pad the route ids to a multiple of 4 with a sentinel above every expert id
    if (tid >= R && tid < ((R + 3) & ~3)) fs.ids[tid] = 0x7fffffff;
    __syncthreads();
    if (tid == 0) trace_ev(a, 6, pcnt, 18, 0);
    const uint32_t par = fs.parity;
    ctr_ready = f.sets + par * kDecSetWords;
    ctr_dn = ctr_ready + kDecReadyWords;
    ctr_ticket = ctr_ready + kDecTicketWord;
    if (blockIdx.x == 0) {
      // the other set, for the next launch (no CTA of this one touches it)
      uint32_t* other = f.sets + (par ^ 1u) * kDecSetWords;
      for (int i = tid; i < kDecSetWords; i += kThreads) other[i] = 0u;
    }
    // route r: its bucket's first position (routes to lower experts), its rank among the
    // routes to the same expert (route order), the bucket size
    const int R4 = (R + 3) >> 2;
    int e = 0, rank = 0, off = 0, cnt = 0;
    if (tid < R) {
      e = fs.ids[tid];
      const int4* ids4 = reinterpret_cast<const int4*>(fs.ids);
#pragma unroll 4
      for (int q = 0; q < R4; ++q) {
        const int4 x = ids4[q];
        const int r0 = 4 * q;
        off += (x.x < e) + (x.y < e) + (x.z < e) + (x.w < e);
        cnt += (x.x == e) + (x.y == e) + (x.z == e) + (x.w == e);
        rank += (x.x == e && r0 < tid) + (x.y == e && r0 + 1 < tid) + (x.z == e && r0 + 2 < tid) +
                (x.w == e && r0 + 3 < tid);
      }
      fs.pos[tid] = off + rank;
      fs.pos_tok[off + rank] = tid / k;
      fs.first[tid] = rank == 0 ? e : 0x7fffffff;  // the expert, at its first route only
    } else if (tid < 4 * R4) {
      fs.first[tid] = 0x7fffffff;
    }
    const int U = __syncthreads_count(tid < R && rank == 0);
    if (tid == 0) trace_ev(a, 6, pcnt, 19, 0);
    if (tid < R && rank == 0) {
      // touched index: the distinct experts below e
      const int4* first4 = reinterpret_cast<const int4*>(fs.first);
      int u = 0;
#pragma unroll 4
      for (int q = 0; q < R4; ++q) {
        const int4 x = first4[q];
        u += (x.x < e) + (x.y < e) + (x.z < e) + (x.w < e);
      }
      fs.touched[u] = e;
      fs.ucnt[u] = cnt;
      fs.uoff[u] = off;
    }
    if (tid == 0) fs.U = U;
    __syncthreads();
    front_U = U;
  } else if constexpr (kGather) {
    // ---- the 8-row passes from the plan's per-expert arrays (every CTA the same) ----
    // thread t takes touched indices 3t .. 3t+2: their experts, rows and bucket starts, and
    // the exclusive prefix of their pass counts (warp scan, then one over the warp totals)
    const int U = __ldg(a.meta + META_U);
    int np[3], run = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int u = 3 * tid + j;
      np[j] = 0;
      if (u < U) {
        const int e = __ldg(a.touched + u);
        const int c = __ldg(a.counts + e);
        gp.a[u] = static_cast<uint32_t>(e) | (static_cast<uint32_t>(c) << 16);
        gp.b[u] = static_cast<uint32_t>(__ldg(a.offsets + e));
        np[j] = (c + kMaxRows - 1) / kMaxRows;
      }
      run += np[j];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) gp.wsum[warp] = incl;
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        const int v = gp.wsum[w];
        gp.wsum[w] = acc;
        acc += v;
      }
      gp.U = U;
      gp.total = acc;
    }
    __syncthreads();
    int p0 = gp.wsum[warp] + incl - run;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int u = 3 * tid + j;
      if (u < U) gp.b[u] |= static_cast<uint32_t>(p0) << 16;
      for (int p = 0; p < np[j]; ++p) gp.pass_u[p0 + p] = static_cast<uint16_t>(u);
      p0 += np[j];
    }
    __syncthreads();
  } else {
    __syncthreads();
  }
  const uint32_t ring0 = smem_addr(&sm.ring[0][0]);
  int tcnt = 0;
  if (tid == 0) trace_ev(a, 5, tcnt, 10, 0);

  if (warp == 0) {
    // ------------- task fetcher + weight producer -------------
    const uint64_t pol = policy_evict_first();
    const int ngu = kFront ? front_U * a.S_gu : kGather ? gp.total * a.S_gu : __ldg(a.meta + META_NGU);
    const int ndn = kFront ? front_U * a.S_dn : kGather ? gp.total * a.S_dn : __ldg(a.meta + META_NDN);
    const TicketMap tmap = ticket_map(ngu, ndn, static_cast<int>(gridDim.x), a.S_dn,
                                      kGather ? kDnGroupGathered : kDnGroupResident);
    const int ntot = ngu + tmap.ndn_tickets + (kFused ? a.ncb : 0);  // tickets
    const TaskEntry kEnd = TaskEntry{-1, 0, 0, 0};
    int stage = 0, issued = 0, n = 0, chunk_seq = 0;
    uint32_t phase = 0;
    int cur = blockIdx.x;
    TaskEntry entry = kEnd;
    if (lane == 0) {
      if (cur >= ntot) entry = kEnd;
      else if (kFront) front_task_of(fs, cur, tmap, a.S_gu, a.S_dn, entry);
      else if (kGather) gather_task_of(gp, cur, tmap, a.S_gu, a.S_dn, a.poison_dn, entry);
      else task_of(a, cur, tmap, entry);
    }
    // the tokens of a gate/up task's routed rows, loaded as soon as its entry is known
    auto load_tokens = [&]() {
      const int ey = __shfl_sync(0xffffffffu, entry.y, 0), ez = __shfl_sync(0xffffffffu, entry.z, 0);
      const bool gu = __shfl_sync(0xffffffffu, cur, 0) < ngu;
      if (!gu || lane >= (ez & 0xffff)) return 0;
      return kFront ? fs.pos_tok[ey + lane] : __ldg(a.pos_tok + ey + lane);
    };
    int tok = load_tokens();
    if (lane == 0 && kFront) trace_ev(a, 0, tcnt, 20, 0);  // first entry and tokens known
    bool ok = true;
    while (ok) {
      const int q = n % kTaskSlots;
      if (!warp_wait(smem_addr(&sm.task_empty[q]), static_cast<uint32_t>(((n / kTaskSlots) & 1) ^ 1),
                     &sm.abort_flag, a.status, a.wait_limit)) {
        ok = false;
        break;
      }
      if (lane == 0 && kFront && n == 0) trace_ev(a, 0, tcnt, 21, 0);
      const bool live = __shfl_sync(0xffffffffu, cur, 0) < ntot;
      // publish the entry (and the tokens, whose load may still be in flight) to the other
      // roles: after the task's first chunk has been issued -- its stage is freed by earlier,
      // already published tasks -- and before any later chunk may wait on a stage that only
      // this task's own chunks would free
      bool published = false;
      auto publish = [&]() {
        int tk[kMaxRows];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) tk[r] = __shfl_sync(0xffffffffu, tok, r);
        if (lane == 0) {
          sm.task[q] = live ? entry : kEnd;
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) sm.task_tok[q][r] = tk[r];
          mbar_arrive(smem_addr(&sm.task_full[q]));
          trace_ev(a, 0, tcnt, 1, cur);
        }
        published = true;
      };
      if (!live) {
        publish();
        break;
      }
      const int x = __shfl_sync(0xffffffffu, entry.x, 0);
      const int z = __shfl_sync(0xffffffffu, entry.z, 0);
      const int s = __shfl_sync(0xffffffffu, entry.w, 0);
      const int e = x & 0xffff;
      const bool is_dn = ((z >> 16) & 1) != 0;
      // a down task streams the chunks of its G stripes one stripe after the other
      const int G = is_dn ? task_group(z) : 1;
      int rA0, nck;
      const CUtensorMap* tm;
      if (!is_dn) {
        rA0 = (e - a.e_lo) * 2 * a.F + s * kGuRows;
        tm = &tm_w13;
        nck = a.d / kChunk;
      } else {
        rA0 = (e - a.e_lo) * a.d + s * kDnRows;
        tm = &tm_w2;
        nck = a.F / kChunk;
      }
      const int half = is_dn ? 64 : a.F;  // second box: 64 rows further (down) or the up rows
      int nall = G * nck;
      if (kFused && ((z >> 18) & 1)) nall = 0;  // un-route task: no weights
      const CUtensorMap* tms = is_dn ? &tm_s2 : &tm_s13;
      ++n;
      for (int c = 0, g = 0, kc = 0; c < nall; ++c) {
        if (!warp_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, &sm.abort_flag, a.status, a.wait_limit)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t sb = ring0 + stage * kStageA;
          const uint32_t fa = smem_addr(&sm.full[stage]);
          const int r0 = rA0 + g * kDnRows, r1 = r0 + half;
          if (kFront && chunk_seq == 0) trace_ev(a, 0, tcnt, 22, 0);
          mbar_arrive_expect_tx(fa, kStageA);
          tma_load_2d(sb, tm, kc * (kChunk / 2), r0, fa, pol);
          if (kFront && chunk_seq == 0) trace_ev(a, 0, tcnt, 23, 0);
          tma_load_2d(sb + kCodeBytes / 2, tm, kc * (kChunk / 2), r1, fa, pol);
          tma_load_2d(sb + kCodeBytes, tms, kc * (kChunk / 16), r0, fa, pol);
          tma_load_2d(sb + kCodeBytes + kScaleBytes / 2, tms, kc * (kChunk / 16), r1, fa, pol);
          trace_ev(a, 0, tcnt, 2, chunk_seq);
        }
        ++chunk_seq;
        ++issued;
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
        if (++kc == nck) { kc = 0; ++g; }
        if (c == 0) publish();
      }
      if (!published) publish();  // un-route task (no chunks), or the first wait gave up
      if (!ok) break;
      // take the next ticket once at most kReserve chunks are in flight (2 among the last
      // gridDim.x tickets, so that the final tasks go to the CTAs that run dry first)
      const int reserve = __shfl_sync(0xffffffffu, cur, 0) + static_cast<int>(gridDim.x) >= ntot ? 2 : kReserve;
      if (issued > reserve) {
        const int sq = issued - 1 - reserve + kStages;  // the issue that reuses that chunk's stage
        if (!warp_wait(smem_addr(&sm.empty[sq % kStages]), static_cast<uint32_t>(((sq / kStages) & 1) ^ 1),
                       &sm.abort_flag, a.status, a.wait_limit)) {
          ok = false;
          break;
        }
      }
      if (lane == 0) {
        cur = static_cast<int>(atomicAdd(ctr_ticket, 1u)) + static_cast<int>(gridDim.x);
        if (cur >= ntot) entry = kEnd;
        else if (kFront) front_task_of(fs, cur, tmap, a.S_gu, a.S_dn, entry);
        else if (kGather) gather_task_of(gp, cur, tmap, a.S_gu, a.S_dn, a.poison_dn, entry);
        else task_of(a, cur, tmap, entry);
      }
      tok = load_tokens();
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int i = 0; i < min(issued, kStages); ++i) {
        if (--st < 0) { st = kStages - 1; ph ^= 1u; }
        drain_wait(smem_addr(&sm.full[st]), ph);
      }
    }
  } else if (warp == 1) {
    // ------------- activation producer: hidden rows (all at once when resident, per gate/up
    // task when gathered), h rows per down task -------------
    if (!kGather && !kFront) {
      if (lane == 0) mbar_arrive_expect_tx(smem_addr(&sm.x_full[0]), static_cast<uint32_t>(a.T * 2 * a.d));
      __syncwarp();
      if (lane < a.T)
        bulk_copy_g2s(smem_addr(xs + lane * ar.xpitch), a.x16 + static_cast<size_t>(lane) * a.d, 2 * a.d,
                      smem_addr(&sm.x_full[0]));
    }
    int n = 0, ndn = 0, ngu = 0;
    while (true) {
      TaskEntry te;
      int tok = 0;
      if (!take_task(sm, n++, te, lane, tok, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if (kFused && is_unroute(te)) continue;
      if (((te.z >> 16) & 1) == 0) {
        if (!kGather) continue;  // gate/up: its rows are resident
        // gate/up: copy the task's routed rows (lane r: the row of token tok_r) into a slot
        const int xslot = ngu % kXSlots;
        if (!warp_wait(smem_addr(&sm.x_empty[xslot]), static_cast<uint32_t>(((ngu / kXSlots) & 1) ^ 1),
                       &sm.abort_flag, a.status, a.wait_limit))
          break;
        const int rows = te.z & 0xffff;
        if (lane == 0) mbar_arrive_expect_tx(smem_addr(&sm.x_full[xslot]), static_cast<uint32_t>(rows * 2 * a.d));
        __syncwarp();
        if (lane < rows)
          bulk_copy_g2s(smem_addr(xs + xslot * ar.xslot_bytes + lane * ar.xpitch),
                        a.x16 + static_cast<size_t>(tok) * a.d, 2 * a.d, smem_addr(&sm.x_full[xslot]));
        ++ngu;
        continue;
      }
      const int slot = ndn % ar.hslots;
      const uint32_t use = static_cast<uint32_t>(ndn / ar.hslots);
      if (!warp_wait(smem_addr(&sm.h_empty[slot]), (use & 1u) ^ 1u, &sm.abort_flag, a.status, a.wait_limit)) break;
      // every gate/up task (all passes, S_gu stripes each) of this expert must have published
      // its h rows; the entry carries the pass count in bits 20+ (0: one pass)
      const int u = (te.x >> 16) & 0xffff, row0 = te.y, rows = te.z & 0xffff;
      const int npass = task_npass(te.z);
      const bool good = warp_wait_counter(ctr_ready + u, static_cast<uint32_t>(npass * a.S_gu), &sm.abort_flag,
                                          a.status, a.wait_limit);
      if (!good) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_addr(&sm.h_full[slot]), static_cast<uint32_t>(rows * 2 * a.F));
        trace_ev(a, 1, tcnt, 3, ndn);
      }
      __syncwarp();
      if (lane < rows)
        bulk_copy_g2s(smem_addr(hs + slot * ar.slot_bytes + lane * ar.hpitch),
                      a.hs16 + static_cast<size_t>(row0 + lane) * a.F, 2 * a.F, smem_addr(&sm.h_full[slot]));
      ++ndn;
    }
    // drain: every copy this warp started has landed before the CTA exits
    if (lane == 0) {
      if (!kGather && !kFront) drain_wait(smem_addr(&sm.x_full[0]), 0);
      for (int i = max(0, ngu - kXSlots); i < ngu; ++i)
        drain_wait(smem_addr(&sm.x_full[i % kXSlots]), static_cast<uint32_t>((i / kXSlots) & 1));
      for (int i = max(0, ndn - ar.hslots); i < ndn; ++i)
        drain_wait(smem_addr(&sm.h_full[i % ar.hslots]), static_cast<uint32_t>((i / ar.hslots) & 1));
    }
  } else if (warp == 2) {
    // ------------- publisher: release each finished gate/up task's h rows (fused: and each
    // finished down task's y rows, counted per stripe) -------------
    int n = 0, pub_n = 0, unused_tok = 0;
    if constexpr (kFront) write_front_plan(a, f, fs, front_U);
    while (true) {
      TaskEntry te;
      if (!take_task(sm, n++, te, 0, unused_tok, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if (kFused && is_unroute(te)) continue;
      const bool dn = ((te.z >> 16) & 1) != 0;
      if (dn && !kFused) continue;  // down task, un-route in its own kernel: nothing to publish
      // one release per gate/up task, one per stripe of a down task
      const int G = dn ? task_group(te.z) : 1;
      bool good = true;
      for (int g = 0; g < G && good; ++g) {
        uint32_t* ctr = dn ? ctr_dn + te.w + g : ctr_ready + ((te.x >> 16) & 0xffff);
        const int slot = pub_n % kPubSlots;
        const uint32_t ph = static_cast<uint32_t>((pub_n / kPubSlots) & 1);
        ++pub_n;
        good = warp_wait(smem_addr(&sm.pub_full[slot]), ph, &sm.abort_flag, a.status, a.wait_limit);
        if (good && lane == 0) {
          fence_acq_rel_gpu();
          red_add_relaxed_gpu_u32(ctr, 1u);
          trace_ev(a, 4, tcnt, 9, pub_n);
        }
        __syncwarp();
      }
      if (!good) break;
    }
  } else {
    // ------------- compute warps: dequantise into A fragments, mma.sync, epilogue -------------
    const int cw = warp - kFirstCompute;  // 0..7
    const int g = lane >> 2, q = lane & 3;
    const int fr = frag_row(g);
    int stage = 0, n = 0, pub_n = 0, ndn = 0, ngu = 0;
    uint32_t phase = 0;
    bool ok = true, have_x = kFront;  // kFront: the prologue wrote the hidden rows
    const bool tr = a.trace != nullptr && lane == 0 && (cw == 0 || cw == kComputeWarps - 1);
    const int trole = cw == 0 ? 2 : 3;
    while (ok) {
      TaskEntry te;
      int tok = 0;
      if (tr) trace_ev(a, trole, tcnt, 15, n);
      if (!take_task(sm, n, te, g, tok, a.status, a.wait_limit)) break;
      if (te.x < 0) break;
      if constexpr (kFused) {
        if (is_unroute(te)) {
          ++n;
          const int t = min(te.y + cw, a.T - 1), c = te.w * kDnRows + 4 * lane;
          Unroute4Pre u;
          unroute4_pre<kFront>(a, t, c, u, fs.pos, fs.w);
          // every down task of the stripe has published its y columns
          const uint32_t dn_per_stripe = static_cast<uint32_t>(
              kFront ? front_U : kGather ? gp.total : __ldg(a.meta + META_NDN) / a.S_dn);
          if (tr) trace_ev(a, trole, tcnt, 12, n);
          if (!warp_wait_counter(ctr_dn + te.w, dn_per_stripe, &sm.abort_flag, a.status, a.wait_limit)) break;
          if (tr) trace_ev(a, trole, tcnt, 13, n);
          if (te.y + cw < a.T) unroute4_post<kFront>(a, t, c, u, fs.pos, fs.w);
          continue;
        }
      }
      if (tr) trace_ev(a, trole, tcnt, 5, (((te.z >> 16) & 1) << 15) | (n & 0x7fff));
      const int row0 = te.y, rows = te.z & 0xffff, s = te.w;
      const bool is_dn = ((te.z >> 16) & 1) != 0;
      const int nck = (is_dn ? a.F : a.d) / kChunk;
      const bool live = g < rows;
      const uint8_t* brow;
      int slot = 0;
      if (!is_dn && kGather) {
        slot = ngu % kXSlots;
        if (!warp_wait(smem_addr(&sm.x_full[slot]), static_cast<uint32_t>((ngu / kXSlots) & 1), &sm.abort_flag,
                       a.status, a.wait_limit))
          break;
        brow = xs + slot * ar.xslot_bytes + g * ar.xpitch;
      } else if (!is_dn) {
        if (!have_x) {
          if (!warp_wait(smem_addr(&sm.x_full[0]), 0u, &sm.abort_flag, a.status, a.wait_limit)) break;
          have_x = true;
        }
        brow = xs + (live ? tok : 0) * ar.xpitch;
      } else {
        slot = ndn % ar.hslots;
        if (!warp_wait(smem_addr(&sm.h_full[slot]), static_cast<uint32_t>((ndn / ar.hslots) & 1), &sm.abort_flag,
                       a.status, a.wait_limit))
          break;
        brow = hs + slot * ar.slot_bytes + g * ar.hpitch;
      }
      // tile rows (0..127) of fragment rows g and g + 8
      const int lra = is_dn ? 16 * cw + fr : 8 * cw + fr;
      const int lrb = is_dn ? 16 * cw + 8 + fr : 64 + 8 * cw + fr;
      float acc[8][4];
      if (!is_dn) {
        ok = run_task_chunks<kStages>(sm, a, stage, phase, acc, lra, lrb, nck, brow, live, q, tr && cw == 0, tcnt);
        if (!ok) break;
        if (kGather) {
          // the slot's hidden rows are consumed
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.x_empty[slot]));
          ++ngu;
        }
        if (tr) trace_ev(a, trole, tcnt, 6, n);
        ++n;
        // ---- epilogue: fragment rows g / g+8, routed rows 2q, 2q + 1 ----
        const int nidx = s * kGuRows + 8 * cw + fr;  // element n of h
        const float sc = ts13_of(a, te.x & 0xffff);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int r = 2 * q + cc;
          if (r < rows)
            a.hs16[static_cast<size_t>(row0 + r) * a.F + nidx] =
                h_store_value(silu_mul(acc[0][cc] * sc, acc[0][2 + cc] * sc), a.status);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.pub_full[pub_n % kPubSlots]));
        ++pub_n;
        continue;
      }
      // down task: its G stripes in turn on the same h rows, one epilogue each
      const int G = task_group(te.z);
      const float sc = ts2_of(a, te.x & 0xffff) * kHUnscale;
      for (int gs = 0; gs < G; ++gs) {
        ok = run_task_chunks<kStages>(sm, a, stage, phase, acc, lra, lrb, nck, brow, live, q, tr && cw == 0, tcnt);
        if (!ok) break;
        if (gs + 1 == G) {
          // the slot's h rows are consumed
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.h_empty[slot]));
          ++ndn;
          if (tr) trace_ev(a, trole, tcnt, 6, n);
        }
        const int ra = (s + gs) * kDnRows + lra, rb = (s + gs) * kDnRows + lrb;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int r = 2 * q + cc;
          if (r < rows) {
            float* yrow = a.y + static_cast<size_t>(row0 + r) * a.d;
            yrow[ra] = acc[0][cc] * sc;
            yrow[rb] = acc[0][2 + cc] * sc;
          }
        }
        if constexpr (kFused) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.pub_full[pub_n % kPubSlots]));
          ++pub_n;
        }
      }
      if (!ok) break;
      ++n;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int c2 = 1;
    trace_ev(a, 5, c2, 11, 0);
    if constexpr (kFront) {
      // the last CTA out hands the other (zeroed) counter set to the next launch
      __threadfence();
      if (atomicAdd(f.done, 1u) == gridDim.x - 1) {
        *f.done = 0u;
        *f.parity = fs.parity ^ 1u;
      }
    }
  }
}

// T at or below which every token's hidden row stays resident; above it (up to kMaxGatherT)
// each gate/up task's rows are gathered, its tasks being 8-row passes.
constexpr int kMaxGatherT = 256;

size_t expert_dec_smem_bytes(int T, int d, int F) {
  if (T <= kMaxRows) {
    const Arena ar = arena_of<false>(T, d, F);
    return fixed_smem_bytes<false>() + ar.x_bytes + static_cast<size_t>(ar.hslots) * ar.slot_bytes;
  }
  const Arena ar = arena_of<true>(T, d, F, static_cast<int>(sizeof(GatherPlan)));
  return fixed_smem_bytes<true>() + ar.x_bytes + static_cast<size_t>(ar.hslots) * ar.slot_bytes + sizeof(GatherPlan);
}

static size_t front_smem_bytes(int T, int d, int F) {
  const Arena ar = arena_of<false>(T, d, F, static_cast<int>(sizeof(FrontSmem)));
  return fixed_smem_bytes<false>() + ar.x_bytes + static_cast<size_t>(ar.hslots) * ar.slot_bytes + sizeof(FrontSmem);
}

bool expert_dec_supports(int T, int d, int F) {
  if (T < 1 || T > kMaxGatherT || !expert_mma_supports(d, F)) return false;
  const int hslots = T <= kMaxRows ? arena_of<false>(T, d, F).hslots
                                   : arena_of<true>(T, d, F, static_cast<int>(sizeof(GatherPlan))).hslots;
  return hslots >= 2 && expert_dec_smem_bytes(T, d, F) <= static_cast<size_t>(kSmemLimit);
}

bool expert_dec_front_supports(int T, int d, int F, int E, int k) {
  if (T < 1 || T > kMaxRows || T * k > kFrontRoutes || E > kDecReadyWords || !expert_mma_supports(d, F)) return false;
  if (d / kDnRows > kDecTicketWord - kDecReadyWords) return false;
  return arena_of<false>(T, d, F, static_cast<int>(sizeof(FrontSmem))).hslots >= 2 &&
         front_smem_bytes(T, d, F) <= static_cast<size_t>(kSmemLimit);
}

bool expert_dec_gathers(int T) { return T > kMaxRows; }

int expert_dec_unroute_tasks(int T, int d, int F) {
  // fused for the resident rows only: above eight tokens the trailing un-route tasks (one
  // CTA's eight warps per stripe and token group, each after its stripe's last down task)
  // measured slower than the separate, fully parallel un-route kernel
  return T <= kMaxRows && expert_dec_supports(T, d, F) ? (d / kDnRows) * ((T + kComputeWarps - 1) / kComputeWarps)
                                                       : 0;
}

cudaError_t launch_expert_dec(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_s13, const CUtensorMap& tm_s2, int num_sms,
                              cudaStream_t stream) {
  const size_t smem = expert_dec_smem_bytes(a.T, a.d, a.F);
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const ExpertArgs,
               const DecFront);
  if (a.T > kMaxRows) kern = expert_dec_kernel<false, true, 0>;  // the un-route is fused for T <= 8 only
  else kern = a.ncb > 0 ? expert_dec_kernel<true, false, 0> : expert_dec_kernel<false, false, 0>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, stream, tm_w13, tm_w2, tm_s13, tm_s2, a, DecFront{});
}

cudaError_t launch_expert_dec_front(const ExpertArgs& a, const DecFront& f, const CUtensorMap& tm_w13,
                                    const CUtensorMap& tm_w2, const CUtensorMap& tm_s13, const CUtensorMap& tm_s2,
                                    int num_sms, cudaStream_t stream) {
  if (a.ncb <= 0 || !expert_dec_front_supports(a.T, a.d, a.F, a.E, a.k)) return cudaErrorInvalidValue;
  const size_t smem = front_smem_bytes(a.T, a.d, a.F);
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const ExpertArgs,
               const DecFront) = a.E <= 512 ? expert_dec_kernel<true, false, 16> : expert_dec_kernel<true, false, 32>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, stream, tm_w13, tm_w2, tm_s13, tm_s2, a, f);
}

}  // namespace moe
