// Shared definitions of the routed-MoE CUDA path: workspace layout, task geometry and
// thin inline-PTX wrappers for sm_103a (mbarrier, TMA, cp.async, tcgen05).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------------
// Geometry of the expert tasks.
//   gate/up task : one expert, 64 F-rows of the gate projection plus the same 64 rows
//                  of the up projection (a 128-row A tile), the full K = d;
//   down task    : one expert, 128 d-rows of W2, the full K = ffn;
//   rows         : at most kRowsPerPass routed rows per pass; experts with more rows
//                  run several passes (each re-reads the weights).
// The weights stream in K chunks of kChunkK elements (64 bytes of codes per row).
// ---------------------------------------------------------------------------------
constexpr int kChunkK = 128;
constexpr int kGuRows = 64;         // F-rows per gate/up task (x2 for gate and up)
constexpr int kDnRows = 128;        // d-rows per down task
// One counter set of the decode kernel that routes its own tokens: gate/up readiness per
// touched expert [1024], down completion per stripe [32], the ticket; two sets alternate
// between launches.  The workspace initialisation zeroes kZeroedPrefix bytes: the status
// block and both sets.
constexpr int kDecSetWords = 1024 + 32 + 32;
constexpr int kDecReadyWords = 1024;
constexpr int kDecTicketWord = 1024 + 32;
constexpr size_t kZeroedPrefix = 256 + size_t(2) * kDecSetWords * 4;
constexpr int kRowsPerPass = 64;    // token rows handled per pass (4 MMA groups of 16)
constexpr int kGroupRows = 16;      // MMA N per group
constexpr int kMaxGroups = kRowsPerPass / kGroupRows;
constexpr int kWideRows = 192;      // routed rows per pass of the wide (many-rows) kernel
constexpr int kPlanSlice = 4096;    // routes per CTA of the multi-CTA plan (many routes)
constexpr long long kDefaultWaitLimit = 1ll << 33;  // clock cycles (~4 s at 2 GHz) before a wait gives up
constexpr float kHScale = 0.0625f;  // h is stored as FP16(h * 2^-4)
constexpr float kHUnscale = 16.0f;

// Dequantisation converts E2M1 codes with the hardware E2M1->FP16 conversion (one
// instruction per code byte, elements (2i, 2i+1) into one FP16x2 register) and multiplies
// by the FP16 block scale: E2M1 x E4M3 needs at most 6 significant bits and lies within
// [2^-10, 2688], so the product is exact in FP16.  Activations are stored in natural order.

struct WsLayout {
  size_t status, meta, counts, offsets, touched, gu_start, dn_start, route_pos, pos_tok, route_w;
  size_t ready, ticket, tasks, tasks_w, hist, x16, hs16, y, total;
  size_t front_done;  // arrival counter of the fused front, inside the zeroed status block
  size_t dec_parity;  // counter set the decode kernel with its own front uses (zeroed block)
  size_t dec_done;    // its CTA arrival counter (zeroed block)
  size_t dec_sets;    // its two counter sets, kDecSetWords words each (zeroed by the init)
  int S_gu;       // gate/up stripes per expert (ffn / 64)
  int S_dn;       // down stripes per expert (d / 128)
  int max_tasks;  // capacity of the task table
  int max_tasks_w;  // capacity of the wide kernel's task table (passes of kWideRows rows)
  int R;          // routes = T * k
};

// meta words
// META_YFMT: format of the per-route down outputs y: 0 FP32, 1 FP16(y * 2^-4) (wide kernel);
// the plan writes 0, the wide kernel's task-table kernel 1, the un-route kernel reads it.
enum { META_U = 0, META_NGU = 1, META_NDN = 2, META_MAXROWS = 3, META_WGU = 4, META_WDN = 5, META_YFMT = 6,
       META_WORDS = 16 };
constexpr float kYScale = 0.0625f;  // FP16 per-route down outputs hold y * 2^-4
constexpr float kYUnscale = 16.0f;

// One expert task as the plan writes it (16 bytes):
//   x = expert id | touched index << 16, y = first routed row (expert-major position),
//   z = rows in this pass | is_down << 16 | (expert has more than one pass) << 17,
//   w = stripe index.
struct alignas(16) TaskEntry {
  int x, y, z, w;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_shape& s) {
  WsLayout L{};
  L.R = s.T * s.k;
  L.S_gu = s.ffn / kGuRows;
  L.S_dn = s.d / kDnRows;
  // passes over all experts: at most one per touched expert plus one per 64 extra rows
  const int max_passes = s.E + (L.R + kRowsPerPass - 1) / kRowsPerPass;
  L.max_tasks = max_passes * (L.S_gu + L.S_dn);
  L.max_tasks_w = (s.E + (L.R + kWideRows - 1) / kWideRows) * (L.S_gu + L.S_dn);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.status = take(64);
  L.front_done = L.status + 64;
  L.dec_parity = L.status + 68;
  L.dec_done = L.status + 72;
  L.dec_sets = take(size_t(2) * kDecSetWords * 4);
  L.meta = take(META_WORDS * 4);
  L.counts = take(size_t(s.E) * 4);
  L.offsets = take(size_t(s.E + 1) * 4);
  L.touched = take(size_t(s.E) * 4);
  L.gu_start = take(size_t(s.E + 1) * 4);
  L.dn_start = take(size_t(s.E + 1) * 4);
  L.route_pos = take(size_t(L.R) * 4);
  L.pos_tok = take(size_t(L.R) * 4);
  L.route_w = take(size_t(L.R) * 4);
  L.ready = take(size_t(s.E + L.S_dn) * 4);  // gate/up readiness [E], down completion per stripe [S_dn]
  L.ticket = take(4);
  L.tasks = take(size_t(L.max_tasks) * sizeof(TaskEntry));
  L.tasks_w = take(size_t(L.max_tasks_w) * sizeof(TaskEntry));
  L.hist = take(size_t((L.R + kPlanSlice - 1) / kPlanSlice) * s.E * 4);  // multi-CTA plan: a histogram per slice
  L.x16 = take(size_t(s.T) * s.d * 2);
  L.hs16 = take(size_t(L.R) * s.ffn * 2);
  L.y = take(size_t(L.R) * s.d * 4);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------------
#define MOE_DEVICE __device__ __forceinline__

MOE_DEVICE uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Order-preserving map from FP32 to uint32 (larger float -> larger key), with -0
// canonicalised to +0 so that the two compare equal.
MOE_DEVICE uint32_t float_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---- mbarrier ----
MOE_DEVICE void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
MOE_DEVICE void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
MOE_DEVICE void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
MOE_DEVICE bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Programmatic dependent launch: every kernel of the library may start while the previous
// kernel in its stream is finishing; pdl_wait() blocks until that kernel has completed and
// its writes are visible, and must precede any access to the workspace, inputs or outputs.
// pdl_launch_dependents() lets the next kernel in the stream start early (it still waits).
MOE_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
MOE_DEVICE void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOE_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
MOE_DEVICE void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
MOE_DEVICE void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---- TMA (tensor) and cp.async ----
MOE_DEVICE uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEVICE void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// 2-D tile load without a cache hint (L2 evict-normal).
MOE_DEVICE void tma_load_2d_plain(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completing on `bar` through its transaction count.
MOE_DEVICE void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
MOE_DEVICE void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
MOE_DEVICE void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
MOE_DEVICE void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
MOE_DEVICE void cp_async_8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
MOE_DEVICE void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
MOE_DEVICE void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- tcgen05 (tensor memory + 5th-generation tensor core) ----
MOE_DEVICE void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
MOE_DEVICE void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// True on one lane of the converged warp (the same lane for every lane's view).
MOE_DEVICE bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 x;\n\t"
      "elect.sync x|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r));
  return r != 0;
}
MOE_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
MOE_DEVICE void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
MOE_DEVICE void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (FP16 inputs, FP32 accumulate), cta_group::1.
MOE_DEVICE void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
MOE_DEVICE void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Instruction descriptor for kind::f16: D format FP32 (bits 4-5 = 1), A and B FP16
// (bits 7-9 / 10-12 = 0), both K-major (bits 15/16 = 0), N>>3 in bits 17-22,
// M>>4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand stored in 128-byte swizzled
// atoms (8 rows x 128 bytes; 16-byte chunk c of row r stored at chunk c ^ (r & 7)).
// Start address >> 4 in bits 0-13, leading byte offset (unused for this layout) in
// 16-29, stride byte offset (distance between 8-row groups) in 32-45, descriptor
// version 1 in bits 46-47, layout type SWIZZLE_128B (2) in bits 61-63.
MOE_DEVICE uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(1u) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1u) << 46;
  d |= uint64_t(2u) << 61;
  return d;
}

// 32 lanes x 32 bits, 64 consecutive columns: thread i of the warp writes row
// (warp_quarter*32 + i) of the TMEM tile at taddr.
MOE_DEVICE void tmem_st_x64(uint32_t taddr, const uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]),
      "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]),
      "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]),
      "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]),
      "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns read back into registers.
MOE_DEVICE void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns read back into registers.
MOE_DEVICE void tmem_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// ---- NVFP4 decode helpers (hardware conversions) ----
// Four E2M1 pairs (one 32-bit word, element 2i in the low nibble of byte i) to four
// f16x2 values, low half = even element.
MOE_DEVICE void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}
// Two E4M3 bytes (low byte -> low half) to f16x2.
MOE_DEVICE uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t o;
  const uint16_t h = static_cast<uint16_t>(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o) : "h"(h));
  return o;
}
MOE_DEVICE uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t o;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(a), "r"(b));
  return o;
}
MOE_DEVICE uint32_t bcast_lo_half(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
MOE_DEVICE uint32_t bcast_hi_half(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

// ---- global-memory synchronisation ----
MOE_DEVICE uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEVICE void red_add_relaxed_gpu_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Warp-wide wait until *ctr >= target: lane 0 polls with acquire loads, giving up after
// `timeout` cycles (sets *abort_flag and MOE_DEV_TIMEOUT) or when *abort_flag is raised.
// On success the warp's later global reads, bulk copies included, are ordered after the
// writes the counter's producers released.  Returns the same value on every lane.
MOE_DEVICE bool warp_wait_counter(const uint32_t* ctr, uint32_t target, volatile int* abort_flag, int* status,
                                  long long timeout) {
  int good = 1;
  if ((threadIdx.x & 31) == 0) {
    const long long t0 = clock64();
    while (ld_acquire_u32(ctr) < target) {
      if (*abort_flag) { good = 0; break; }
      if (clock64() - t0 > timeout) {
        *abort_flag = 1;
        atomicOr(status, static_cast<int>(MOE_DEV_TIMEOUT));
        good = 0;
        break;
      }
      __nanosleep(32);
    }
  }
  __syncwarp();
  fence_proxy_async_global();
  return __shfl_sync(0xffffffffu, good, 0) != 0;
}
MOE_DEVICE uint32_t atom_add_acqrel_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
MOE_DEVICE void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier over `nthreads` threads that also returns the AND of every thread's predicate,
// so that a group of warps takes one decision together.
MOE_DEVICE bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

}  // namespace moe
