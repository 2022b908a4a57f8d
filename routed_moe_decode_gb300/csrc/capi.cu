// Host entry points of the C ABI declared in include/moe.h.
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/moe_selftest.h"
#include "moe_kernels.cuh"

namespace {

using moe::WsLayout;

thread_local char g_last_error[256] = "";

void set_error(const char* where, cudaError_t e) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
}

// Per-device launch properties, filled once per device and read-only afterwards.
struct DeviceInfo {
  int num_sms = 0;
  bool ready = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

int device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { set_error("cudaGetDevice", e); return MOE_ERR_CUDA; }
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev[dev].ready) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) { set_error("cudaDeviceGetAttribute", e); return MOE_ERR_CUDA; }
    g_dev[dev].num_sms = sms;
    g_dev[dev].ready = true;
  }
  *out = g_dev[dev];
  return MOE_OK;
}

int get_encoder(EncodeTiledFn* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  *fn = g_encode;
  return g_encode ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

namespace moe {

// 2-D uint8 tensor map over a [rows, row_bytes] code matrix: box_bytes x 64-row boxes
// with the swizzle of the same width (64 or 128 bytes), so that threads reading 16-byte
// chunks of consecutive rows hit distinct banks.
int encode_codes_map(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes) {
  EncodeTiledFn enc = nullptr;
  if (get_encoder(&enc) != MOE_OK) { snprintf(g_last_error, sizeof g_last_error, "no cuTensorMapEncodeTiled"); return MOE_ERR_CUDA; }
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  if (box_bytes != 64 && box_bytes != 128) return MOE_ERR_INVALID_ARG;
  cuuint32_t box[2] = {box_bytes, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int encode_scales_map(CUtensorMap* tm, const void* base, uint32_t row_bytes, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = nullptr;
  if (get_encoder(&enc) != MOE_OK) { snprintf(g_last_error, sizeof g_last_error, "no cuTensorMapEncodeTiled"); return MOE_ERR_CUDA; }
  if (row_bytes < 16 || row_bytes % 16 || box_rows == 0 || box_rows > 256) return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {16, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// 2-D FP16 tensor map over a row-major [rows, cols] matrix: 64-element (128-byte) wide boxes
// of box_rows rows with the 128-byte swizzle (the K-major operand layout of the MMAs).
int encode_f16_rows_map(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = nullptr;
  if (get_encoder(&enc) != MOE_OK) { snprintf(g_last_error, sizeof g_last_error, "no cuTensorMapEncodeTiled"); return MOE_ERR_CUDA; }
  if (cols % 64 || box_rows == 0 || box_rows > 256) return MOE_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

void set_last_error_message(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

}  // namespace moe

namespace {

using moe::encode_codes_map;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->d <= 0 || s->ffn <= 0 || s->E <= 0 || s->k <= 0) return MOE_ERR_INVALID_ARG;
  if (s->k > s->E) return MOE_ERR_INVALID_ARG;
  if (s->T > 65536 || s->k > 32 || s->E > 1024) return MOE_ERR_UNSUPPORTED;
  if (s->d % 128 || s->ffn % 128 || s->d < 128 || s->ffn < 128 || s->d > 16384 || s->ffn > 8192)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_ws(const moe_shape* s, const void* ws, size_t bytes) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (bytes < moe::ws_layout(*s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Experts a call plans and computes, [lo, hi): every expert for the ordinary entry points,
// one block of experts for the expert-parallel ones (the weights passed in then hold that
// block only, expert e at entry e - lo).  Passed explicitly through every internal call.
struct ExpertRange {
  int lo, hi;
};
ExpertRange all_experts(const moe_shape* s) { return ExpertRange{0, s->E}; }

moe::ExpertArgs expert_args(const moe_shape* s, const WsLayout& L, void* ws, const uint8_t* w13c,
                            const uint8_t* w13s, float w13_ts, const uint8_t* w2c, const uint8_t* w2s, float w2_ts,
                            const void* residual, void* out, ExpertRange r) {
  moe::ExpertArgs a{};
  a.T = s->T; a.d = s->d; a.F = s->ffn; a.E = s->E; a.k = s->k; a.R = L.R;
  a.S_gu = L.S_gu; a.S_dn = L.S_dn;
  a.nck_gu = s->d / moe::kChunkK;
  a.nck_dn = s->ffn / moe::kChunkK;
  a.w13_ts = w13_ts; a.w2_ts = w2_ts;
  a.w13_codes = w13c; a.w13_scales = w13s; a.w2_codes = w2c; a.w2_scales = w2s;
  a.meta = at<int>(ws, L.meta);
  a.counts = at<int>(ws, L.counts);
  a.offsets = at<int>(ws, L.offsets);
  a.touched = at<int>(ws, L.touched);
  a.pos_tok = at<int>(ws, L.pos_tok);
  a.route_pos = at<int>(ws, L.route_pos);
  a.route_w = at<float>(ws, L.route_w);
  a.tasks = at<moe::TaskEntry>(ws, L.tasks);
  a.task_cap = L.max_tasks;
  a.x16 = at<__half>(ws, L.x16);
  a.hs16 = at<__half>(ws, L.hs16);
  a.y = at<float>(ws, L.y);
  a.ready = at<uint32_t>(ws, L.ready);
  a.dn_done = a.ready + s->E;
  a.ticket = at<uint32_t>(ws, L.ticket);
  a.status = at<int>(ws, L.status);
  a.residual = static_cast<const __nv_bfloat16*>(residual);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.e_lo = r.lo;
  a.wait_limit = moe::kDefaultWaitLimit;
  a.poison_dn = -1;
  return a;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer, bad size or misaligned pointer";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape outside the implemented range";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace null, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: device-side status bits are set";
    default: return "unknown moe_status";
  }
}

const char* moe_last_cuda_error(void) { return g_last_error; }

int moe_check_shape(const moe_shape* shape) { return check_shape(shape); }

// The kernel MOE_ALGO_AUTO runs: the wide tcgen05 kernel when the routes average at least
// kWideAutoRows rows per expert (prefill chunks: each weight pass is then a real dense
// contraction), else the warp-MMA decode kernel where its shape limits allow, else the
// 16-row-group tcgen05 kernel.
constexpr int kWideAutoRows = 32;
static int auto_choice(const moe_shape* s) {
  if (static_cast<long long>(s->T) * s->k >= static_cast<long long>(kWideAutoRows) * s->E) return MOE_ALGO_WIDE;
  return moe::expert_mma_supports(s->d, s->ffn) ? MOE_ALGO_MMA : MOE_ALGO_TCGEN05;
}

int moe_auto_algo(const moe_shape* shape) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc < 0 ? rc : -rc;
  return auto_choice(shape);
}

// Un-route tasks the warp-MMA path's expert kernel runs itself for `shape` (0: the un-route is
// a kernel of its own): the decode kernel wherever it serves the shape, else the batch
// kernel for at most eight tokens.
static int fused_unroute_tasks(const moe_shape* s) {
  if (moe::expert_dec_supports(s->T, s->d, s->ffn)) return moe::expert_dec_unroute_tasks(s->T, s->d, s->ffn);
  return moe::expert_mma_unroute_tasks(s->T, moe::ws_layout(*s).S_dn);
}

int moe_unroute_fused(const moe_shape* shape, int algo) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc < 0 ? rc : -rc;
  if (algo < MOE_ALGO_AUTO || algo > MOE_ALGO_WIDE) return MOE_ERR_INVALID_ARG;
  const bool mma_ok = moe::expert_mma_supports(shape->d, shape->ffn);
  const int run = algo == MOE_ALGO_AUTO ? auto_choice(shape) : algo;
  if (run != MOE_ALGO_MMA || !mma_ok) return 0;  // MOE_ALGO_WIDE, MOE_ALGO_TCGEN05, MOE_ALGO_SIMT
  return fused_unroute_tasks(shape) > 0 ? 1 : 0;
}

size_t moe_workspace_bytes(const moe_shape* shape) {
  if (check_shape(shape) != MOE_OK) return 0;
  return moe::ws_layout(*shape).total;
}

int moe_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < 256) return MOE_ERR_WORKSPACE;
  cudaError_t e = cudaMemsetAsync(workspace, 0, std::min(workspace_bytes, moe::kZeroedPrefix), stream);
  if (e != cudaSuccess) { set_error("cudaMemsetAsync", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

int moe_route_topk(const moe_shape* shape, const float* logits, int32_t* ids, float* weights,
                   moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!logits || !ids || !weights || !aligned(logits, 16) || !aligned(ids, 4) || !aligned(weights, 4))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = moe::launch_route_topk(logits, shape->T, shape->E, shape->k, ids, weights, stream);
  if (e != cudaSuccess) { set_error("route_topk launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

static void fill_plan_args(moe::PlanArgs& a, const moe_shape* shape, const WsLayout& L, void* workspace,
                           const int32_t* ids, const float* weights, ExpertRange r) {
  a.T = shape->T; a.E = shape->E; a.k = shape->k; a.S_gu = L.S_gu; a.S_dn = L.S_dn;
  a.ids = ids; a.weights = weights;
  a.status = at<int>(workspace, L.status);
  a.meta = at<int>(workspace, L.meta);
  a.counts = at<int>(workspace, L.counts);
  a.offsets = at<int>(workspace, L.offsets);
  a.touched = at<int>(workspace, L.touched);
  a.gu_start = at<int>(workspace, L.gu_start);
  a.dn_start = at<int>(workspace, L.dn_start);
  a.route_pos = at<int>(workspace, L.route_pos);
  a.pos_tok = at<int>(workspace, L.pos_tok);
  a.route_w = at<float>(workspace, L.route_w);
  a.tasks = at<moe::TaskEntry>(workspace, L.tasks);
  a.hist = at<int>(workspace, L.hist);
  a.e_lo = r.lo;
  a.e_hi = r.hi;
  a.no_table = 0;
}

static int plan_impl(const moe_shape* shape, const int32_t* ids, const float* weights, void* workspace,
                     size_t workspace_bytes, ExpertRange r, moe_stream_t stream, bool table = true) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!ids || !weights) return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const WsLayout L = moe::ws_layout(*shape);
  moe::PlanArgs a{};
  fill_plan_args(a, shape, L, workspace, ids, weights, r);
  a.no_table = table ? 0 : 1;
  cudaError_t e = moe::launch_plan(a, stream);
  if (e != cudaSuccess) { set_error("plan launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

int moe_plan(const moe_shape* shape, const int32_t* ids, const float* weights, void* workspace,
             size_t workspace_bytes, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return plan_impl(shape, ids, weights, workspace, workspace_bytes, all_experts(shape), stream);
}

int moe_forward_prepare(const moe_shape* shape, const void* hidden, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!hidden || !aligned(hidden, 16)) return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const WsLayout L = moe::ws_layout(*shape);
  moe::PrepArgs p{};
  p.T = shape->T; p.d = shape->d; p.E = shape->E; p.S_dn = L.S_dn;
  p.hidden = static_cast<const __nv_bfloat16*>(hidden);
  p.x16 = at<__half>(workspace, L.x16);
  p.ready = at<uint32_t>(workspace, L.ready);
  p.ticket = at<uint32_t>(workspace, L.ticket);
  p.status = at<int>(workspace, L.status);
  cudaError_t e = moe::launch_prep(p, stream);
  if (e != cudaSuccess) { set_error("prep launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

// kStageExperts: the expert kernel and the kernels that prepare its input (the wide path's
// route-order gather and task table); kStagePrepOnly / kStageKernelOnly narrow it to either.
enum { kStageExperts = 1, kStageUnroute = 2, kStagePrepOnly = 4, kStageKernelOnly = 8 };

static int forward_experts_impl(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                                float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                const void* residual, void* out, void* workspace, size_t workspace_bytes, int algo,
                                unsigned long long* trace, moe_stream_t stream, ExpertRange r,
                                int stages = kStageExperts | kStageUnroute,
                                long long wait_limit = moe::kDefaultWaitLimit, int poison_dn_task = -1,
                                const float* w13_ts_e = nullptr, const float* w2_ts_e = nullptr,
                                const moe::DecFront* own_front = nullptr) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if ((stages & kStageExperts) &&
      (!w13_codes || !w13_scales || !w2_codes || !w2_scales || !aligned(w13_codes, 16) || !aligned(w13_scales, 16) ||
       !aligned(w2_codes, 16) || !aligned(w2_scales, 16)))
    return MOE_ERR_INVALID_ARG;
  if ((stages & kStageUnroute) && (!out || !aligned(out, 16) || (residual && !aligned(residual, 16))))
    return MOE_ERR_INVALID_ARG;
  if (algo < MOE_ALGO_AUTO || algo > MOE_ALGO_WIDE) return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const WsLayout L = moe::ws_layout(*shape);
  moe::ExpertArgs a = expert_args(shape, L, workspace, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales,
                                  w2_scale, residual, out, r);
  a.trace = trace;
  a.wait_limit = wait_limit;
  a.w13_ts_e = w13_ts_e;
  a.w2_ts_e = w2_ts_e;
  cudaError_t e;
  if (!(stages & kStageExperts)) {
    e = moe::launch_combine(a, stream);
    if (e != cudaSuccess) { set_error("combine launch", e); return MOE_ERR_CUDA; }
    return MOE_OK;
  }
  if (algo == MOE_ALGO_SIMT && (stages & kStagePrepOnly)) return MOE_OK;
  if (algo == MOE_ALGO_SIMT) {
    e = moe::launch_expert_simt(a, stream);
    if (e != cudaSuccess) { set_error("simt launch", e); return MOE_ERR_CUDA; }
    if (stages & kStageUnroute) {
      e = moe::launch_combine(a, stream);
      if (e != cudaSuccess) { set_error("combine launch", e); return MOE_ERR_CUDA; }
    }
    return MOE_OK;
  }
  DeviceInfo di;
  rc = device_info(&di);
  if (rc != MOE_OK) return rc;
  const bool mma_ok = moe::expert_mma_supports(shape->d, shape->ffn);
  if (algo == MOE_ALGO_MMA && !mma_ok) return MOE_ERR_UNSUPPORTED;
  const int run = algo == MOE_ALGO_AUTO ? auto_choice(shape) : algo;
  const bool use_wide = run == MOE_ALGO_WIDE;
  const bool use_mma = run == MOE_ALGO_MMA;
  // only the wide path has kernels that prepare the expert kernel's input
  if ((stages & kStagePrepOnly) && !use_wide) return MOE_OK;
  const uint32_t box = use_mma ? 128u : 64u;
  CUtensorMap tm13, tm2;
  rc = encode_codes_map(&tm13, w13_codes, static_cast<uint64_t>(shape->d) / 2,
                        static_cast<uint64_t>(r.hi - r.lo) * 2 * shape->ffn, box);
  if (rc != MOE_OK) return rc;
  rc = encode_codes_map(&tm2, w2_codes, static_cast<uint64_t>(shape->ffn) / 2,
                        static_cast<uint64_t>(r.hi - r.lo) * shape->d, box);
  if (rc != MOE_OK) return rc;
  // self test of the failure path: down task `poison_dn_task` of the table the expert kernel
  // will read is made to wait for a touched-expert index that no gate/up task publishes
  auto poison = [&](moe::TaskEntry* table, int meta_ngu_word) -> int {
    if (poison_dn_task < 0) return MOE_OK;
    int32_t meta[moe::META_WORDS];
    cudaError_t pe = cudaMemcpyAsync(meta, static_cast<char*>(workspace) + L.meta, sizeof meta, cudaMemcpyDeviceToHost,
                                     stream);
    if (pe == cudaSuccess) pe = cudaStreamSynchronize(stream);
    if (pe != cudaSuccess) { set_error("self test meta read", pe); return MOE_ERR_CUDA; }
    const int U = meta[moe::META_U], ngu = meta[meta_ngu_word], ndn = meta[meta_ngu_word + 1];
    if (poison_dn_task >= ndn || U >= shape->E) return MOE_ERR_INVALID_ARG;
    moe::TaskEntry t;
    pe = cudaMemcpyAsync(&t, table + ngu + poison_dn_task, sizeof t, cudaMemcpyDeviceToHost, stream);
    if (pe == cudaSuccess) pe = cudaStreamSynchronize(stream);
    if (pe != cudaSuccess) { set_error("self test task read", pe); return MOE_ERR_CUDA; }
    t.x = (t.x & 0xffff) | (U << 16);
    pe = cudaMemcpyAsync(table + ngu + poison_dn_task, &t, sizeof t, cudaMemcpyHostToDevice, stream);
    if (pe == cudaSuccess) pe = cudaStreamSynchronize(stream);
    if (pe != cudaSuccess) { set_error("self test task write", pe); return MOE_ERR_CUDA; }
    return MOE_OK;
  };
  if (use_mma) {
    if (!(moe::expert_dec_supports(shape->T, shape->d, shape->ffn) && moe::expert_dec_gathers(shape->T))) {
      rc = poison(at<moe::TaskEntry>(workspace, L.tasks), moe::META_NGU);
      if (rc != MOE_OK) return rc;
    }
    CUtensorMap ts13, ts2;
    rc = moe::encode_scales_map(&ts13, w13_scales, static_cast<uint32_t>(shape->d / 16),
                                static_cast<uint64_t>(r.hi - r.lo) * 2 * shape->ffn, 64);
    if (rc != MOE_OK) return rc;
    rc = moe::encode_scales_map(&ts2, w2_scales, static_cast<uint32_t>(shape->ffn / 16),
                                static_cast<uint64_t>(r.hi - r.lo) * shape->d, 64);
    if (rc != MOE_OK) return rc;
    // the decode kernel runs the un-route as trailing tasks of its own
    a.ncb = (stages & kStageUnroute) ? fused_unroute_tasks(shape) : 0;
    // up to 256 tokens: the decode kernel with the hidden rows in shared memory (all of them
    // for <= 8 tokens; per task, from its own table of 8-row passes, above)
    if (own_front) {
      // the layer in one launch: the decode kernel routes and plans for itself
      e = moe::launch_expert_dec_front(a, *own_front, tm13, tm2, ts13, ts2, di.num_sms, stream);
      if (e != cudaSuccess) { set_error("expert_dec (own front) launch", e); return MOE_ERR_CUDA; }
    } else if (moe::expert_dec_supports(shape->T, shape->d, shape->ffn)) {
      moe::ExpertArgs ad = a;
      // gathered rows: the kernel derives its 8-row passes from the plan's per-expert arrays;
      // the failure-path self test names the down task to poison instead of rewriting a table
      if (moe::expert_dec_gathers(shape->T)) ad.poison_dn = poison_dn_task;
      e = moe::launch_expert_dec(ad, tm13, tm2, ts13, ts2, di.num_sms, stream);
      if (e != cudaSuccess) { set_error("expert_dec launch", e); return MOE_ERR_CUDA; }
    } else {
      e = moe::launch_expert_mma(a, tm13, tm2, ts13, ts2, di.num_sms, stream);
      if (e != cudaSuccess) { set_error("expert_mma launch", e); return MOE_ERR_CUDA; }
    }
    if (a.ncb > 0) return MOE_OK;
  } else if (use_wide) {
    // the hidden rows in route order, in the upper half of the per-route output buffer (the
    // wide kernel's per-route outputs are FP16 and fill only the lower half)
    __half* xs = reinterpret_cast<__half*>(a.y) + static_cast<size_t>(L.R) * shape->d;
    moe::TaskEntry* tasks_w = at<moe::TaskEntry>(workspace, L.tasks_w);
    if (!(stages & kStageKernelOnly)) {
      e = moe::launch_wide_gather(a, xs, di.num_sms, stream);
      if (e != cudaSuccess) { set_error("wide gather launch", e); return MOE_ERR_CUDA; }
      // the wide kernel's own task table (passes of kWideRows rows), from the plan's arrays
      e = moe::launch_wide_plan(a, tasks_w, stream);
      if (e != cudaSuccess) { set_error("wide plan launch", e); return MOE_ERR_CUDA; }
      rc = poison(tasks_w, moe::META_WGU);
      if (rc != MOE_OK) return rc;
    }
    if (stages & kStagePrepOnly) return MOE_OK;
    moe::ExpertArgs aw = a;
    aw.tasks = tasks_w;
    aw.task_cap = L.max_tasks_w;
    // gate/up passes read their hidden rows, down passes the expert's h rows, as contiguous
    // rows in boxes of 64, 128 or 192 rows
    moe::WideActMaps am;
    for (int j = 0; j < 3; ++j) {
      const uint32_t rows = static_cast<uint32_t>(64 * (j + 1));
      rc = moe::encode_f16_rows_map(&am.xs[j], xs, static_cast<uint64_t>(shape->d), static_cast<uint64_t>(L.R), rows);
      if (rc != MOE_OK) return rc;
      rc = moe::encode_f16_rows_map(&am.h[j], a.hs16, static_cast<uint64_t>(shape->ffn), static_cast<uint64_t>(L.R), rows);
      if (rc != MOE_OK) return rc;
    }
    e = moe::launch_expert_wide(aw, tm13, tm2, am, di.num_sms, stream);
    if (e != cudaSuccess) { set_error("expert_wide launch", e); return MOE_ERR_CUDA; }
  } else {
    rc = poison(at<moe::TaskEntry>(workspace, L.tasks), moe::META_NGU);
    if (rc != MOE_OK) return rc;
    e = moe::launch_expert_tc(a, tm13, tm2, di.num_sms, stream);
    if (e != cudaSuccess) { set_error("expert_tc launch", e); return MOE_ERR_CUDA; }
  }
  if (stages & kStageUnroute) {
    e = moe::launch_combine(a, stream);
    if (e != cudaSuccess) { set_error("combine launch", e); return MOE_ERR_CUDA; }
  }
  return MOE_OK;
}

int moe_forward_expert_kernels(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                               float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                               void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, nullptr,
                              nullptr, workspace, workspace_bytes, algo, nullptr, stream, all_experts(shape),
                              kStageExperts);
}

int moe_selftest_expert_part(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                             float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                             void* workspace, size_t workspace_bytes, int algo, int part, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (part != 0 && part != 1) return MOE_ERR_INVALID_ARG;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, nullptr,
                              nullptr, workspace, workspace_bytes, algo, nullptr, stream, all_experts(shape),
                              kStageExperts | (part == 0 ? kStagePrepOnly : kStageKernelOnly));
}

int moe_forward_unroute(const moe_shape* shape, const void* residual, void* out, void* workspace,
                        size_t workspace_bytes, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, nullptr, nullptr, 0.f, nullptr, nullptr, 0.f, residual, out, workspace,
                              workspace_bytes, MOE_ALGO_AUTO, nullptr, stream, all_experts(shape), kStageUnroute);
}

int moe_forward_experts(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                        float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                        const void* residual, void* out, void* workspace, size_t workspace_bytes, int algo,
                        moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                              workspace, workspace_bytes, algo, nullptr, stream, all_experts(shape));
}

static int check_range(const moe_shape* shape, int e_begin, int e_end) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (e_begin < 0 || e_end > shape->E || e_begin >= e_end) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int moe_plan_expert_range(const moe_shape* shape, int e_begin, int e_end, const int32_t* ids, const float* weights,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  const int rc = check_range(shape, e_begin, e_end);
  if (rc != MOE_OK) return rc;
  return plan_impl(shape, ids, weights, workspace, workspace_bytes, ExpertRange{e_begin, e_end}, stream);
}

int moe_forward_experts_expert_range(const moe_shape* shape, int e_begin, int e_end, const uint8_t* w13_codes,
                                     const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes,
                                     const uint8_t* w2_scales, float w2_scale, const void* residual, void* out,
                                     void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream) {
  const int rc = check_range(shape, e_begin, e_end);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                              workspace, workspace_bytes, algo, nullptr, stream, ExpertRange{e_begin, e_end});
}

int moe_selftest_expert_trace(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                              float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                              const void* residual, void* out, void* workspace, size_t workspace_bytes,
                              unsigned long long* trace, moe_stream_t stream) {
  if (!trace) return MOE_ERR_INVALID_ARG;
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                              workspace, workspace_bytes, MOE_ALGO_AUTO, trace, stream, all_experts(shape));
}

int moe_selftest_expert_timeout(const moe_shape* shape, const uint8_t* w13_codes, const uint8_t* w13_scales,
                                float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                                const void* residual, void* out, void* workspace, size_t workspace_bytes, int algo,
                                int dn_task, long long wait_limit_cycles, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (dn_task < 0 || wait_limit_cycles <= 0 || algo == MOE_ALGO_SIMT) return MOE_ERR_INVALID_ARG;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                              workspace, workspace_bytes, algo, nullptr, stream, all_experts(shape),
                              kStageExperts | kStageUnroute, wait_limit_cycles, dn_task);
}

int moe_forward_algo(const moe_shape* shape, const void* hidden, const uint8_t* w13_codes,
                     const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes,
                     const uint8_t* w2_scales, float w2_scale, const void* residual, void* out,
                     void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!hidden || !w13_codes || !w13_scales || !w2_codes || !w2_scales || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(hidden, 16)) return MOE_ERR_INVALID_ARG;
  if (algo < MOE_ALGO_AUTO || algo > MOE_ALGO_WIDE) return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  rc = moe_forward_prepare(shape, hidden, workspace, workspace_bytes, stream);
  if (rc != MOE_OK) return rc;
  return moe_forward_experts(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                             workspace, workspace_bytes, algo, stream);
}

int moe_forward(const moe_shape* shape, const void* hidden, const uint8_t* w13_codes, const uint8_t* w13_scales,
                float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                const void* residual, void* out, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return moe_forward_algo(shape, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual,
                          out, workspace, workspace_bytes, MOE_ALGO_AUTO, stream);
}

// table = false: the plan's task table is left unwritten (the caller's expert kernel does not
// read it).
static int front_impl(const moe_shape* shape, const float* logits, const void* hidden, int32_t* ids, float* weights,
                      void* workspace, size_t workspace_bytes, ExpertRange r, moe_stream_t stream,
                      bool table = true) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (shape->T * shape->k > moe::kFrontMaxRoutes) {
    // large batches: separate router, plan and preparation kernels
    rc = moe_route_topk(shape, logits, ids, weights, stream);
    if (rc != MOE_OK) return rc;
    rc = plan_impl(shape, ids, weights, workspace, workspace_bytes, r, stream, table);
    if (rc != MOE_OK) return rc;
    return moe_forward_prepare(shape, hidden, workspace, workspace_bytes, stream);
  }
  if (!logits || !hidden || !ids || !weights || !aligned(logits, 16) || !aligned(hidden, 16) || !aligned(ids, 4) ||
      !aligned(weights, 4))
    return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const WsLayout L = moe::ws_layout(*shape);
  moe::FrontArgs f{};
  fill_plan_args(f.plan, shape, L, workspace, ids, weights, r);
  f.plan.no_table = table ? 0 : 1;
  f.d = shape->d;
  f.logits = logits;
  f.hidden = static_cast<const __nv_bfloat16*>(hidden);
  f.x16 = at<__half>(workspace, L.x16);
  f.ready = at<uint32_t>(workspace, L.ready);
  f.ticket = at<uint32_t>(workspace, L.ticket);
  f.done = at<uint32_t>(workspace, L.front_done);
  cudaError_t e = moe::launch_front(f, stream);
  if (e != cudaSuccess) { set_error("front launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

int moe_front(const moe_shape* shape, const float* logits, const void* hidden, int32_t* ids, float* weights,
              void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return front_impl(shape, logits, hidden, ids, weights, workspace, workspace_bytes, all_experts(shape), stream);
}

// Whether a whole layer runs as one launch of the decode kernel with its own front: at most
// eight tokens (un-route fused), all experts, the warp-MMA path chosen by MOE_ALGO_AUTO.
static bool use_own_front(const moe_shape* s, ExpertRange r) {
  return r.lo == 0 && r.hi == s->E && s->T >= 1 && auto_choice(s) == MOE_ALGO_MMA &&
         fused_unroute_tasks(s) > 0 &&
         moe::expert_dec_front_supports(s->T, s->d, s->ffn, s->E, s->k);
}

// Router, plan and forward of a layer: one launch when use_own_front holds, else the fused
// front (or its separate steps) followed by the expert kernels.
static int layer_steps(const moe_shape* shape, const float* logits, const void* hidden, const uint8_t* w13_codes,
                       const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales,
                       float w2_scale, const void* residual, void* out, int32_t* ids, float* weights,
                       void* workspace, size_t workspace_bytes, ExpertRange r, moe_stream_t stream,
                       const float* w13_ts_e = nullptr, const float* w2_ts_e = nullptr,
                       unsigned long long* trace = nullptr) {
  if (use_own_front(shape, r)) {
    if (!logits || !hidden || !ids || !weights || !aligned(logits, 16) || !aligned(hidden, 16) || !aligned(ids, 4) ||
        !aligned(weights, 4))
      return MOE_ERR_INVALID_ARG;
    const int rc = check_ws(shape, workspace, workspace_bytes);
    if (rc != MOE_OK) return rc;
    const WsLayout L = moe::ws_layout(*shape);
    moe::DecFront f{};
    f.logits = logits;
    f.hidden = static_cast<const __nv_bfloat16*>(hidden);
    f.ids = ids;
    f.weights = weights;
    f.meta = at<int>(workspace, L.meta);
    f.counts = at<int>(workspace, L.counts);
    f.offsets = at<int>(workspace, L.offsets);
    f.touched = at<int>(workspace, L.touched);
    f.gu_start = at<int>(workspace, L.gu_start);
    f.dn_start = at<int>(workspace, L.dn_start);
    f.route_pos = at<int>(workspace, L.route_pos);
    f.pos_tok = at<int>(workspace, L.pos_tok);
    f.route_w = at<float>(workspace, L.route_w);
    f.tasks = at<moe::TaskEntry>(workspace, L.tasks);
    f.x16 = at<__half>(workspace, L.x16);
    f.sets = at<uint32_t>(workspace, L.dec_sets);
    f.parity = at<uint32_t>(workspace, L.dec_parity);
    f.done = at<uint32_t>(workspace, L.dec_done);
    return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual,
                                out, workspace, workspace_bytes, MOE_ALGO_AUTO, trace, stream, r,
                                kStageExperts | kStageUnroute, moe::kDefaultWaitLimit, -1, w13_ts_e, w2_ts_e, &f);
  }
  // the gathered decode kernel derives its passes from the plan's per-expert arrays and the wide
  // kernel builds its own table: neither reads the plan's task table
  const int run = auto_choice(shape);
  const bool table = !((run == MOE_ALGO_MMA && moe::expert_dec_supports(shape->T, shape->d, shape->ffn) &&
                        moe::expert_dec_gathers(shape->T)) ||
                       run == MOE_ALGO_WIDE);
  const int rc = front_impl(shape, logits, hidden, ids, weights, workspace, workspace_bytes, r, stream, table);
  if (rc != MOE_OK) return rc;
  return forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual, out,
                              workspace, workspace_bytes, MOE_ALGO_AUTO, trace, stream, r,
                              kStageExperts | kStageUnroute, moe::kDefaultWaitLimit, -1, w13_ts_e, w2_ts_e);
}

static int layer_impl(const moe_shape* shape, const float* logits, const void* hidden, const uint8_t* w13_codes,
                      const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales,
                      float w2_scale, const void* residual, void* out, int32_t* ids, float* weights, void* workspace,
                      size_t workspace_bytes, ExpertRange r, moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales || !out) return MOE_ERR_INVALID_ARG;
  return layer_steps(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale,
                     residual, out, ids, weights, workspace, workspace_bytes, r, stream);
}

int moe_layer(const moe_shape* shape, const float* logits, const void* hidden, const uint8_t* w13_codes,
              const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales,
              float w2_scale, const void* residual, void* out, int32_t* ids, float* weights, void* workspace,
              size_t workspace_bytes, moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  return layer_impl(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual,
                    out, ids, weights, workspace, workspace_bytes, all_experts(shape), stream);
}

int moe_layer_expert_range(const moe_shape* shape, int e_begin, int e_end, const float* logits, const void* hidden,
                           const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                           const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale, const void* residual,
                           void* out, int32_t* ids, float* weights, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
  const int rc = check_range(shape, e_begin, e_end);
  if (rc != MOE_OK) return rc;
  return layer_impl(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual,
                    out, ids, weights, workspace, workspace_bytes, ExpertRange{e_begin, e_end}, stream);
}

int moe_router_logits(const moe_shape* shape, const void* hidden, const void* router_w, float* logits,
                      moe_stream_t stream) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!hidden || !router_w || !logits || !aligned(hidden, 16) || !aligned(router_w, 16) || !aligned(logits, 4))
    return MOE_ERR_INVALID_ARG;
  if (!moe::router_gemv_supports(shape->T, shape->d, shape->E)) return MOE_ERR_UNSUPPORTED;
  const cudaError_t e = moe::launch_router_gemv(static_cast<const __nv_bfloat16*>(hidden),
                                                static_cast<const __nv_bfloat16*>(router_w), logits, shape->T,
                                                shape->d, shape->E, stream);
  if (e != cudaSuccess) { set_error("router launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

int moe_layer_from_hidden(const moe_shape* shape, const void* hidden, const void* router_w, float* logits,
                          const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                          const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale, const void* residual,
                          void* out, int32_t* ids, float* weights, void* workspace, size_t workspace_bytes,
                          moe_stream_t stream) {
  const int rc = moe_router_logits(shape, hidden, router_w, logits, stream);
  if (rc != MOE_OK) return rc;
  return layer_impl(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, residual,
                    out, ids, weights, workspace, workspace_bytes, all_experts(shape), stream);
}

int moe_forward_unroute_gated(const moe_shape* shape, int G, const void* residual, const float* inject_logits,
                              const void* norm_weight, float eps, void* residual_out, void* normed_out,
                              void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (G < 1 || !(eps >= 0.f) || !(eps < 1e30f)) return MOE_ERR_INVALID_ARG;
  if (!moe::gated_unroute_supports(shape->d, G)) return MOE_ERR_UNSUPPORTED;
  if (shape->T == 0) return MOE_OK;
  if (!residual || !inject_logits || !norm_weight || !residual_out || !normed_out || !aligned(residual, 16) ||
      !aligned(norm_weight, 16) || !aligned(residual_out, 16) || !aligned(normed_out, 16) || !aligned(inject_logits, 4))
    return MOE_ERR_INVALID_ARG;
  rc = check_ws(shape, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  const WsLayout L = moe::ws_layout(*shape);
  const moe::ExpertArgs a = expert_args(shape, L, workspace, nullptr, nullptr, 0.f, nullptr, nullptr, 0.f, nullptr,
                                        nullptr, all_experts(shape));
  const cudaError_t e = moe::launch_gated_unroute(
      a, G, static_cast<const __nv_bfloat16*>(residual), inject_logits, static_cast<const __nv_bfloat16*>(norm_weight),
      eps, static_cast<__nv_bfloat16*>(residual_out), static_cast<__nv_bfloat16*>(normed_out), stream);
  if (e != cudaSuccess) { set_error("gated un-route launch", e); return MOE_ERR_CUDA; }
  return MOE_OK;
}

int moe_layer_gated(const moe_shape* shape, int G, const float* logits, const void* hidden, const uint8_t* w13_codes,
                    const uint8_t* w13_scales, float w13_scale, const uint8_t* w2_codes, const uint8_t* w2_scales,
                    float w2_scale, const void* residual, const float* inject_logits, const void* norm_weight,
                    float eps, void* residual_out, void* normed_out, int32_t* ids, float* weights, void* workspace,
                    size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (G < 1 || !(eps >= 0.f) || !(eps < 1e30f)) return MOE_ERR_INVALID_ARG;
  if (!moe::gated_unroute_supports(shape->d, G)) return MOE_ERR_UNSUPPORTED;
  if (shape->T == 0) return MOE_OK;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales) return MOE_ERR_INVALID_ARG;
  rc = front_impl(shape, logits, hidden, ids, weights, workspace, workspace_bytes, all_experts(shape), stream);
  if (rc != MOE_OK) return rc;
  rc = forward_experts_impl(shape, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale, nullptr, nullptr,
                            workspace, workspace_bytes, MOE_ALGO_AUTO, nullptr, stream, all_experts(shape),
                            kStageExperts);
  if (rc != MOE_OK) return rc;
  return moe_forward_unroute_gated(shape, G, residual, inject_logits, norm_weight, eps, residual_out, normed_out,
                                   workspace, workspace_bytes, stream);
}

int moe_layer_expert_scales(const moe_shape* shape, const float* logits, const void* hidden,
                            const uint8_t* w13_codes, const uint8_t* w13_scales, const float* w13_scales_e,
                            const uint8_t* w2_codes, const uint8_t* w2_scales, const float* w2_scales_e,
                            const void* residual, void* out, int32_t* ids, float* weights, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales || !out || !w13_scales_e || !w2_scales_e ||
      !aligned(w13_scales_e, 4) || !aligned(w2_scales_e, 4))
    return MOE_ERR_INVALID_ARG;
  return layer_steps(shape, logits, hidden, w13_codes, w13_scales, 1.f, w2_codes, w2_scales, 1.f, residual, out, ids,
                     weights, workspace, workspace_bytes, all_experts(shape), stream, w13_scales_e, w2_scales_e);
}

int moe_selftest_layer_trace(const moe_shape* shape, const float* logits, const void* hidden,
                             const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                             const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale, const void* residual,
                             void* out, int32_t* ids, float* weights, void* workspace, size_t workspace_bytes,
                             unsigned long long* trace, moe_stream_t stream) {
  if (!trace) return MOE_ERR_INVALID_ARG;
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (shape->T == 0) return MOE_OK;
  if (!w13_codes || !w13_scales || !w2_codes || !w2_scales || !out) return MOE_ERR_INVALID_ARG;
  return layer_steps(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale,
                     residual, out, ids, weights, workspace, workspace_bytes, all_experts(shape), stream, nullptr,
                     nullptr, trace);
}

int moe_layer_launches(const moe_shape* shape) {
  const int rc = check_shape(shape);
  if (rc != MOE_OK) return rc < 0 ? rc : -rc;
  if (shape->T == 0) return 0;
  if (use_own_front(shape, all_experts(shape))) return 1;
  const long long R = static_cast<long long>(shape->T) * shape->k;
  // router + plan + FP16 staging: one fused launch, or router, plan (three launches above
  // the one-CTA plan's limit) and staging
  const int front = R <= moe::kFrontMaxRoutes ? 1 : 2 + (R <= 16 * 1024 ? 1 : 3);
  const int algo = auto_choice(shape);
  int experts = 1;
  if (algo == MOE_ALGO_WIDE) experts = 3;  // route-order gather + task-table kernel + wide kernel
  const int unroute =
      (algo == MOE_ALGO_MMA && fused_unroute_tasks(shape) > 0) ? 0 : 1;
  return front + experts + unroute;
}

int moe_read_device_status(const void* workspace, int clear, uint32_t* status_bits, moe_stream_t stream) {
  if (!workspace || !status_bits || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) { set_error("status read", e); return MOE_ERR_CUDA; }
  if (clear) {
    e = cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof v, stream);
    if (e != cudaSuccess) { set_error("status clear", e); return MOE_ERR_CUDA; }
  }
  *status_bits = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

int moe_plan_summary(const moe_shape* shape, const void* workspace, int32_t* touched_experts, int32_t* max_rows,
                     moe_stream_t stream) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (!workspace || !aligned(workspace, 256) || !touched_experts || !max_rows) return MOE_ERR_INVALID_ARG;
  const WsLayout L = moe::ws_layout(*shape);
  int32_t meta[moe::META_WORDS];
  cudaError_t e = cudaMemcpyAsync(meta, static_cast<const char*>(workspace) + L.meta, sizeof meta,
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) { set_error("plan summary", e); return MOE_ERR_CUDA; }
  *touched_experts = meta[moe::META_U];
  *max_rows = meta[moe::META_MAXROWS];
  return MOE_OK;
}

int moe_plan_views(const moe_shape* shape, void* workspace, int32_t** counts, int32_t** offsets, int32_t** touched,
                   int32_t** route_pos, int32_t** pos_token) {
  int rc = check_shape(shape);
  if (rc != MOE_OK) return rc;
  if (!workspace || !counts || !offsets || !touched || !route_pos || !pos_token) return MOE_ERR_INVALID_ARG;
  const WsLayout L = moe::ws_layout(*shape);
  *counts = at<int32_t>(workspace, L.counts);
  *offsets = at<int32_t>(workspace, L.offsets);
  *touched = at<int32_t>(workspace, L.touched);
  *route_pos = at<int32_t>(workspace, L.route_pos);
  *pos_token = at<int32_t>(workspace, L.pos_tok);
  return MOE_OK;
}

}  // extern "C"
