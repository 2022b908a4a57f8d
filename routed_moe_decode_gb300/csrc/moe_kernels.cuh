// Kernel argument blocks and host-side launchers of the routed-MoE CUDA path.
#pragma once

#include <cuda.h>

#include "moe_common.cuh"

namespace moe {

struct PlanArgs {
  int T, E, k, S_gu, S_dn;
  const int32_t* ids;
  const float* weights;
  int* status;
  int* meta;
  int* counts;
  int* offsets;
  int* touched;
  int* gu_start;
  int* dn_start;
  int* route_pos;
  int* pos_tok;
  float* route_w;
  TaskEntry* tasks;
};

// The fused front (router + plan + FP16 hidden) for T * k up to kFrontMaxRoutes.
struct FrontArgs {
  PlanArgs plan;  // plan.ids / plan.weights receive the router's output
  int d;
  const float* logits;
  const __nv_bfloat16* hidden;
  __half* x16;
  uint32_t* ready;
  uint32_t* ticket;
  uint32_t* done;  // CTA arrival counter: zero between calls
  int tpc;         // tokens routed per CTA (one warp each), at most 32
};
constexpr int kFrontMaxRoutes = 16384;

struct PrepArgs {
  int T, d, E;
  const __nv_bfloat16* hidden;
  __half* x16;
  uint32_t* ready;
  uint32_t* ticket;
  int* status;
};

// Everything the expert kernels read besides the two tensor maps.
struct ExpertArgs {
  int T, d, F, E, k, R, S_gu, S_dn, nck_gu, nck_dn;
  float w13_ts, w2_ts;
  const uint8_t* w13_codes;
  const uint8_t* w13_scales;
  const uint8_t* w2_codes;
  const uint8_t* w2_scales;
  const int* meta;
  const int* counts;
  const int* offsets;
  const int* touched;
  const int* pos_tok;
  const int* route_pos;
  const float* route_w;
  const TaskEntry* tasks;
  const __half* x16;
  __half* hs16;
  float* y;
  uint32_t* ready;
  uint32_t* ticket;
  int* status;
  const __nv_bfloat16* residual;
  __nv_bfloat16* out;
  // optional timeline (diagnostics, off when null): per CTA kTraceRoles x kTracePerRole
  // uint64 events = event code << 56 | index << 40 | %globaltimer low 40 bits
  unsigned long long* trace;
};

constexpr int kTraceRoles = 8;
constexpr int kTracePerRole = 128;

// Launch `kernel` as a programmatic dependent of the preceding work in `stream` (it may
// begin while its predecessor finishes; the kernels order themselves with pdl_wait).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* weights,
                              cudaStream_t stream);
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
cudaError_t launch_front(FrontArgs f, cudaStream_t stream);
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t stream);
cudaError_t launch_expert_tc(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                             int num_sms, cudaStream_t stream);
cudaError_t launch_expert_mma(const ExpertArgs& a, const CUtensorMap& tm_w13, const CUtensorMap& tm_w2,
                              const CUtensorMap& tm_s13, const CUtensorMap& tm_s2, int num_sms,
                              cudaStream_t stream);
cudaError_t launch_expert_simt(const ExpertArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const ExpertArgs& a, cudaStream_t stream);
size_t expert_tc_smem_bytes();
size_t expert_mma_smem_bytes();
int encode_codes_map(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes);
// Tensor map of a [rows, row_bytes] uint8 matrix (row_bytes a multiple of 16) loaded in
// unswizzled boxes of 16 bytes x box_rows rows.
int encode_scales_map(CUtensorMap* tm, const void* base, uint32_t row_bytes, uint64_t rows, uint32_t box_rows);
// Shapes the decode (warp-MMA) kernel handles: d and ffn powers of two from 256 to 2048.
bool expert_mma_supports(int d, int F);
// Record a message for moe_last_cuda_error on the calling host thread.
void set_last_error_message(const char* msg);

}  // namespace moe
