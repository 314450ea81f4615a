// Internal declarations shared by the translation units of libmoe_decode:
// the handle, the scratch layout, the kernels' parameter blocks and their
// host-side launchers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/moe_decode.h"

namespace moe {

// ---------------------------------------------------------------- limits
constexpr int kMaxTokens = 48;     // the pages' MAX_TOKENS; also the largest MMA N used
constexpr int kMaxTopk = 16;
constexpr int kMaxExperts = 512;
constexpr int kBoxRows = 16;       // TMA box height of the activation (B) operand
constexpr int kStages = 8;         // smem ring depth of the expert kernel
constexpr int kTileM = 128;        // MMA M: weight rows per tile
constexpr int kStageK = 128;       // K bytes per stage (one 128-byte swizzle row)
constexpr int kRouterWarps = 8;    // experts per router CTA (one per warp)
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // bounded waits: 1 s

// error bits in the device error word
constexpr int kErrTimeout = 1;
constexpr int kErrBounds = 2;

// counters region (int32 words at the start of the scratch)
constexpr int kCtrErr = 0;       // device error word (bit set)
constexpr int kCtrTicket = 1;    // top-k: token CTAs done
constexpr int kCtrUnits = 2;     // active experts this step (routed + 1 shared)
constexpr int kCtrRouted = 3;    // distinct routed experts this step
constexpr int kCtrWords = 64;

// One active expert of a step: what the expert kernels need to find its
// weights and its token rows.
struct ActiveExpert {
  int expert;    // 0..E-1 routed, E = the shared expert
  int pos_base;  // first row of its tokens in the gathered activation rows
  int rows;      // number of its tokens (1..M)
  int pad;
};

// ---------------------------------------------------------------- kernel params
struct SeamParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* norm_w;
  __nv_bfloat16* normed;
  uint8_t* x8;
  uint8_t* x8c;
  __nv_bfloat16* dbg_normed;
  uint8_t* dbg_x8;
  uint8_t* dbg_x8c;
  int H;
  float eps;
};

struct RouterParams {
  const __nv_bfloat16* normed;
  const __nv_bfloat16* gate_w;
  float* logit_part;  // [KS][M][E]
  int M, H, E, KS, Hs;
};

struct TopkParams {
  const float* logit_part;    // [KS][M][E]
  const float* bias;
  int* counters;
  unsigned long long* mask;   // [E]: bit m set if token m picked the expert (zero between steps)
  int* ids;                   // [M][k]
  ActiveExpert* act;          // [E + 1]
  float* route_w;             // [M][k]
  int* tok_pos;               // [M][k + 1]: gathered row of (token, pick); pick k = shared
  int* pos_tok;               // [M (k + 1)]: token of each gathered row
  int32_t* dbg_ids;
  float* dbg_w;
  float* dbg_logits;
  int M, E, K, KS;
};

struct GatherParams {
  const uint8_t* x8;
  const uint8_t* x8c;
  const int* counters;
  const ActiveExpert* act;
  const int* pos_tok;
  uint8_t* xg;     // [rows][H]
  uint4* sfb13;    // [units][H/128][32] 16-byte image rows
  int M, H, K, G;  // G = H / 128
  int units_max, rows_max;
};

// The expert kernel's parameters. PHASE 13: A = w13 rows (gate + up halves),
// B = gathered x8 rows, epilogue = SwiGLU + requant into h8 and the w2 scale
// images. PHASE 2: A = w2 rows, B = h8 rows, epilogue = fp32 partial rows.
struct ExpertParams {
  CUtensorMap tm_a;         // routed experts' weight rows (PHASE 13: 3D [expert half][row][col])
  CUtensorMap tm_a_shared;  // the shared expert's weight rows
  CUtensorMap tm_b[3];      // activation rows, boxes of 16 / 32 / 48 rows x 128 bytes
  const int* counters;
  const ActiveExpert* act;
  const uint4* sfa;         // [E + 1][tiles][G] compact weight-scale entries
  const uint8_t* sfb;       // [units][G][512] activation-scale images
  uint8_t* h8;              // PHASE 13 out: [rows][I]
  uint8_t* sfb_next;        // PHASE 13 out: [units][I/128][512] images of h8's codes
  float* part;              // PHASE 2 out: [rows][H]
  int* err;
  int E;        // routed experts (index E = shared)
  int tiles;    // tiles per expert: I/64 (PHASE 13) or H/128 (PHASE 2)
  int G;        // K stages per tile: H/128 (PHASE 13) or I/128 (PHASE 2)
  int a_rows;   // rows of one routed expert's A matrix: 2I (PHASE 13) or H (PHASE 2)
  int inter;    // I
  int hidden;   // H
  int next_G;   // PHASE 13: I/128 (groups of the w2 B operand)
  int units_max;  // capacity of the active-expert table
  int rows_max;   // capacity of the gathered rows
};

struct CombineParams {
  const float* part;
  const float* route_w;
  const int* tok_pos;
  __nv_bfloat16* out;
  int M, H, K;
};

struct SfaPackParams {
  const uint8_t* w13_s;
  const uint8_t* sw13_s;
  const uint8_t* w2_s;
  const uint8_t* sw2_s;
  uint4* sfa13;
  uint4* sfa2;
  int E, H, I;
};

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes; it must call griddep_wait()
// before it reads that kernel's outputs or writes what that kernel reads.
template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_seam(const SeamParams& p, int M, cudaStream_t s);
cudaError_t launch_router(const RouterParams& p, cudaStream_t s);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t s);
cudaError_t router_setup();
size_t router_smem_bytes(int M, int Hs);
int router_ksplit(int hidden, int experts);
cudaError_t launch_gather(const GatherParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_expert13(const ExpertParams& p, int grid, cudaStream_t s);
cudaError_t launch_expert2(const ExpertParams& p, int grid, cudaStream_t s);
cudaError_t expert_kernel_setup();
size_t expert_smem_bytes(int phase);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_sfa_pack(const SfaPackParams& p, cudaStream_t s);

}  // namespace moe
