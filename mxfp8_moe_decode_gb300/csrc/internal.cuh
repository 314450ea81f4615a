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
constexpr int kCtrUnits = 2;     // active experts this step (routed + 1 shared)
constexpr int kCtrRouted = 3;    // distinct routed experts this step
constexpr int kCtrTasks = 4;     // expert kernel: next task to hand out (zeroed by the router)
constexpr int kCtrWords = 64;
constexpr int kW2SplitMaxM = 4;  // steps of at most this many tokens split their last w2 tiles
constexpr int kPrefetchMaxM = 8;  // steps of at most this many tokens prefetch the shared expert
constexpr int kSeamFuseMaxM = 4;  // steps of at most this many tokens run the seam in the router
// Steps of at most kPickPrefetchMaxM tokens with E4M3 routed experts prefetch
// the first kPickPrefetchStages K stages of every w13 tile of their picks into
// L2 as soon as the top-k kernel has chosen them (on one GB300: M=1 -0.5 us,
// the 384-expert layer at M=1 -1.2 us; 3 stages about the same, 12 slower)
constexpr int kPickPrefetchMaxM = 4;
constexpr int kPickPrefetchStages = 6;

// One active expert of a step: what the expert kernels need to find its
// weights and its token rows.
struct ActiveExpert {
  int expert;    // 0..E-1 routed, E = the shared expert
  int pos_base;  // first of its partial-output rows
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
  uint8_t* xpan_shared;  // [H/128] x panels of the shared expert (row = token), or null
  int H;
  float eps;
};

struct RouterParams {
  const __nv_bfloat16* normed;  // [M][H] the seam's rows (read when x is null)
  const __nv_bfloat16* gate_w;
  float* logit_part;  // [KS][M][E]
  // Fused seam (M <= kSeamFuseMaxM, Hs a multiple of 32): every CTA makes its
  // K-slice of the normed rows from x itself; the CTAs of expert block 0 also
  // write the slice's MXFP8 bytes, codes, shared-expert panel rows and the
  // debug copies (null: not wanted).
  const __nv_bfloat16* x;       // [M][H] hidden rows, or null: no fusion
  const __nv_bfloat16* norm_w;  // [H]
  uint8_t* x8;                  // [M][H]
  uint8_t* x8c;                 // [M][H/32]
  uint8_t* xpan_shared;         // [H/128] x panels of the shared expert
  __nv_bfloat16* dbg_normed;
  uint8_t* dbg_x8;
  uint8_t* dbg_x8c;
  float eps;
  // Byte ranges (16-byte aligned, sizes multiples of 16, or null) that the
  // CTAs prefetch into L2 (evict-last) while the routing runs: the shared
  // expert's weights, which the expert kernel reads whatever the routing.
  // Prefetches are issued at a limited rate per SM: each CTA takes a share.
  const uint8_t* pf_ptr[2];
  uint64_t pf_bytes[2];
  // int arrays (or null) that CTA (0, 0) sets to zero once the previous
  // kernel is complete -- the previous step's readers of the per-expert row
  // counts, the readiness counts and the task counter are done by then, and
  // this step's top-k kernel runs after this grid
  int* clear[4];
  int clear_n[4];
  float* zero_rows;  // floats all CTAs set to zero (the partial rows that w2 halves add into), or null
  size_t zero_n;
  int* err;          // device error word: a bulk-copy wait that gives up sets kErrTimeout
  int M, H, E, KS, Hs;
};

// Activation panels. The B operand of one K stage of one expert is stored as
// the exact shared-memory image the MMA reads, behind its scale image, so that
// one contiguous bulk copy stages both:
//   bytes [0, 512): 32 rows x 16 bytes, row r holding in its 32-bit cell j the
//     four E8M0 codes of the stage's K blocks for the expert's row 32 j + r;
//   bytes [512, 1024): unused (the rows start 1024-aligned);
//   bytes [1024, 1024 + nt * 128): the rows (nt = rows rounded up to 16), 128
//     bytes of K each, 128-byte swizzled: the 16-byte chunk c of row r sits at
//     chunk c ^ (r % 8) of that row (the layout a 128B-swizzle TMA box writes).
// Nothing in a panel depends on the final row count, so rows can be written as
// soon as their position is known. Panels sit at a fixed pitch. Rows past an
// expert's token count hold stale finite data: an MMA output column depends on
// its own row alone and is never read.
constexpr uint32_t kPanelRows = 1024;
constexpr uint32_t kPanelPitch = kPanelRows + kMaxTokens * 128;
static_assert(kPanelPitch % 16 == 0, "bulk copies need 16-byte multiples");

__host__ __device__ __forceinline__ uint32_t panel_byte(int r, int k) {
  return kPanelRows + static_cast<uint32_t>(r) * 128u +
         ((static_cast<uint32_t>(k >> 4) ^ (r & 7)) << 4) + static_cast<uint32_t>(k & 15);
}
__host__ __device__ __forceinline__ uint32_t panel_code_byte(int r) {
  return static_cast<uint32_t>(r & 31) * 16u + static_cast<uint32_t>(r >> 5) * 4u;
}

struct TopkParams {
  const float* logit_part;    // [KS][M][E]
  const float* bias;
  int* counters;
  int* cnt;                   // [E]: rows taken per expert this step (zero before the step)
  int* ids;                   // [M][k]
  int* slots;                 // [M][k]: the token's row among the expert's rows
  float* route_w;             // [M][k]
  const uint8_t* x8;          // [M][H] the seam's MXFP8 rows and codes [M][H/32]
  const uint8_t* x8c;
  uint8_t* xpan;              // [E + 1][H/128] x panels by expert id (or null: no panels);
                              // the routed ones (at M > 1; the seam writes the shared one)
  int* picks_early;           // small steps: [0] tokens whose picks are published (zeroed by
                              // the router), then the picks [M][k]; else null
  int32_t* dbg_ids;
  float* dbg_w;
  float* dbg_logits;
  int M, E, K, KS, H;
};

// The grouped-expert kernel's parameters. One launch runs both GEMM phases:
// first every (unit, w13 tile) task, then every (unit, w2 tile) task.
//  w13 task = (unit, 64 intermediate columns): A = the 64 gate rows over the
//    matching 64 up rows, B = the expert's x panels (MXFP8 token rows), K = H; epilogue:
//    SwiGLU + requant into h8 rows and the w2 activation-scale images.
//  w2 task = (unit, 128 hidden rows): A = w2 rows, B = the unit's h8 rows,
//    K = I; epilogue: fp32 rows of y for the combine. It waits until all
//    w13 tiles of its unit are done (the unit's readiness counter).
struct ExpertParams {
  CUtensorMap tm_w13;         // routed w13 as [2E halves][I rows][H] (3D)
  CUtensorMap tm_w13_shared;  // shared w13 as [2 halves][I][H]
  CUtensorMap tm_w2;          // routed w2 as [E H rows][I]
  CUtensorMap tm_w2_shared;   // shared w2 [H][I]
  const int* cnt;             // [E]: each routed expert's rows this step (top-k's counts)
  int* counters;              // the step's unit counts go to kCtrUnits / kCtrRouted (diagnostics)
  ActiveExpert* act;          // [units] the unit table, written by CTA 0 (diagnostics)
  const uint4* sfa13;         // [E + 1][I/64][H/128] compact weight-scale entries
  const uint4* sfa2;          // [E + 1][H/128][I/128]
  const uint4* img13;         // MXFP4 routed experts: [E][I/64][H/128][32] per-row scale
  const uint4* img2;          // images ([E][H/128][I/128][32]), else null
  int fp4;                    // routed experts are E2M1 with per-row scales
  const uint8_t* xpan;        // [E + 1][H/128] x panels by expert id (the routed ones written by
                              // the top-k kernel, the shared one -- rows = tokens -- by the seam;
                              // at M = 1 every unit reads the shared one: its single row is token 0)
  uint8_t* hpan;              // [units][I/128] h panels by unit (written by the w13 epilogue)
  float* part;                // [rows][H]
  int* ready;                 // [units_max]: finished w13 tiles per unit (zeroed by the router)
  int* task_ctr;              // next task id to hand out (zeroed by the router)
  int* err;
  int E;                      // routed experts (index E = shared)
  int inter, hidden;
  int t13, g13;               // w13: tiles per unit (I/64), K stages (H/128)
  int t2, g2;                 // w2: tiles per unit (H/128), K stages (I/128)
  int split_tiles;            // the step's last w2 tiles (at most this many) run as two K-halves
                              // added into zeroed rows (0: none; only steps of <= kW2SplitMaxM
                              // tokens, g2 >= 4)
  int units_max;              // capacity of the active-expert table
  int rows_max;               // capacity of the partial-output rows
  int withhold_unit;          // test hook: this unit's w13 tiles never report ready, so its
                              // w2 tasks' bounded waits expire (-1: off)
  const int* picks_early;     // small steps: the top-k kernel's picks as soon as they are known
                              // (TopkParams::picks_early); the idle epilogue warps prefetch the
                              // picked experts' first w13 stages into L2 (else null)
  int M, K;                   // this step's tokens, picks per token
};

// The step's units, as every expert CTA and every combine CTA derives them
// from the per-expert row counts: the routed experts with rows in increasing
// id, each owning a run of partial-output rows that starts at the sum of the
// rows of the experts before it, then the shared expert with the M tokens at
// rows M k .. M k + M - 1. Packed unit entry: expert id (bits 0-9), rows
// (10-15), first row (16-31).
__host__ __device__ __forceinline__ uint32_t pack_unit(int e, int rows, int first) {
  return static_cast<uint32_t>(e) | (static_cast<uint32_t>(rows) << 10) |
         (static_cast<uint32_t>(first) << 16);
}
static_assert(kMaxExperts < 1024 && kMaxTokens < 64 && kMaxTokens * (kMaxTopk + 1) < 65536,
              "unit entries fit 32 bits");

struct CombineParams {
  const float* part;
  const float* route_w;       // [M][k]
  const int* ids;             // [M][k] picked experts
  const int* slots;           // [M][k] the token's row among the expert's rows
  const int* cnt;             // [E] each routed expert's rows this step
  int* tok_pos;               // [M][k + 1] partial-output row of (token, pick), written for
                              // diagnostics (pick k = the shared expert)
  __nv_bfloat16* out;
  int M, H, K, E;
};

struct SfaPackParams {
  const uint8_t* w13_s;
  const uint8_t* sw13_s;
  const uint8_t* w2_s;
  const uint8_t* sw2_s;
  uint4* sfa13;
  uint4* sfa2;
  uint4* img13;  // MXFP4 routed experts: per-row scale images (else null)
  uint4* img2;
  int fp4;       // routed w13_s / w2_s hold per-row codes: only the shared
                 // expert gets compact 32 x 32 entries
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
cudaError_t launch_experts(const ExpertParams& p, int grid, cudaStream_t s);
cudaError_t expert_kernel_setup();
// CTAs of the expert kernel (routed format: fp4 = 1 for E2M1) one SM can hold
cudaError_t expert_occupancy(int fp4, int* per_sm);
size_t expert_smem_bytes(int phase);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_sfa_pack(const SfaPackParams& p, cudaStream_t s);

}  // namespace moe
