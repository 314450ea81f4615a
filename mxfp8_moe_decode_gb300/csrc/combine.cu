// Weighted combine: out[m] = bf16(sum_j w[m, j] * y_{id(m, j)}[m] + y_shared[m]).
//
// "vllm.models.deepseek_v41.amd.mono.runner", DSV41MonoLayer._outs: the MoE
// output is out [M, HIDDEN] bf16 (the residual is a separate output, not added
// here). The routed partial rows and the shared expert's row are fp32 rows of
// the expert kernel; they are summed in a fixed order (picks 0..k-1, then the
// shared expert) in fp32 and rounded to bf16 once (round to nearest even).
//
// Grid (ceil(H / 1024), M) x 128 threads; a thread owns 8 adjacent columns.
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
  ptx::griddep_wait();  // partial rows come from the w2 kernel
  ptx::griddep_launch_dependents();
  const int m = blockIdx.y;
  const int H = p.H, K = p.K;
  const int col = (blockIdx.x * kThreads + threadIdx.x) * 8;
  if (col >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < K; ++j) {
    const int pos = p.tok_pos[m * (K + 1) + j];
    const float w = p.route_w[m * K + j];
    const float4* src = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(pos) * H + col);
    const float4 a = src[0], b = src[1];
    acc[0] = fmaf(w, a.x, acc[0]);
    acc[1] = fmaf(w, a.y, acc[1]);
    acc[2] = fmaf(w, a.z, acc[2]);
    acc[3] = fmaf(w, a.w, acc[3]);
    acc[4] = fmaf(w, b.x, acc[4]);
    acc[5] = fmaf(w, b.y, acc[5]);
    acc[6] = fmaf(w, b.z, acc[6]);
    acc[7] = fmaf(w, b.w, acc[7]);
  }
  {
    const int pos = p.tok_pos[m * (K + 1) + K];
    const float4* src = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(pos) * H + col);
    const float4 a = src[0], b = src[1];
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
  }
  __align__(16) __nv_bfloat162 o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(m) * H + col) =
      *reinterpret_cast<const uint4*>(o);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  dim3 grid((p.H / 8 + kThreads - 1) / kThreads, p.M);
  return launch_pdl(combine_kernel, grid, dim3(kThreads), 0, s, p);
}

}  // namespace moe
