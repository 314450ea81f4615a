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
  const int m = blockIdx.y;
  const int H = p.H, K = p.K;
  const int col = (blockIdx.x * kThreads + threadIdx.x) * 8;
  // The picks, slots and per-expert row counts come from the top-k kernel,
  // complete before this grid is launched (the expert kernel lets it launch
  // only after waiting for top-k). Before waiting for the expert grid's
  // partial rows, every CTA lays out the step's units from the counts as the
  // expert kernel does (pack_unit: one block-wide exclusive scan of the rows
  // in expert order) and finds its token's partial-output rows.
  __shared__ uint16_t first_s[kMaxExperts];  // (small: this CTA shares an SM with an expert CTA)
  __shared__ uint8_t rows_s[kMaxExperts];
  __shared__ int warp_s[kThreads / 32];
  __shared__ int pos_s[kMaxTopk + 1];
  static_assert(kMaxExperts <= 4 * kThreads, "four experts per thread");
  {
    int n[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * static_cast<int>(threadIdx.x) + i;
      n[i] = e < p.E ? __ldcg(p.cnt + e) : 0;
      sum += n[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if ((threadIdx.x & 31) >= off) incl += o;
    }
    if ((threadIdx.x & 31) == 31) warp_s[threadIdx.x >> 5] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < static_cast<int>(threadIdx.x >> 5); ++w) run += warp_s[w];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * static_cast<int>(threadIdx.x) + i;
      if (e < p.E) {
        first_s[e] = static_cast<uint16_t>(run);
        rows_s[e] = static_cast<uint8_t>(n[i] < 255 ? n[i] : 255);
      }
      run += n[i];
    }
  }
  __syncthreads();
  if (static_cast<int>(threadIdx.x) <= K) {
    const int j = threadIdx.x;
    int pos = p.M * K + m;  // pick k: the shared expert's row of this token
    if (j < K) {
      const int e = __ldcg(p.ids + m * K + j), sl = __ldcg(p.slots + m * K + j);
      pos = e >= 0 && e < p.E && sl >= 0 && sl < rows_s[e] ? first_s[e] + sl : 0;
    }
    pos_s[j] = pos;
    if (blockIdx.x == 0) p.tok_pos[m * (K + 1) + j] = pos;  // diagnostics
  }
  float w[kMaxTopk];
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) w[j] = j < K ? __ldcg(p.route_w + m * K + j) : 0.0f;
  __syncthreads();
  int pos[kMaxTopk + 1];
#pragma unroll
  for (int j = 0; j <= kMaxTopk; ++j) pos[j] = j <= K ? pos_s[j] : 0;
  ptx::griddep_wait();  // the partial rows come from the expert kernel
  ptx::griddep_launch_dependents();
  if (col >= H) return;
  // picks 0 .. k-1 weighted, then the shared expert (pick k), in this order;
  // the partial rows of up to 9 picks in flight at once
  constexpr int kBatch = 9;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int j0 = 0; j0 <= kMaxTopk; j0 += kBatch) {
    if (j0 > K) break;
    float4 v[kBatch][2];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (j0 + q <= K && j0 + q <= kMaxTopk) {
        const float4* src =
            reinterpret_cast<const float4*>(p.part + static_cast<size_t>(pos[j0 + q]) * H + col);
        v[q][0] = src[0];
        v[q][1] = src[1];
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int j = j0 + q;
      if (j < K) {
        const float wj = w[j < kMaxTopk ? j : kMaxTopk - 1];
        acc[0] = fmaf(wj, v[q][0].x, acc[0]);
        acc[1] = fmaf(wj, v[q][0].y, acc[1]);
        acc[2] = fmaf(wj, v[q][0].z, acc[2]);
        acc[3] = fmaf(wj, v[q][0].w, acc[3]);
        acc[4] = fmaf(wj, v[q][1].x, acc[4]);
        acc[5] = fmaf(wj, v[q][1].y, acc[5]);
        acc[6] = fmaf(wj, v[q][1].z, acc[6]);
        acc[7] = fmaf(wj, v[q][1].w, acc[7]);
      } else if (j == K) {
        acc[0] += v[q][0].x;
        acc[1] += v[q][0].y;
        acc[2] += v[q][0].z;
        acc[3] += v[q][0].w;
        acc[4] += v[q][1].x;
        acc[5] += v[q][1].y;
        acc[6] += v[q][1].z;
        acc[7] += v[q][1].w;
      }
    }
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
