// Router: gate GEMV, sigmoid scores, bias-adjusted top-k, normalised weights,
// and the token -> expert compaction the expert kernels run on.
//
// "vllm.models.deepseek_v41.amd.mono.runner", MonoLayerWeights: gate_w
// [E, 5120] bf16 and bias [E] f32 (e_score_correction_bias); the bf16 MoE input
// row is the router's input ("vllm.models.deepseek_v41.amd.mono.layer",
// store_normed). Scores are sigmoid(logit); the bias only shifts the choice;
// the weights are the chosen scores over their sum. Ties in the choice go to
// the lower expert index.
//
// Launch: grid (E / 8, KS) x 256 threads. CTA (b, ks) stages the normed rows'
// K-slice [ks * Hs, (ks + 1) * Hs) in shared memory and each warp reduces one
// expert row over it (fp32) into logit_part[ks][m][e]. The CTA that finishes
// last (a device-scope ticket) sums the KS partials in a fixed order and does
// the per-token top-k (one warp per token: k rounds of a warp arg-max) and
// the compaction: each active expert gets a contiguous run of gathered rows
// (experts in increasing id, tokens in increasing index), the shared expert
// last with all M tokens.
#include <cfloat>
#include <cmath>

#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kRouterWarps * 32;
constexpr int kMaxChunks = 8;  // Hs <= 2048
constexpr int kMaxPerLane = kMaxExperts / 32;

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 u = __bfloat1622float2(x[j]);
    const float2 v = __bfloat1622float2(y[j]);
    acc = fmaf(u.x, v.x, acc);
    acc = fmaf(u.y, v.y, acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kThreads) router_kernel(const RouterParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int M = p.M, H = p.H, E = p.E, K = p.K, Hs = p.Hs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.y * Hs;

  // ---- one expert row per warp: lane holds 8 columns of every 256-chunk.
  // The gate weights do not depend on the previous kernel: load them first.
  const int e = blockIdx.x * kRouterWarps + warp;
  uint4 g[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int col = c * 256 + lane * 8;
    if (col < Hs) {
      g[c] = *reinterpret_cast<const uint4*>(p.gate_w + static_cast<size_t>(e) * H + k0 + col);
    } else {
      g[c] = make_uint4(0, 0, 0, 0);
    }
  }
  ptx::griddep_wait();  // the normed rows come from the seam kernel
  ptx::griddep_launch_dependents();

  // ---- stage the K-slice of the normed rows
  uint4* xs = reinterpret_cast<uint4*>(smem);  // [M][Hs / 8]
  const int oct = Hs >> 3;
  for (int i = tid; i < M * oct; i += kThreads) {
    const int m = i / oct, o = i - m * oct;
    xs[i] = reinterpret_cast<const uint4*>(p.normed + static_cast<size_t>(m) * H + k0)[o];
  }
  __syncthreads();

  for (int m = 0; m < M; ++m) {
    float acc = 0.0f;
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int col = c * 256 + lane * 8;
      if (col < Hs) acc = dot8(g[c], xs[m * oct + (col >> 3)], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) p.logit_part[(static_cast<size_t>(blockIdx.y) * M + m) * E + e] = acc;
  }

  // ---- last CTA: top-k and compaction
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int total = gridDim.x * gridDim.y;
    is_last = (atomicAdd(&p.counters[kCtrTicket], 1) == total - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  __shared__ int ids_s[kMaxTokens * kMaxTopk];
  __shared__ unsigned long long mask_s[kMaxExperts];
  __shared__ int base_s[kMaxExperts];
  for (int i = tid; i < E; i += kThreads) mask_s[i] = 0ull;
  __syncthreads();

  // every logit of the step into shared memory (the K-slice staging is dead):
  // the KS partials summed in a fixed order, all loads in flight at once
  const int KS = gridDim.y;
  float* lg = reinterpret_cast<float*>(smem);  // [M][E]
  {
    const int n4 = M * E / 4;
    const float4* lp = reinterpret_cast<const float4*>(p.logit_part);
#pragma unroll 4
    for (int i = tid; i < n4; i += kThreads) {
      float4 a = __ldcg(lp + i);
      for (int ks = 1; ks < KS; ++ks) {
        const float4 b = __ldcg(lp + static_cast<size_t>(ks) * n4 + i);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      reinterpret_cast<float4*>(lg)[i] = a;
      if (p.dbg_logits) reinterpret_cast<float4*>(p.dbg_logits)[i] = a;
    }
  }
  __syncthreads();

  for (int m = warp; m < M; m += kRouterWarps) {
    float cv[kMaxPerLane], sv[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int ex = lane + 32 * i;
      cv[i] = -INFINITY;
      sv[i] = 0.0f;
      if (ex < E) {
        const float logit = lg[m * E + ex];
        const float s = 1.0f / (1.0f + expf(-logit));
        sv[i] = s;
        cv[i] = s + p.bias[ex];
      }
    }
    float ssum = 0.0f;
    float sel_s[kMaxTopk];
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) sel_s[j] = 0.0f;
    for (int j = 0; j < K; ++j) {
      // lane-local best: larger choice, then lower index (indices grow with i)
      float bc = -INFINITY, bs = 0.0f;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        if (cv[i] > bc) {
          bc = cv[i];
          bs = sv[i];
          bi = lane + 32 * i;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float oc = __shfl_xor_sync(0xffffffffu, bc, off);
        const float os = __shfl_xor_sync(0xffffffffu, bs, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oc > bc || (oc == bc && oi < bi)) {
          bc = oc;
          bs = os;
          bi = oi;
        }
      }
      if (bi >= E || bi < 0) {  // only on non-finite scores
        if (lane == 0) atomicOr(&p.counters[kCtrErr], kErrBounds);
        bi = 0;
      }
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (lane + 32 * i == bi) cv[i] = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kMaxTopk; ++jj)
        if (jj == j) sel_s[jj] = bs;
      ssum += bs;
      if (lane == 0) {
        ids_s[m * K + j] = bi;
        atomicOr(&mask_s[bi], 1ull << m);
      }
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) {
      if (j < K && lane == j) {
        const float w = sel_s[j] / ssum;
        p.route_w[m * K + j] = w;
        if (p.dbg_w) p.dbg_w[m * K + j] = w;
        if (p.dbg_ids) p.dbg_ids[m * K + j] = ids_s[m * K + j];
      }
    }
  }
  __syncthreads();

  // ---- active experts in increasing id: counts, run starts, unit index
  if (warp == 0) {
    const int per = E / 32;
    int cnt = 0, act = 0;
    for (int i = 0; i < per; ++i) {
      const int n = __popcll(mask_s[lane * per + i]);
      cnt += n;
      act += n > 0;
    }
    int icnt = cnt, iact = act;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, icnt, off);
      const int b = __shfl_up_sync(0xffffffffu, iact, off);
      if (lane >= off) {
        icnt += a;
        iact += b;
      }
    }
    int pos = icnt - cnt, u = iact - act;
    for (int i = 0; i < per; ++i) {
      const int ex = lane * per + i;
      const int n = __popcll(mask_s[ex]);
      base_s[ex] = pos;
      if (n > 0) {
        ActiveExpert a;
        a.expert = ex;
        a.pos_base = pos;
        a.rows = n;
        a.pad = 0;
        p.act[u] = a;
        ++u;
        pos += n;
      }
    }
    if (lane == 31) {
      ActiveExpert a;
      a.expert = E;
      a.pos_base = icnt;  // == M * K
      a.rows = M;
      a.pad = 0;
      p.act[iact] = a;
      p.counters[kCtrUnits] = iact + 1;
      p.counters[kCtrRouted] = iact;
    }
  }
  __syncthreads();
  for (int i = tid; i < M * K; i += kThreads) {
    const int m = i / K, j = i - m * K;
    const int ex = ids_s[i];
    const int rank = __popcll(mask_s[ex] & ((1ull << m) - 1ull));
    const int pos = base_s[ex] + rank;
    p.tok_pos[m * (K + 1) + j] = pos;
    p.pos_tok[pos] = m;
  }
  for (int m = tid; m < M; m += kThreads) {
    const int pos = M * K + m;
    p.tok_pos[m * (K + 1) + K] = pos;
    p.pos_tok[pos] = m;
  }
  if (tid == 0) p.counters[kCtrTicket] = 0;  // ready for the next step
}

}  // namespace

size_t router_smem_bytes(int M, int Hs, int E) {
  const size_t stage = static_cast<size_t>(M) * Hs * 2;  // normed K-slice
  const size_t logits = static_cast<size_t>(M) * E * 4;  // the tail's logits
  return stage > logits ? stage : logits;
}

cudaError_t router_setup() {
  return cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(router_smem_bytes(kMaxTokens, 2048, kMaxExperts)));
}

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  const size_t smem = router_smem_bytes(p.M, p.Hs, p.E);
  dim3 grid(p.E / kRouterWarps, p.KS);
  return launch_pdl(router_kernel, grid, dim3(kThreads), smem, s, p);
}

}  // namespace moe
