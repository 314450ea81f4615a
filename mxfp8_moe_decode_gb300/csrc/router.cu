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
// router_kernel: grid (E / 8, KS) x 256 threads. CTA (b, ks) holds the gate
// rows of experts 8b .. 8b+7 restricted to the K-slice [ks Hs, (ks + 1) Hs)
// (loaded before the grid-dependency wait: they do not depend on the seam) and
// bulk-copies the normed rows' K-slice into shared memory; warp w reduces
// expert 8b + w over it for every token at once (each lane keeps one fp32 sum
// per token over its 8-column slices), then one butterfly reduce-scatter
// across the warp's lanes yields logit_part[ks][m][e].
//
// topk_kernel: one CTA per token. A thread per expert sums the KS partial
// logits in a fixed order (all partial loads issued before the sum), takes
// sigmoid and score + bias; warp 0 picks the k largest choices with 64-bit
// keys (order-preserving bits of the choice, then the inverted expert index,
// so equal choices go to the lower index), one warp-wide max per pick, and
// sets the token's bit in each picked expert's mask. The last token CTA (a
// device-scope ticket) compacts: active experts in increasing id each get a
// contiguous run of gathered rows (tokens in increasing index), the shared
// expert last with all M tokens; it clears the masks and the ticket.
#include <cfloat>
#include <cmath>

#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = kRouterWarps * 32;
constexpr int kMaxHs = 1536;                    // K-slice columns per router CTA
constexpr int kMaxChunks = kMaxHs / 256;        // 256-column chunks (8 per lane)
constexpr int kMaxPerLane = kMaxExperts / 32;
constexpr int kSlots = 64;                      // token sums per lane (>= kMaxTokens)
constexpr int kMaxKsplit = 16;                  // K-slices of the router GEMV
constexpr int kTopkThreads = 256;

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16);
  f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16);
  f[7] = __uint_as_float(u.w & 0xffff0000u);
}

// One step of the butterfly reduce-scatter: lanes whose `off` bit is clear keep
// the lower half of the N live slots, the others the upper half; each adds the
// partner's copy of the half it keeps.
template <int N>
__device__ __forceinline__ void reduce_scatter_step(float* v, int off, int lane) {
  const bool hi = (lane & off) != 0;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float send = hi ? v[i] : v[i + N / 2];
    const float keep = hi ? v[i + N / 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
  }
}

__global__ void __launch_bounds__(kThreads) router_kernel(const RouterParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;  // completion of the bulk copies into smem
  const int M = p.M, H = p.H, E = p.E, Hs = p.Hs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.y * Hs;
  const int oct = Hs >> 3;  // 16-byte pieces of one row slice
  const uint4* xs = reinterpret_cast<const uint4*>(smem);                      // [M][oct]
  uint4* gs = reinterpret_cast<uint4*>(smem) + static_cast<size_t>(M) * oct;  // [8][oct]
  const int e = blockIdx.x * kRouterWarps + warp;

  // ---- gate rows first: they do not depend on the previous kernel
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.gate_w + static_cast<size_t>(e) * H + k0);
    uint4 g[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int i = c * 32 + lane;
      g[c] = i < oct ? src[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int i = c * 32 + lane;
      if (i < oct) gs[warp * oct + i] = g[c];
    }
  }
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  ptx::griddep_wait();  // the normed rows come from the seam kernel
  ptx::griddep_launch_dependents();
  __syncthreads();

  // ---- the K-slice of every normed row: one bulk copy per row, all in flight
  if (tid == 0) {
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_arrive_expect_tx(b, static_cast<uint32_t>(M) * Hs * 2);
    for (int m = 0; m < M; ++m)
      ptx::bulk_load(ptx::smem_u32(smem + static_cast<size_t>(m) * Hs * 2),
                     p.normed + static_cast<size_t>(m) * H + k0, Hs * 2, b);
  }
  int never = 0;
  ptx::mbar_wait(ptx::smem_u32(&bar), 0, &never, kWaitLimitNs);

  // ---- every token's sum over this lane's 8-column slices
  float acc[kSlots];
#pragma unroll
  for (int m = 0; m < kSlots; ++m) acc[m] = 0.0f;
#pragma unroll 1
  for (int c = 0; c < kMaxChunks; ++c) {
    const int i = c * 32 + lane;
    if (i < oct) {
      float gf[8];
      unpack_bf16x8(gs[warp * oct + i], gf);
#pragma unroll
      for (int m = 0; m < kMaxTokens; ++m) {
        if (m < M) {
          float xf[8];
          unpack_bf16x8(xs[m * oct + i], xf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[m] = fmaf(gf[j], xf[j], acc[m]);
        }
      }
    }
  }

  // ---- across the warp: a few tokens directly, many by reduce-scatter
  float* out = p.logit_part + static_cast<size_t>(blockIdx.y) * M * E + e;
  if (M <= 4) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      if (m < M) {
        float v = acc[m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) out[static_cast<size_t>(m) * E] = v;
      }
    }
  } else {
    reduce_scatter_step<64>(acc, 16, lane);
    reduce_scatter_step<32>(acc, 8, lane);
    reduce_scatter_step<16>(acc, 4, lane);
    reduce_scatter_step<8>(acc, 2, lane);
    reduce_scatter_step<4>(acc, 1, lane);
    const int m0 = ((lane >> 4) & 1) * 32 + ((lane >> 3) & 1) * 16 + ((lane >> 2) & 1) * 8 +
                   ((lane >> 1) & 1) * 4 + (lane & 1) * 2;
    if (m0 < M) out[static_cast<size_t>(m0) * E] = acc[0];
    if (m0 + 1 < M) out[static_cast<size_t>(m0 + 1) * E] = acc[1];
  }
}

// Order-preserving key of a choice value with its expert index: larger choice
// first, then the lower index.
__device__ __forceinline__ unsigned long long choice_key(float c, int idx) {
  uint32_t b = __float_as_uint(c);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | static_cast<uint32_t>(0x7fffffff - idx);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkParams p) {
  ptx::griddep_wait();  // partial logits come from the router kernel
  ptx::griddep_launch_dependents();
  const int M = p.M, E = p.E, K = p.K, KS = p.KS;
  const int m = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ unsigned long long key_s[kMaxExperts];
  __shared__ float s_s[kMaxExperts];
  __shared__ int is_last;

  // ---- one thread per expert: the KS partials (all loads in flight), then
  // their sum in a fixed order, the score and the choice key
  for (int ex = tid; ex < E; ex += kTopkThreads) {
    float part[kMaxKsplit];
#pragma unroll
    for (int ks = 0; ks < kMaxKsplit; ++ks)
      part[ks] = ks < KS ? __ldcg(p.logit_part + (static_cast<size_t>(ks) * M + m) * E + ex) : 0.0f;
    float logit = 0.0f;
#pragma unroll
    for (int ks = 0; ks < kMaxKsplit; ++ks)
      if (ks < KS) logit += part[ks];
    const float s = 1.0f / (1.0f + expf(-logit));
    s_s[ex] = s;
    key_s[ex] = choice_key(s + p.bias[ex], ex);
    if (p.dbg_logits) p.dbg_logits[static_cast<size_t>(m) * E + ex] = logit;
  }
  __syncthreads();

  // ---- warp 0: the k largest keys, one warp-wide max per pick
  if (warp == 0) {
    unsigned long long key[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) key[i] = lane + 32 * i < E ? key_s[lane + 32 * i] : 0ull;
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) best = key[i] > best ? key[i] : best;
    float ssum = 0.0f, my_s = 0.0f;
    int my_id = 0;
    for (int j = 0; j < K; ++j) {
      unsigned long long w = best;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, w, off);
        w = o > w ? o : w;
      }
      int ex = 0x7fffffff - static_cast<int>(static_cast<uint32_t>(w));
      if (w == 0ull || ex < 0 || ex >= E) {  // only with non-finite scores
        if (lane == 0) atomicOr(&p.counters[kCtrErr], kErrBounds);
        ex = 0;
      }
      if (lane == (ex & 31)) {
        const int slot = ex >> 5;
        best = 0ull;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          if (i == slot) key[i] = 0ull;
          best = key[i] > best ? key[i] : best;
        }
      }
      const float s = s_s[ex];
      ssum += s;
      if (lane == j) {
        my_s = s;
        my_id = ex;
      }
      if (lane == 0) atomicOr(p.mask + ex, 1ull << m);
    }
    if (lane < K) {
      const float wgt = my_s / ssum;
      p.route_w[m * K + lane] = wgt;
      p.ids[m * K + lane] = my_id;
      if (p.dbg_w) p.dbg_w[m * K + lane] = wgt;
      if (p.dbg_ids) p.dbg_ids[m * K + lane] = my_id;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) is_last = (atomicAdd(&p.counters[kCtrTicket], 1) == M - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- the last token CTA: every mask and pick into shared memory at once
  __shared__ int base_s[kMaxExperts];
  __shared__ unsigned long long mask_s[kMaxExperts];
  __shared__ int ids_s[kMaxTokens * kMaxTopk];
  for (int ex = tid; ex < E; ex += kTopkThreads) {
    mask_s[ex] = __ldcg(p.mask + ex);
    p.mask[ex] = 0ull;  // ready for the next step
  }
  for (int i = tid; i < M * K; i += kTopkThreads) ids_s[i] = __ldcg(p.ids + i);
  if (p.ready)  // the expert kernel's per-unit readiness counts start at zero
    for (int u = tid; u <= E; u += kTopkThreads) p.ready[u] = 0;
  __syncthreads();

  // ---- warp 0: active experts in increasing id, their row runs
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
      p.counters[kCtrTicket] = 0;  // ready for the next step
      p.counters[kCtrTasks] = 0;   // the expert kernel hands out tasks from zero
    }
  }
  __syncthreads();
  for (int i = tid; i < M * K; i += kTopkThreads) {
    const int mm = i / K, j = i - mm * K;
    const int ex = ids_s[i];
    const int rank = __popcll(mask_s[ex] & ((1ull << mm) - 1ull));
    const int pp = base_s[ex] + rank;
    p.tok_pos[mm * (K + 1) + j] = pp;
    p.pos_tok[pp] = mm;
  }
  for (int mm = tid; mm < M; mm += kTopkThreads) {
    const int pp = M * K + mm;
    p.tok_pos[mm * (K + 1) + K] = pp;
    p.pos_tok[pp] = mm;
  }
}

}  // namespace

int router_ksplit(int hidden, int experts) {
  // about 128 CTAs, slices of at most kMaxHs columns, a multiple of 8 columns
  int ks = 128 / (experts / kRouterWarps);
  if (ks < 1) ks = 1;
  if (ks > 16) ks = 16;
  while (hidden / ks > kMaxHs) ks *= 2;
  while (hidden % (ks * 8)) ks /= 2;
  return ks;
}

size_t router_smem_bytes(int M, int Hs) {
  return static_cast<size_t>(M + kRouterWarps) * Hs * 2;  // normed slice + gate slice
}

cudaError_t router_setup() {
  return cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(router_smem_bytes(kMaxTokens, kMaxHs)));
}

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
  dim3 grid(p.E / kRouterWarps, p.KS);
  return launch_pdl(router_kernel, grid, dim3(kThreads), router_smem_bytes(p.M, p.Hs), s, p);
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  return launch_pdl(topk_kernel, dim3(p.M), dim3(kTopkThreads), 0, s, p);
}

}  // namespace moe
