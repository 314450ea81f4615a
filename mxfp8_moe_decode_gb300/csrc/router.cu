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
// bulk-copies the normed rows' K-slice into shared memory. The product is a
// small dense contraction, done on the tensor cores with warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate): tokens are the MMA's rows (16 per tile, up to
// 3 tiles), the CTA's 8 experts its columns; warp w takes the K-slice's
// 16-column steps w, w + 8, ...; the 8 warps' partial tiles are then summed
// in a fixed order into logit_part[ks][m][e]. Row pitches in shared memory are
// padded by 16 bytes so the fragment loads hit 32 distinct banks.
//
// topk_kernel: one CTA per token. A thread per expert sums the KS partial
// logits in a fixed order (all partial loads issued before the sum), takes
// sigmoid and score + bias and forms a 64-bit key (order-preserving bits of
// the choice, then the inverted expert index, so equal choices go to the
// lower index); the k largest keys are found by rank (rank within each group
// of 32 experts, then among the groups' candidates). Lane j of warp 0 keeps
// pick j and takes the token's row (slot) among the expert's rows with an
// atomic on the expert's row counter (a lone token's slots are 0 and it sets
// the counts); then the CTA writes the token's MXFP8 row and codes into the x
// panels of its k experts (the expert kernel's B operand; the seam writes the
// shared expert's, and a lone token's experts read that one). The per-expert
// row counts are all the expert and combine kernels need to lay out the
// step's units (see pack_unit); the router clears them before the next step.
#include <cfloat>
#include <cmath>

#include "internal.cuh"
#include "ptx.cuh"
#include "seam.cuh"

namespace moe {
namespace {

constexpr int kThreads = kRouterWarps * 32;
constexpr int kMaxHs = 1536;                    // K-slice columns per router CTA
constexpr int kMaxChunks = kMaxHs / 256;        // 256-column chunks (8 columns per lane)
constexpr int kMaxKsplit = 16;                  // K-slices of the router GEMV
constexpr int kTopkThreads = 256;
static_assert(8192 / 16 <= 2 * kTopkThreads && 8192 / 128 <= kTopkThreads,
              "the top-k kernel holds a token row of up to 8192 columns in registers");

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// D (16 x 8, f32) += A (16 x 16, bf16, row-major) . B (16 x 8, bf16, column-major)
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kMTiles = (kMaxTokens + 15) / 16;
// fused seam: slice octets per thread (kSeamFuseMaxM rows of at most kMaxHs columns)
constexpr int kFuseIters = (kSeamFuseMaxM * (kMaxHs / 8) + kThreads - 1) / kThreads;
static_assert(kSeamFuseMaxM <= 4, "the fused seam's sums of squares take rows two at a time");

__host__ __device__ constexpr int router_pitch(int Hs) { return Hs * 2 + 16; }

__global__ void __launch_bounds__(kThreads) router_kernel(const RouterParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;  // completion of the bulk copies into smem
  const int M = p.M, H = p.H, E = p.E, Hs = p.Hs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = blockIdx.y * Hs;
  const int e0 = blockIdx.x * kRouterWarps;
  const int mtiles = (M + 15) >> 4;
  const int ld = router_pitch(Hs);  // bytes per row in shared memory
  const int rows = 16 * mtiles;
  uint8_t* xs = smem;                                        // [rows][ld] normed rows
  uint8_t* gs = smem + static_cast<size_t>(rows) * ld;       // [8][ld] gate rows
  float* red = reinterpret_cast<float*>(gs + static_cast<size_t>(kRouterWarps) * ld);  // [8][rows][8]

  // ---- gate rows first: they do not depend on the previous kernel
  {
    const int oct = Hs >> 3;  // 16-byte pieces of one row slice
    const uint4* src =
        reinterpret_cast<const uint4*>(p.gate_w + static_cast<size_t>(e0 + warp) * H + k0);
    uint4 g[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int i = c * 32 + lane;
      g[c] = i < oct ? src[i] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      const int i = c * 32 + lane;
      if (i < oct) *reinterpret_cast<uint4*>(gs + warp * ld + 16 * i) = g[c];
    }
  }
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  // fused seam: the norm weight of this thread's slice octets, before waiting
  const int nsl = Hs >> 3;  // octets of the K-slice
  uint4 wpre[kFuseIters];
  if (p.x) {
#pragma unroll
    for (int s = 0; s < kFuseIters; ++s) {
      const int q = s * kThreads + tid;
      wpre[s] = q < M * nsl ? __ldg(reinterpret_cast<const uint4*>(p.norm_w) + (k0 >> 3) + q % nsl)
                            : make_uint4(0, 0, 0, 0);
    }
  }
  ptx::griddep_wait();  // the normed rows (or x) come from the previous kernel
  ptx::griddep_launch_dependents();
  if (blockIdx.x == 0 && blockIdx.y == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (p.clear[r])
        for (int i = tid; i < p.clear_n[r]; i += kThreads) p.clear[r][i] = 0;
  }
  if (p.zero_rows) {
    const size_t stride = static_cast<size_t>(gridDim.x) * gridDim.y * kThreads;
    for (size_t i = (static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x) * kThreads + tid;
         i < p.zero_n; i += stride)
      p.zero_rows[i] = 0.0f;
  }
  __syncthreads();

  bool landed = true;  // the K-slice of the normed rows is in shared memory
  if (p.x) {
    // ---- fused seam, in the seam's arithmetic and order (seam.cuh): first
    // every row's sum of squares -- thread t plays owner t & 127 for rows
    // (t >> 7) and (t >> 7) + 2 -- then this CTA's K-slice of the normed rows
    // straight into shared memory
    __shared__ float warp_sums[kSeamFuseMaxM][4];
    __shared__ float scale_s[kSeamFuseMaxM];
    {
      const int own = tid & (kSeamOwners - 1), m0 = tid >> 7, noct = H >> 3;
      uint4 raw[2][kSeamMaxOct];
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int m = m0 + 2 * ps;
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * H);
#pragma unroll
        for (int i = 0; i < kSeamMaxOct; ++i) {
          const int o = own + i * kSeamOwners;
          raw[ps][i] = m < M && o < noct ? __ldg(xr + o) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        const int m = m0 + 2 * ps;  // the same in the whole warp
        if (m < M) {
          float ss = 0.0f;
#pragma unroll
          for (int i = 0; i < kSeamMaxOct; ++i) {
            if (own + i * kSeamOwners < noct) {
              float v[8];
              unpack_bf16x8(raw[ps][i], v);
              ss = seam_sumsq_octet(v, ss);
            }
          }
          ss = seam_warp_sum(ss);
          if (lane == 0) warp_sums[m][warp & 3] = ss;
        }
      }
    }
    __syncthreads();
    if (tid < M) scale_s[tid] = seam_scale(warp_sums[tid], H, p.eps);
    __syncthreads();
    // octet q of the slice tasks: row q / nsl, octet k0 / 8 + q % nsl; the 4
    // octets of a 32-group are 4 adjacent lanes (nsl is a multiple of 4)
    const bool writer = blockIdx.x == 0;
#pragma unroll
    for (int s = 0; s < kFuseIters; ++s) {
      const int q0 = s * kThreads;
      if (q0 >= M * nsl) break;  // uniform
      const int q = q0 + tid;
      const bool live = q < M * nsl;
      const int m = live ? q / nsl : 0, ol = q - m * nsl, o = (k0 >> 3) + ol;
      float v[8];
      unpack_bf16x8(live ? __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * H) + o)
                         : make_uint4(0, 0, 0, 0),
                    v);
      uint4 nv;
      int code;
      const uint2 q8 = seam_quant_octet(v, wpre[s], scale_s[m], &nv, &code);
      if (live) {
        *reinterpret_cast<uint4*>(xs + static_cast<size_t>(m) * ld + 16 * ol) = nv;
        if (writer) {
          const size_t row = static_cast<size_t>(m) * H;
          reinterpret_cast<uint2*>(p.x8 + row)[o] = q8;
          if (p.dbg_normed) reinterpret_cast<uint4*>(p.dbg_normed + row)[o] = nv;
          if (p.dbg_x8) reinterpret_cast<uint2*>(p.dbg_x8 + row)[o] = q8;
          if ((o & 3) == 0) {
            const size_t ci = static_cast<size_t>(m) * (H >> 5) + (o >> 2);
            p.x8c[ci] = static_cast<uint8_t>(code);
            if (p.dbg_x8c) p.dbg_x8c[ci] = static_cast<uint8_t>(code);
          }
          seam_store_panel(p.xpan_shared, m, o, q8, code);
        }
      }
    }
    __syncthreads();
  } else {
    // ---- the K-slice of every normed row: one bulk copy per row, all in
    // flight (rows M .. rows - 1 are left as they are: they only feed output
    // rows that are dropped)
    if (tid == 0) {
      const uint32_t b = ptx::smem_u32(&bar);
      ptx::mbar_arrive_expect_tx(b, static_cast<uint32_t>(M) * Hs * 2);
      for (int m = 0; m < M; ++m)
        ptx::bulk_load(ptx::smem_u32(xs + static_cast<size_t>(m) * ld),
                       p.normed + static_cast<size_t>(m) * H + k0, Hs * 2, b);
    }
    int never = 0;
    landed = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &never, kWaitLimitNs);
  }
  // A bulk-copy wait that gave up: record it in the error word, let the
  // copies still in flight land (bounded) so none writes into the shared
  // memory of a later CTA, and skip the product and its stores.
  if (!__syncthreads_and(landed)) {
    if (tid == 0) {
      if (p.err) atomicOr(p.err, kErrTimeout);
      int never = 0;
      ptx::mbar_wait(ptx::smem_u32(&bar), 0, &never, kWaitLimitNs);
    }
    return;
  }
  // ---- this CTA's share of the L2 prefetch (chunks b, b + ctas, ... of each
  // range), issued once the CTA's own loads have landed so that it does not
  // delay them
  if (tid < 32) {
    constexpr uint32_t kChunk = 32 * 1024;
    const uint32_t ctas = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
    const uint64_t pol = ptx::policy_evict_last();
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!p.pf_ptr[r]) continue;
      const uint64_t n = (p.pf_bytes[r] + kChunk - 1) / kChunk;
      for (uint64_t c = b + ctas * static_cast<uint64_t>(tid); c < n; c += ctas * 32ull) {
        const uint64_t off = c * kChunk;
        const uint64_t len = p.pf_bytes[r] - off < kChunk ? p.pf_bytes[r] - off : kChunk;
        ptx::prefetch_l2(p.pf_ptr[r] + off, static_cast<uint32_t>(len), pol);
      }
    }
  }

  // ---- tensor-core partial products over this warp's 16-column steps
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group, column pair
  float d[kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < kMTiles; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[mt][i] = 0.0f;
  const uint8_t* brow = gs + gq * ld + 4 * tq;  // B column gq = gate row e0 + gq
  for (int st = warp; st < (Hs >> 4); st += kRouterWarps) {
    const int kb = st * 32;  // byte offset of the step's 16 columns
    const uint32_t b0 = lds32(brow + kb), b1 = lds32(brow + kb + 16);
#pragma unroll
    for (int mt = 0; mt < kMTiles; ++mt) {
      if (mt < mtiles) {
        const uint8_t* r0 = xs + (16 * mt + gq) * ld + kb + 4 * tq;
        const uint8_t* r1 = r0 + 8 * ld;
        mma_bf16_16816(d[mt], lds32(r0), lds32(r1), lds32(r0 + 16), lds32(r1 + 16), b0, b1);
      }
    }
  }

  // ---- the 8 warps' tiles summed in a fixed order
#pragma unroll
  for (int mt = 0; mt < kMTiles; ++mt) {
    if (mt < mtiles) {
      float* t = red + (static_cast<size_t>(warp) * rows + 16 * mt + gq) * 8 + 2 * tq;
      t[0] = d[mt][0];
      t[1] = d[mt][1];
      t[64] = d[mt][2];  // row + 8
      t[65] = d[mt][3];
    }
  }
  __syncthreads();
  float* out = p.logit_part + static_cast<size_t>(blockIdx.y) * M * E + e0;
  for (int i = tid; i < M * kRouterWarps; i += kThreads) {
    const int m = i >> 3, c = i & 7;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) v += red[(static_cast<size_t>(w) * rows + m) * 8 + c];
    out[static_cast<size_t>(m) * E + c] = v;
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
  const int M = p.M, E = p.E, K = p.K, KS = p.KS;
  const int m = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ unsigned long long key_s[kMaxExperts];
  __shared__ unsigned long long cand_s[kMaxExperts];  // (E / 32) groups x K
  __shared__ float s_s[kMaxExperts];
  __shared__ int pick_s[kMaxTopk];
  __shared__ int slot_s[kMaxTopk];
  int pk_id = 0, pk_slot = 0;  // lane j < k of warp 0: pick j
  float pk_w = 0.0f;
  static_assert(kMaxExperts <= 2 * kTopkThreads, "two experts per thread");
  // the bias does not depend on the router: fetch it before waiting
  float bias[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int ex = tid + i * kTopkThreads;
    bias[i] = ex < E ? p.bias[ex] : 0.0f;
  }
  // this token's MXFP8 row (16-byte pieces) and scale codes (one word per 128
  // columns), loaded once the grid dependency is met so that their latency
  // hides behind the selection; they are stored into the picked experts'
  // panels below
  constexpr int kMaxPieces = 2;  // 16-byte pieces per thread: H <= 8192
  const int H = p.H, G = H >> 7, n16 = H >> 4;
  uint4 xv[kMaxPieces];
  uint32_t cw = 0;
  // (a lone token's experts read the shared expert's panels, which the seam
  // writes: nothing to store then)
  const bool panels = p.xpan != nullptr && M > 1;
#pragma unroll
  for (int q = 0; q < kMaxPieces; ++q) xv[q] = make_uint4(0, 0, 0, 0);

  // Two passes over the same code: the first, before the grid dependency
  // wait, selects on scores of 1/2 (no loads, no global writes) so that the
  // selection's instructions are fetched while this CTA would only wait; the
  // second selects on the router's logits.
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const bool real = pass != 0;
    if (real) {
      ptx::griddep_wait();  // partial logits come from the router kernel
      ptx::griddep_launch_dependents();
      if (panels) {
        const uint4* xrow = reinterpret_cast<const uint4*>(p.x8 + static_cast<size_t>(m) * H);
#pragma unroll
        for (int q = 0; q < kMaxPieces; ++q) {
          const int c = tid + q * kTopkThreads;
          xv[q] = c < n16 ? __ldcg(xrow + c) : make_uint4(0, 0, 0, 0);
        }
        if (tid < G)
          cw = __ldcg(reinterpret_cast<const uint32_t*>(p.x8c + static_cast<size_t>(m) * (H >> 5)) +
                      tid);
      }
    }

    // ---- one thread per expert: the KS partials (all loads in flight), then
    // their sum in a fixed order, the score and the choice key
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int ex = tid + i * kTopkThreads;
      if (ex < E) {
        float logit = 0.0f;
        if (real) {
          float part[kMaxKsplit];
#pragma unroll
          for (int ks = 0; ks < kMaxKsplit; ++ks)
            part[ks] =
                ks < KS ? __ldcg(p.logit_part + (static_cast<size_t>(ks) * M + m) * E + ex) : 0.0f;
#pragma unroll
          for (int ks = 0; ks < kMaxKsplit; ++ks)
            if (ks < KS) logit += part[ks];
        }
        const float s = 1.0f / (1.0f + expf(-logit));
        s_s[ex] = s;
        key_s[ex] = choice_key(s + bias[i], ex);
        if (real && p.dbg_logits) p.dbg_logits[static_cast<size_t>(m) * E + ex] = logit;
      }
    }
    __syncthreads();

    // ---- the k largest keys by rank (keys are distinct: they hold the expert
    // index): first each expert's rank within its group of 32 (a group's k best
    // are candidates), then each candidate's rank among all candidates; the
    // candidate of rank j is pick j
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int ex = tid + i * kTopkThreads;
      if (ex < E) {
        const unsigned long long mine = key_s[ex];
        const unsigned long long* grp = key_s + (ex & ~31);
        int rank = 0;
#pragma unroll 8
        for (int o = 0; o < 32; ++o) rank += grp[o] > mine;
        if (rank < K) cand_s[(ex >> 5) * K + rank] = mine;
      }
    }
    __syncthreads();
    // (four adjacent lanes per candidate, each counting over a quarter)
    const int ncand = (E >> 5) * K;
    for (int c0 = 0; c0 < ncand; c0 += kTopkThreads / 4) {
      const int c = c0 + (tid >> 2);
      const bool live = c < ncand;
      const unsigned long long mine = live ? cand_s[c] : 0ull;
      int rank = 0;
      if (live)
        for (int o = tid & 3; o < ncand; o += 4) rank += cand_s[o] > mine;
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      rank += __shfl_xor_sync(0xffffffffu, rank, 2);
      if (live && (tid & 3) == 0 && rank < K) {
        const int ex = 0x7fffffff - static_cast<int>(static_cast<uint32_t>(mine));
        pick_s[rank] = ex;
      }
    }
    __syncthreads();
    if (warp == 0) {
      // small steps: publish the picks at once (the expert kernel, already
      // resident, prefetches the picked experts' first stages into L2 while
      // this grid and its successor's dependency wait finish)
      if (real && p.picks_early) {
        if (lane < K) p.picks_early[1 + m * K + lane] = pick_s[lane];
        __syncwarp();
        if (lane == 0)
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.picks_early) : "memory");
      }
      // the chosen scores' sum in pick order (the same in every lane)
      float ssum = 0.0f;
      bool bad = false;
      for (int j = 0; j < K; ++j) {
        int ex = pick_s[j];
        if (ex < 0 || ex >= E) {  // only with non-finite scores
          bad = true;
          ex = 0;
        }
        ssum += s_s[ex];
      }
      if (real && bad && lane == 0) atomicOr(&p.counters[kCtrErr], kErrBounds);
      if (lane < K) {
        int my_id = pick_s[lane];
        if (my_id < 0 || my_id >= E) my_id = 0;
        pk_w = s_s[my_id] / ssum;
        // the token's row among the expert's rows this step (any order: an MMA
        // output column depends on its own row only); a lone token's is row 0
        pk_slot = real && M > 1 ? atomicAdd(p.cnt + my_id, 1) : 0;
        pk_id = my_id;
        pick_s[lane] = my_id;
        slot_s[lane] = pk_slot;
      }
    }
    // (global stores go after the barriers where they can: a block barrier
    // waits for the stores before it)
    __syncthreads();
  }

  // ---- this token's MXFP8 row and codes into the x panels of its experts
  // (row = its slot): each 16-byte piece is read once and stored k times.
  // Only the next kernel reads them: they go out last, after the picks.
  auto write_panels = [&]() {
    if (!panels) return;
#pragma unroll
    for (int q = 0; q < kMaxPieces; ++q) {
      const int c = tid + q * kTopkThreads;
      if (c >= n16) break;
      const uint4 v = xv[q];
      for (int d = 0; d < K; ++d) {
        const int e = pick_s[d], r = slot_s[d];
        if (r < 0 || r >= kMaxTokens) continue;
        *reinterpret_cast<uint4*>(p.xpan + (static_cast<size_t>(e) * G + (c >> 3)) * kPanelPitch +
                                  panel_byte(r, (c & 7) << 4)) = v;
      }
    }
    if (tid < G) {
      const int g = tid;
      const uint32_t code = cw;
      for (int d = 0; d < K; ++d) {
        const int e = pick_s[d], r = slot_s[d];
        if (r < 0 || r >= kMaxTokens) continue;
        *reinterpret_cast<uint32_t*>(p.xpan + (static_cast<size_t>(e) * G + g) * kPanelPitch +
                                     panel_code_byte(r)) = code;
      }
    }
  };

  if (warp == 0 && lane < K) {
    p.route_w[m * K + lane] = pk_w;
    p.ids[m * K + lane] = pk_id;
    p.slots[m * K + lane] = pk_slot;
    if (M == 1) p.cnt[pk_id] = 1;  // (a lone token takes no slot atomics)
    if (p.dbg_w) p.dbg_w[m * K + lane] = pk_w;
    if (p.dbg_ids) p.dbg_ids[m * K + lane] = pk_id;
  }
  write_panels();
}

}  // namespace

int router_ksplit(int hidden, int experts) {
  // about 128 CTAs, slices of at most kMaxHs columns, a multiple of 8 columns
  int ks = 128 / (experts / kRouterWarps);
  if (ks < 1) ks = 1;
  if (ks > 16) ks = 16;
  while (hidden / ks > kMaxHs) ks *= 2;
  while (ks > 1 && hidden % (ks * 16)) ks /= 2;  // whole 16-column MMA steps
  return ks;
}

size_t router_smem_bytes(int M, int Hs) {
  const size_t rows = 16 * static_cast<size_t>((M + 15) / 16);
  // normed rows (padded to whole MMA tiles) + gate rows + the warps' partial tiles
  return (rows + kRouterWarps) * router_pitch(Hs) + kRouterWarps * rows * 8 * sizeof(float);
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
