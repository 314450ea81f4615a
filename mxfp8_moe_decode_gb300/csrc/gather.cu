// Operand staging for the expert kernel.
//
// gather_kernel (every step): builds each active expert's activation panels
// (the layout is described beside kPanelPitch): for every 128-column K stage,
// the expert's MXFP8 token rows (the order the router chose) as the 128-byte
// swizzled image the MMA reads, then the stage's scale image -- row r holds in
// 32-bit cell j the four E8M0 codes (4 consecutive 32-column blocks) of the
// expert's token 32 j + r. That image is the layout the block-scaled MMA reads
// from TMEM (row n of the operand at TMEM lane n % 32, column n / 32; byte b of
// a cell = K block b of the stage), copied there by tcgen05.cp. Cells of
// absent tokens are left as they are: they only scale output columns that are
// dropped. One warp per gathered row: every lane issues all its loads of the
// token's row and codes, then scatters them into the unit's panels.
//
// sfa_pack_kernel (once, at handle creation): the weights' 32 x 32-block E8M0
// codes ("vllm.models.deepseek_v41.amd.mono.runner", MonoLayerWeights.check:
// [rows / 32, cols / 32] uint8) regrouped per (expert, 128-row tile, 128-column
// stage) into one 16-byte entry: cell c (4 bytes) = the codes of the tile's
// c-th 32-row block for the stage's 4 K blocks. A w13 tile is 64 gate rows
// (blocks 2t, 2t + 1) over the matching 64 up rows (blocks I/32 + 2t, + 1).
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;        // sfa_pack_kernel
constexpr int kGatherThreads = 128;  // gather_kernel: 4 warps, <= 80 registers each
constexpr int kMaxRows = kMaxTokens * (kMaxTopk + 1);
static_assert(kMaxTokens <= 64, "scale images use cells 0 and 1 only");

__global__ void __launch_bounds__(kGatherThreads, 1) gather_kernel(const GatherParams p) {
  // gathered row -> (unit << 16) | (row within the unit << 8) | the unit's padded rows
  __shared__ uint32_t row_map[kMaxRows];
  constexpr uint32_t kNone = 0xffffffffu;
  const int H = p.H, G = p.G;
  const int rows = min(p.M * (p.K + 1), min(p.rows_max, kMaxRows));
  for (int i = threadIdx.x; i < rows; i += kGatherThreads) row_map[i] = kNone;
  ptx::griddep_wait();  // routing tables and x8 come from the previous kernels
  ptx::griddep_launch_dependents();
  int units = p.counters[kCtrUnits];
  if (units < 0 || units > p.units_max) units = 0;  // the expert kernel reports it
  __syncthreads();
  for (int u = threadIdx.x; u < units; u += kGatherThreads) {
    const int4 a = *reinterpret_cast<const int4*>(p.act + u);  // expert, first row, rows, pad
    if (a.y < 0 || a.z < 1 || a.z > kMaxTokens || a.y + a.z > rows) continue;
    const uint32_t nt = static_cast<uint32_t>((a.z + 15) & ~15);
    for (int r = 0; r < a.z; ++r)
      row_map[a.y + r] = (static_cast<uint32_t>(u) << 16) | (static_cast<uint32_t>(r) << 8) | nt;
  }
  __syncthreads();

  // one warp per gathered row
  constexpr int kWarps = kGatherThreads / 32;
  constexpr int kPassChunks = 10;  // 16-byte chunks per lane and pass (one pass for H <= 5120)
  constexpr int kMaxStageLanes = 8192 / 128 / 32;  // K stages per lane
  const int lane = threadIdx.x & 31;
  const int n16 = H >> 4;
  const int cstride = H >> 5;  // codes per token row
  for (int row = blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows; row += gridDim.x * kWarps) {
    const uint32_t map = row_map[row];
    const int m = p.pos_tok[row];
    if (map == kNone || m < 0 || m >= p.M) continue;
    const int u = static_cast<int>(map >> 16), r = static_cast<int>((map >> 8) & 255u);
    const int nt = static_cast<int>(map & 255u);
    const uint4* src = reinterpret_cast<const uint4*>(p.x8 + static_cast<size_t>(m) * H);
    const uint8_t* csrc = p.x8c + static_cast<size_t>(m) * cstride;
    uint32_t code[kMaxStageLanes];
#pragma unroll
    for (int j = 0; j < kMaxStageLanes; ++j) {
      const int g = lane + 32 * j;
      if (g < G) code[j] = *reinterpret_cast<const uint32_t*>(csrc + 4 * g);
    }
    uint8_t* base = p.xpan + static_cast<size_t>(u) * G * kPanelPitch;
    for (int c0 = 0; c0 < n16; c0 += 32 * kPassChunks) {
      uint4 v[kPassChunks];
#pragma unroll
      for (int i = 0; i < kPassChunks; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < n16) v[i] = src[c];
      }
#pragma unroll
      for (int i = 0; i < kPassChunks; ++i) {
        const int c = c0 + lane + 32 * i;
        if (c < n16)
          *reinterpret_cast<uint4*>(base + (c >> 3) * kPanelPitch + panel_byte(r, (c & 7) << 4)) =
              v[i];
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxStageLanes; ++j) {
      const int g = lane + 32 * j;
      if (g < G)
        *reinterpret_cast<uint32_t*>(base + g * kPanelPitch + nt * 128 + (r & 31) * 16 + (r >> 5) * 4) =
            code[j];
    }
  }
}

__global__ void __launch_bounds__(kThreads) sfa_pack_kernel(const SfaPackParams p) {
  const int E = p.E, H = p.H, I = p.I;
  const int t13 = I / 64, g13 = H / 128, t2 = H / 128, g2 = I / 128;
  const long long n13 = static_cast<long long>(E + 1) * t13 * g13;
  const long long n2 = static_cast<long long>(E + 1) * t2 * g2;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n13 + n2;
       i += stride) {
    uint32_t cell[4];
    if (i < n13) {
      const int g = static_cast<int>(i % g13);
      const int t = static_cast<int>((i / g13) % t13);
      const int e = static_cast<int>(i / (static_cast<long long>(g13) * t13));
      const int ld = H / 32;
      const uint8_t* s = (e < E) ? p.w13_s + static_cast<size_t>(e) * (2 * I / 32) * ld : p.sw13_s;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int rb = (c < 2) ? (2 * t + c) : (I / 32 + 2 * t + (c - 2));
        const uint8_t* q = s + static_cast<size_t>(rb) * ld + 4 * g;
        cell[c] = q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<uint32_t>(q[3]) << 24);
      }
      p.sfa13[i] = make_uint4(cell[0], cell[1], cell[2], cell[3]);
    } else {
      const long long j = i - n13;
      const int g = static_cast<int>(j % g2);
      const int t = static_cast<int>((j / g2) % t2);
      const int e = static_cast<int>(j / (static_cast<long long>(g2) * t2));
      const int ld = I / 32;
      const uint8_t* s = (e < E) ? p.w2_s + static_cast<size_t>(e) * (H / 32) * ld : p.sw2_s;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint8_t* q = s + static_cast<size_t>(4 * t + c) * ld + 4 * g;
        cell[c] = q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<uint32_t>(q[3]) << 24);
      }
      p.sfa2[j] = make_uint4(cell[0], cell[1], cell[2], cell[3]);
    }
  }
}

}  // namespace

// One CTA of 128 threads per SM: its registers fit beside the expert kernel's
// CTA, which then starts (and streams its first weight stages) while the
// gather still runs.
cudaError_t launch_gather(const GatherParams& p, int num_sms, cudaStream_t s) {
  return launch_pdl(gather_kernel, dim3(num_sms), dim3(kGatherThreads), 0, s, p);
}

cudaError_t launch_sfa_pack(const SfaPackParams& p, cudaStream_t s) {
  sfa_pack_kernel<<<1024, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
