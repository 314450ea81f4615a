// Weight-scale packing for the expert kernel.
//
// sfa_pack_kernel (once, at handle creation): the weights' 32 x 32-block E8M0
// codes ("vllm.models.deepseek_v41.amd.mono.runner", MonoLayerWeights.check:
// [rows / 32, cols / 32] uint8) regrouped per (expert, 128-row tile, 128-column
// stage) into one 16-byte entry: cell c (4 bytes) = the codes of the tile's
// c-th 32-row block for the stage's 4 K blocks. A w13 tile is 64 gate rows
// (blocks 2t, 2t + 1) over the matching 64 up rows (blocks I/32 + 2t, + 1).
// The expert kernel copies an entry into all 32 lanes of a stage's scale
// image: lane i, cell c serves MMA row 32 c + i.
//
// img_pack_kernel (MXFP4 routed experts, whose codes are per row per 32
// columns: MonoLayerWeights, w13_s [E * 2 inter, HIDDEN / 32]): the image
// itself per (expert, tile, stage), 32 lanes x 16 bytes, lane i cell c = the
// 4 codes of MMA row 32 c + i for the stage's 4 K blocks (MMA rows 0-63 of a
// w13 tile are gate rows 64 t .., rows 64-127 the up rows I + 64 t ..).
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

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
      if (p.fp4 && e < E) continue;  // routed codes are per row: img_pack_kernel
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
      if (p.fp4 && e < E) continue;
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

// 4 consecutive codes as one little-endian word (byte b = K block 4 g + b)
__device__ __forceinline__ uint32_t codes4(const uint8_t* q) {
  return q[0] | (q[1] << 8) | (q[2] << 16) | (static_cast<uint32_t>(q[3]) << 24);
}

__global__ void __launch_bounds__(kThreads) img_pack_kernel(const SfaPackParams p) {
  const int E = p.E, H = p.H, I = p.I;
  const int t13 = I / 64, g13 = H / 128, t2 = H / 128, g2 = I / 128;
  const long long n13 = static_cast<long long>(E) * t13 * g13 * 32;
  const long long n2 = static_cast<long long>(E) * t2 * g2 * 32;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n13 + n2;
       i += stride) {
    uint32_t cell[4];
    if (i < n13) {
      const int lane = static_cast<int>(i & 31);
      const long long q = i >> 5;
      const int g = static_cast<int>(q % g13);
      const int t = static_cast<int>((q / g13) % t13);
      const int e = static_cast<int>(q / (static_cast<long long>(g13) * t13));
      const int ld = H / 32;
      const uint8_t* s = p.w13_s + static_cast<size_t>(e) * (2 * I) * ld;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int row = (c < 2) ? (64 * t + 32 * c + lane) : (I + 64 * t + 32 * (c - 2) + lane);
        cell[c] = codes4(s + static_cast<size_t>(row) * ld + 4 * g);
      }
      p.img13[i] = make_uint4(cell[0], cell[1], cell[2], cell[3]);
    } else {
      const long long j = i - n13;
      const int lane = static_cast<int>(j & 31);
      const long long q = j >> 5;
      const int g = static_cast<int>(q % g2);
      const int t = static_cast<int>((q / g2) % t2);
      const int e = static_cast<int>(q / (static_cast<long long>(g2) * t2));
      const int ld = I / 32;
      const uint8_t* s = p.w2_s + static_cast<size_t>(e) * H * ld;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        cell[c] = codes4(s + static_cast<size_t>(128 * t + 32 * c + lane) * ld + 4 * g);
      p.img2[j] = make_uint4(cell[0], cell[1], cell[2], cell[3]);
    }
  }
}

}  // namespace

cudaError_t launch_sfa_pack(const SfaPackParams& p, cudaStream_t s) {
  sfa_pack_kernel<<<1024, kThreads, 0, s>>>(p);
  if (p.fp4) img_pack_kernel<<<1024, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
