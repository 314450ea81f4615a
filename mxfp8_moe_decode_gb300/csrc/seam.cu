// FFN seam kernel: RMSNorm of each bf16 token row -> bf16 MoE input row ->
// MXFP8 (E4M3 bytes + one E8M0 code per 32 columns); the arithmetic and its
// sources are in seam.cuh. Steps of up to kSeamFuseMaxM tokens run the same
// arithmetic inside the router kernel instead.
//
// One CTA per token row, 128 threads: thread i is owner i, holding the
// 8-column octets i, i + 128, ... so the 4 octets of a 32-group sit in 4
// adjacent lanes.
#include "internal.cuh"
#include "ptx.cuh"
#include "seam.cuh"

namespace moe {
namespace {

constexpr int kThreads = kSeamOwners;

__global__ void __launch_bounds__(kThreads) seam_kernel(const SeamParams p) {
  const int t = blockIdx.x;
  const int H = p.H;
  const int noct = H >> 3;
  const int tid = threadIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
  const uint4* wr = reinterpret_cast<const uint4*>(p.norm_w);
  // the norm weight does not depend on earlier work: fetch it before waiting
  uint4 wraw[kSeamMaxOct];
#pragma unroll
  for (int i = 0; i < kSeamMaxOct; ++i) {
    const int o = tid + i * kThreads;
    wraw[i] = o < noct ? wr[o] : make_uint4(0, 0, 0, 0);
  }
  // x comes from the previous kernel on the stream; the router may start now
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  float v[kSeamMaxOct][8];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kSeamMaxOct; ++i) {
    const int o = tid + i * kThreads;
    if (o < noct) {
      unpack_bf16x8(xr[o], v[i]);
      ss = seam_sumsq_octet(v[i], ss);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
    }
  }
  ss = seam_warp_sum(ss);
  __shared__ float red[kThreads / 32];
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  const float r = seam_scale(red, H, p.eps);

  const size_t row = static_cast<size_t>(t) * H;
#pragma unroll
  for (int i = 0; i < kSeamMaxOct; ++i) {
    const int o = tid + i * kThreads;
    if (i * kThreads >= noct) break;  // uniform across the CTA
    const bool live = o < noct;
    uint4 nv;
    int code;
    const uint2 q = seam_quant_octet(v[i], wraw[i], r, &nv, &code);  // zero past the row
    if (live) {
      reinterpret_cast<uint4*>(p.normed + row)[o] = nv;
      reinterpret_cast<uint2*>(p.x8 + row)[o] = q;
      if (p.dbg_normed) reinterpret_cast<uint4*>(p.dbg_normed + row)[o] = nv;
      if (p.dbg_x8) reinterpret_cast<uint2*>(p.dbg_x8 + row)[o] = q;
      if ((o & 3) == 0) {
        const size_t ci = static_cast<size_t>(t) * (H >> 5) + (o >> 2);
        p.x8c[ci] = static_cast<uint8_t>(code);
        if (p.dbg_x8c) p.dbg_x8c[ci] = static_cast<uint8_t>(code);
      }
      if (p.xpan_shared) seam_store_panel(p.xpan_shared, t, o, q, code);
    }
  }
}

}  // namespace

cudaError_t launch_seam(const SeamParams& p, int M, cudaStream_t s) {
  return launch_pdl(seam_kernel, dim3(M), dim3(kThreads), 0, s, p);
}

}  // namespace moe
