// FFN seam: RMSNorm of each bf16 token row -> bf16 MoE input row -> MXFP8
// (E4M3 bytes + one E8M0 code per 32 columns).
//
// "vllm.models.deepseek_v41.amd.mono.layer", run_ffn: per token, the seam's
// norm (seam.stage_norm, f32 outputs) then store_normed (the bf16 MoE input
// row); store_x8: amax of a 32-group reduced over the 4 lanes that hold its 8
// columns each (butterfly over lane xor 1, 2), the code, then E4M3 packing of
// the clamped scaled values. The norm is x * (mean(x^2) + eps)^(-1/2) * w
// computed in fp32; the quantisation reads the bf16-rounded normed values.
//
// One CTA per token row, 128 threads; thread i owns the 8-column octets
// i, i + 128, ... so the 4 octets of a 32-group sit in 4 adjacent lanes.
#include "internal.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxOct = 8;  // H <= 8192

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

__global__ void __launch_bounds__(kThreads) seam_kernel(const SeamParams p) {
  const int t = blockIdx.x;
  const int H = p.H;
  const int noct = H >> 3;
  const int tid = threadIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
  const uint4* wr = reinterpret_cast<const uint4*>(p.norm_w);
  // the norm weight does not depend on earlier work: fetch it before waiting
  uint4 wraw[kMaxOct];
#pragma unroll
  for (int i = 0; i < kMaxOct; ++i) {
    const int o = tid + i * kThreads;
    wraw[i] = o < noct ? wr[o] : make_uint4(0, 0, 0, 0);
  }
  // x comes from the previous kernel on the stream; the router may start now
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  float v[kMaxOct][8];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxOct; ++i) {
    const int o = tid + i * kThreads;
    if (o < noct) {
      unpack_bf16x8(xr[o], v[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(v[i][j], v[i][j], ss);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
    }
  }
  // sum of squares: warp tree, then the 4 warp sums in a fixed order
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float red[kThreads / 32];
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  const float tot = (red[0] + red[1]) + (red[2] + red[3]);
  const float r = rsqrtf(tot / static_cast<float>(H) + p.eps);

  const size_t row = static_cast<size_t>(t) * H;
#pragma unroll
  for (int i = 0; i < kMaxOct; ++i) {
    const int o = tid + i * kThreads;
    if (i * kThreads >= noct) break;  // uniform across the CTA
    const bool live = o < noct;
    float w[8];
    unpack_bf16x8(wraw[i], w);  // zero past the row
    float n[8];
    __align__(16) __nv_bfloat16 nb[8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      nb[j] = __float2bfloat16_rn((v[i][j] * r) * w[j]);
      n[j] = __bfloat162float(nb[j]);
      amax = fmaxf(amax, fabsf(n[j]));
    }
    // the 32-group's 4 octets are in lanes 4a .. 4a+3
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int code = mx_code(amax);
    const float mul = mx_mul(code);
    uint2 q;
    q.x = static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[0] * mul), clamp_e4m3(n[1] * mul))) |
          (static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[2] * mul), clamp_e4m3(n[3] * mul))) << 16);
    q.y = static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[4] * mul), clamp_e4m3(n[5] * mul))) |
          (static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[6] * mul), clamp_e4m3(n[7] * mul))) << 16);
    if (live) {
      const uint4 nv = *reinterpret_cast<const uint4*>(nb);
      reinterpret_cast<uint4*>(p.normed + row)[o] = nv;
      reinterpret_cast<uint2*>(p.x8 + row)[o] = q;
      if (p.dbg_normed) reinterpret_cast<uint4*>(p.dbg_normed + row)[o] = nv;
      if (p.dbg_x8) reinterpret_cast<uint2*>(p.dbg_x8 + row)[o] = q;
      if ((tid & 3) == 0) {
        const size_t ci = static_cast<size_t>(t) * (H >> 5) + (o >> 2);
        p.x8c[ci] = static_cast<uint8_t>(code);
        if (p.dbg_x8c) p.dbg_x8c[ci] = static_cast<uint8_t>(code);
      }
      if (p.xpan_shared) {
        // row t of the shared expert's x panels: the 8 code bytes at column
        // 8 o of the panel (o >> 4), and the group's scale code in its image
        uint8_t* pan = p.xpan_shared + static_cast<size_t>(o >> 4) * kPanelPitch;
        *reinterpret_cast<uint2*>(pan + panel_byte(t, (o & 15) << 3)) = q;
        if ((tid & 3) == 0) pan[panel_code_byte(t) + ((o >> 2) & 3)] = static_cast<uint8_t>(code);
      }
    }
  }
}

}  // namespace

cudaError_t launch_seam(const SeamParams& p, int M, cudaStream_t s) {
  return launch_pdl(seam_kernel, dim3(M), dim3(kThreads), 0, s, p);
}

}  // namespace moe
