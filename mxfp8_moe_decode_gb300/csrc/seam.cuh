// The FFN seam's per-row arithmetic, shared by the seam kernel and the router
// kernel's fused seam (small steps): RMSNorm of a bf16 token row in fp32, the
// bf16 MoE input row, and its MXFP8 quantisation (E4M3 bytes, one E8M0 code
// per 32 columns).
//
// "vllm.models.deepseek_v41.amd.mono.layer", run_ffn: per token, the seam's
// norm (seam.stage_norm, f32 outputs) then store_normed (the bf16 MoE input
// row); store_x8: amax of a 32-group reduced over the 4 lanes that hold its 8
// columns each (butterfly over lane xor 1, 2), the code, then E4M3 packing of
// the clamped scaled values. The norm is x * (mean(x^2) + eps)^(-1/2) * w
// computed in fp32; the quantisation reads the bf16-rounded normed values.
//
// The sum of squares has one fixed order, whoever computes it: 128 owners,
// owner i holding the 8-column octets i, i + 128, ...; each owner's fmaf chain
// over its octets in increasing order, a butterfly tree over each 32-owner
// warp, then the four warp sums as (w0 + w1) + (w2 + w3).
#pragma once

#include "internal.cuh"
#include "mx.cuh"

namespace moe {

constexpr int kSeamOwners = 128;
constexpr int kSeamMaxOct = 8192 / 8 / kSeamOwners;  // octets per owner (H <= 8192)

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

// One octet into an owner's fmaf chain.
__device__ __forceinline__ float seam_sumsq_octet(const float* v, float ss) {
#pragma unroll
  for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
  return ss;
}

// The butterfly over the 32 owners of a warp (every lane gets the warp sum).
__device__ __forceinline__ float seam_warp_sum(float ss) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  return ss;
}

// The row's scale from the four warp sums.
__device__ __forceinline__ float seam_scale(const float* warp_sums, int H, float eps) {
  const float tot = (warp_sums[0] + warp_sums[1]) + (warp_sums[2] + warp_sums[3]);
  return rsqrtf(tot / static_cast<float>(H) + eps);
}

// One octet of the normed row: its bf16 values (nv) and, with the other three
// octets of its 32-group in lanes 4a .. 4a + 3 of the same warp (all 32 lanes
// call this together), the group's code and the octet's 8 E4M3 bytes.
__device__ __forceinline__ uint2 seam_quant_octet(const float* v, const uint4& wraw, float r,
                                                  uint4* nv, int* code_out) {
  float w[8];
  unpack_bf16x8(wraw, w);
  __align__(16) __nv_bfloat16 nb[8];
  float n[8];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    nb[j] = __float2bfloat16_rn((v[j] * r) * w[j]);
    n[j] = __bfloat162float(nb[j]);
    amax = fmaxf(amax, fabsf(n[j]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int code = mx_code(amax);
  const float mul = mx_mul(code);
  uint2 q;
  q.x = static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[0] * mul), clamp_e4m3(n[1] * mul))) |
        (static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[2] * mul), clamp_e4m3(n[3] * mul))) << 16);
  q.y = static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[4] * mul), clamp_e4m3(n[5] * mul))) |
        (static_cast<uint32_t>(e4m3x2(clamp_e4m3(n[6] * mul), clamp_e4m3(n[7] * mul))) << 16);
  *nv = *reinterpret_cast<const uint4*>(nb);
  *code_out = code;
  return q;
}

// Octet o of token row t into the shared expert's x panels (rows = tokens):
// its 8 code bytes, and (from the group's first octet) the group's scale code.
__device__ __forceinline__ void seam_store_panel(uint8_t* xpan_shared, int t, int o, uint2 q,
                                                 int code) {
  uint8_t* pan = xpan_shared + static_cast<size_t>(o >> 4) * kPanelPitch;
  *reinterpret_cast<uint2*>(pan + panel_byte(t, (o & 15) << 3)) = q;
  if ((o & 3) == 0) pan[panel_code_byte(t) + ((o >> 2) & 3)] = static_cast<uint8_t>(code);
}

}  // namespace moe
