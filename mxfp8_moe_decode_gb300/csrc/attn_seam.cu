// Attention-seam MXFP8: RMSNorm of each bf16 token row in fp32, then MXFP8
// of the fp32 norm outputs themselves (E4M3 bytes + one E8M0 code per 32
// columns), with no bf16 rounding in between.
//
// "vllm.models.deepseek_v41.amd.mono.layer", store_x8: the attention seam's
// norm output (seam.stage_norm's 8 f32 columns per lane) goes to the
// attention's input quant: amax over the lane's 8 values, then over the 4
// lanes holding the group (butterfly over lane xor 1, 2), the code
// (mx_code), the multiplier 2^(127 - code), and E4M3 packing of the clamped
// products; 2 words of bytes per 8 columns and one code byte per 32. The
// norm is the FFN seam's (same fp32 order: see seam.cuh) with the attention
// norm weight; unlike the FFN seam, the quant reads the fp32 values.
//
// One CTA per token row, 128 threads (owner i holds the octets i, i + 128, ...).
#include "internal.cuh"
#include "ptx.cuh"
#include "seam.cuh"

namespace moe {
namespace {

constexpr int kThreads = kSeamOwners;

struct AttnSeamParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* norm_w;
  uint8_t* x8;
  uint8_t* x8c;
  float* ys;  // optional fp32 norm outputs
  int H;
  float eps;
};

// The 8 fp32 norm outputs of one octet -> 8 E4M3 bytes; the group's code
// from the 4 lanes 4a .. 4a + 3 (all 32 lanes call this together).
__device__ __forceinline__ uint2 quant_octet_f32(const float* y, int* code_out) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(y[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int code = mx_code(amax);
  const float mul = mx_mul(code);
  uint2 q;
  q.x = static_cast<uint32_t>(e4m3x2(clamp_e4m3(y[0] * mul), clamp_e4m3(y[1] * mul))) |
        (static_cast<uint32_t>(e4m3x2(clamp_e4m3(y[2] * mul), clamp_e4m3(y[3] * mul))) << 16);
  q.y = static_cast<uint32_t>(e4m3x2(clamp_e4m3(y[4] * mul), clamp_e4m3(y[5] * mul))) |
        (static_cast<uint32_t>(e4m3x2(clamp_e4m3(y[6] * mul), clamp_e4m3(y[7] * mul))) << 16);
  *code_out = code;
  return q;
}

__global__ void __launch_bounds__(kThreads) attn_seam_kernel(const AttnSeamParams p) {
  const int t = blockIdx.x;
  const int H = p.H;
  const int noct = H >> 3;
  const int tid = threadIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
  const uint4* wr = reinterpret_cast<const uint4*>(p.norm_w);
  uint4 wraw[kSeamMaxOct];
#pragma unroll
  for (int i = 0; i < kSeamMaxOct; ++i) {
    const int o = tid + i * kThreads;
    wraw[i] = o < noct ? wr[o] : make_uint4(0, 0, 0, 0);
  }
  ptx::griddep_wait();  // x may come from the previous kernel on the stream
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
    float w[8], y[8];
    unpack_bf16x8(wraw[i], w);
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = (v[i][j] * r) * w[j];  // zero past the row
    int code;
    const uint2 q = quant_octet_f32(y, &code);
    if (o < noct) {
      reinterpret_cast<uint2*>(p.x8 + row)[o] = q;
      if ((o & 3) == 0) p.x8c[static_cast<size_t>(t) * (H >> 5) + (o >> 2)] = static_cast<uint8_t>(code);
      if (p.ys) {
        float4* d = reinterpret_cast<float4*>(p.ys + row + 8 * static_cast<size_t>(o));
        d[0] = make_float4(y[0], y[1], y[2], y[3]);
        d[1] = make_float4(y[4], y[5], y[6], y[7]);
      }
    }
  }
}

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_attn_seam_x8(const void* x, const void* norm_w, int M, int hidden, float eps,
                                uint8_t* x8, uint8_t* x8_codes, float* ys, void* stream) {
  using namespace moe;
  if (!x || !norm_w || !x8 || !x8_codes) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(norm_w, 16) || !aligned(x8, 16) || (ys && !aligned(ys, 16)))
    return MOE_ERR_ALIGN;
  if (M < 1 || M > kMaxTokens) return MOE_ERR_RANGE;
  if (hidden % 32 || hidden < 32 || hidden > 8 * kSeamOwners * kSeamMaxOct)
    return MOE_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f)) return MOE_ERR_ARG;
  AttnSeamParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.norm_w = static_cast<const __nv_bfloat16*>(norm_w);
  p.x8 = x8;
  p.x8c = x8_codes;
  p.ys = ys;
  p.H = hidden;
  p.eps = eps;
  const cudaError_t e = launch_pdl(attn_seam_kernel, dim3(M), dim3(kThreads), 0,
                                   static_cast<cudaStream_t>(stream), p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
