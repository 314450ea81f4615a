// Allocation-free routing entry point: the router kernels (gate GEMV, then
// sigmoid, bias-adjusted top-k and normalised weights) run with their scratch
// in a fixed file-scope device array instead of memory the library allocates.
//
// Who needs this: callers that may not allocate device memory at the time
// they route. A serving engine that hands all GPU memory to its own pool, or
// that plans every buffer before it starts, cannot let a library call
// cudaMalloc behind its back; code that runs while a CUDA graph is being
// captured cannot call cudaMalloc at all (the call is illegal there and breaks
// the capture); and a caller that only wants routing decisions for rows it has
// already normalised does not want a whole moe_create handle, which allocates
// the full step's scratch. Here the caller passes its inputs and outputs and
// nothing is allocated.
//
// The array is a static __device__ object of kStaticScratchBytes: every GPU
// that loads the library holds it until the process exits. Host code may not
// use the array's name as a device address (on the host it names a stand-in
// object), so the device address is looked up once per device with
// cudaGetSymbolAddress and handed to the kernel.
#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 256 * 1024;
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices];
bool g_ready[kMaxDevices];

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// First call on a device (that device current): find the array's device
// address and raise the router kernel's shared-memory limit. The address is
// kept for the life of the process: a cudaDeviceReset, which unloads the
// library's device code, makes it stale, so calls after a reset are not
// supported.
int device_scratch(int dev, void** addr) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  if (!g_ready[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    e = moe::router_setup();
    if (e != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_addr[dev] = p;
    g_ready[dev] = true;
  }
  *addr = g_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_static(const void* normed, const void* gate_w, const float* bias, int M,
                                int hidden, int experts, int topk, int32_t* topk_ids,
                                float* topk_w, void* stream) {
  using namespace moe;
  if (!normed || !gate_w || !bias || !topk_ids || !topk_w) return MOE_ERR_ARG;
  if (!aligned(normed, 16) || !aligned(gate_w, 16) || !aligned(bias, 4) ||
      !aligned(topk_ids, 4) || !aligned(topk_w, 4))
    return MOE_ERR_ALIGN;
  if (M < 1 || M > kMaxTokens) return MOE_ERR_RANGE;
  if (hidden % 128 || hidden < 256 || hidden > 8192) return MOE_ERR_UNSUPPORTED;
  if (experts % 32 || experts < 32 || experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (topk < 1 || topk > kMaxTopk || topk > experts) return MOE_ERR_UNSUPPORTED;

  const int ks = router_ksplit(hidden, experts);

  // layout inside the static array; refuse problems that do not fit
  const size_t o_ctr = 0;
  const size_t o_rw = o_ctr + align256(kCtrWords * 4);
  const size_t o_sl = o_rw + align256(static_cast<size_t>(M) * topk * 4);
  const size_t o_cn = o_sl + align256(static_cast<size_t>(M) * topk * 4);
  const size_t o_id = o_cn + align256(static_cast<size_t>(experts + 1) * 4);
  const size_t o_lp = o_id + align256(static_cast<size_t>(M) * topk * 4);
  const size_t need = o_lp + align256(static_cast<size_t>(ks) * M * experts * 4);
  if (need > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  void* base_v = nullptr;
  const int rc = device_scratch(dev, &base_v);
  if (rc != MOE_OK) return rc;
  uint8_t* base = static_cast<uint8_t*>(base_v);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // the error word and the per-expert row counters must start at zero; the
  // array keeps whatever the previous call left
  if (cudaMemsetAsync(base + o_ctr, 0, kCtrWords * 4, st) != cudaSuccess ||
      cudaMemsetAsync(base + o_cn, 0, static_cast<size_t>(experts + 1) * 4, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  RouterParams rp;
  rp.normed = static_cast<const __nv_bfloat16*>(normed);
  rp.gate_w = static_cast<const __nv_bfloat16*>(gate_w);
  rp.logit_part = reinterpret_cast<float*>(base + o_lp);
  rp.x = nullptr;  // the rows come normalised
  rp.norm_w = nullptr;
  rp.x8 = rp.x8c = rp.xpan_shared = nullptr;
  rp.dbg_normed = nullptr;
  rp.dbg_x8 = rp.dbg_x8c = nullptr;
  rp.eps = 0.0f;
  rp.pf_ptr[0] = rp.pf_ptr[1] = nullptr;  // nothing to prefetch
  for (int r = 0; r < 4; ++r) {  // the memsets above clear the counters
    rp.clear[r] = nullptr;
    rp.clear_n[r] = 0;
  }
  rp.err = reinterpret_cast<int*>(base + o_ctr) + kCtrErr;
  rp.zero_rows = nullptr;
  rp.zero_n = 0;
  rp.pf_bytes[0] = rp.pf_bytes[1] = 0;
  rp.M = M;
  rp.H = hidden;
  rp.E = experts;
  rp.KS = ks;
  rp.Hs = hidden / ks;
  TopkParams tp;
  tp.logit_part = rp.logit_part;
  tp.bias = bias;
  tp.counters = reinterpret_cast<int*>(base + o_ctr);
  tp.ids = reinterpret_cast<int*>(base + o_id);
  tp.route_w = reinterpret_cast<float*>(base + o_rw);
  tp.slots = reinterpret_cast<int*>(base + o_sl);
  tp.cnt = reinterpret_cast<int*>(base + o_cn);
  tp.x8 = nullptr;
  tp.x8c = nullptr;
  tp.xpan = nullptr;
  tp.picks_early = nullptr;
  tp.H = hidden;
  tp.dbg_ids = topk_ids;
  tp.dbg_w = topk_w;
  tp.dbg_logits = nullptr;
  tp.M = M;
  tp.E = experts;
  tp.K = topk;
  tp.KS = ks;
  if (launch_router(rp, st) != cudaSuccess || launch_topk(tp, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

extern "C" int moe_route_static_status(void* stream) {
  using namespace moe;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CAPTURE;
  }
  if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_CAPTURE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    if (!g_ready[dev]) return MOE_OK;  // no call has run on this device
    base = g_addr[dev];
  }
  // the error word is the first counter word of the array (see the layout in
  // moe_route_static); read it behind the calls already enqueued on the stream
  int word = 0;
  if (cudaMemcpyAsync(&word, static_cast<int*>(base) + kCtrErr, 4, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word & kErrBounds) return MOE_ERR_ARG;
  return MOE_OK;
}
