// The C ABI (include/moe_decode.h): handle creation with the whole scratch
// allocated up front, the step as a fixed sequence of kernel launches on the
// caller's stream, and the status / timing helpers.
//
// "vllm.models.deepseek_v41.amd.mono.runner": DSV41MonoLayer.ffn (the step),
// supports (1 <= M <= MAX_TOKENS), scratch (allocated before any capture;
// here all widths share one scratch sized for max_tokens), _check_tensors
// (inputs are validated because the kernels' loads are unbounded).
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.cuh"

using namespace moe;

struct moe_handle {
  moe_config cfg;
  moe_weights w;
  int device;
  int num_sms;
  int ks, hs;
  int units_max, rows_max;
  uint8_t* scratch;
  size_t scratch_bytes;
  int* counters;
  ActiveExpert* act;
  float* route_w;
  int* tok_pos;
  int* slots;
  int* cnt;
  __nv_bfloat16* normed;
  uint8_t* x8;
  uint8_t* x8c;
  float* logit_part;
  int* ids;
  uint8_t* xpan;
  uint8_t* hpan;
  float* part;
  uint4* sfa13;
  uint4* sfa2;
  ExpertParams pe;
  int* ready;
  int* picks_early;  // [1 + kPickPrefetchMaxM * k]: the published-picks count, then the picks
  cudaEvent_t events[16];
  int n_events;
  cudaStream_t last_stream;
  int withhold_unit;  // test hook (moe_test_withhold_ready): -1 = off
};

namespace {

const char* const kKernelNames[] = {"seam", "router", "topk", "experts", "combine"};
constexpr int kNumKernels = 5;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int cuda_code(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  if (e == cudaErrorStreamCaptureUnsupported || e == cudaErrorStreamCaptureInvalidated ||
      e == cudaErrorStreamCaptureImplicit || e == cudaErrorStreamCaptureWrongThread)
    return MOE_ERR_CAPTURE;
  return MOE_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Element type of a weight tensor map: E4M3 bytes, or E2M1 pairs (two 4-bit
// codes per byte in global memory) that the copy spreads into 16-byte
// shared-memory units of 16 codes (8 bytes of codes, 8 bytes of gap): the
// operand form the tensor cores read for an E2M1 matrix, one byte per element
// of shared memory like E4M3 (so the stage's layout and descriptors are the same).
struct WeightType {
  CUtensorMapDataType dt;
  uint64_t bytes_num, bytes_den;  // global bytes per element = num / den
};
constexpr WeightType kE4M3Map = {CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 1};
constexpr WeightType kE2M1Map = {CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 1, 2};

// 2D matrix [rows][cols] (cols elements per row), box = 128 elements x
// box_rows, 128-byte swizzle (the layout the MMA's shared-memory descriptors describe).
bool encode_rows(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                 uint32_t box_rows, WeightType wt = kE4M3Map) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * wt.bytes_num / wt.bytes_den};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStageK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, wt.dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D tensor [planes][rows][cols], box = 128 elements x box_rows x box_planes,
// 128-byte swizzle.
bool encode_planes(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t planes, uint32_t box_rows, uint32_t box_planes,
                   WeightType wt = kE4M3Map) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const uint64_t row_bytes = cols * wt.bytes_num / wt.bytes_den;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {row_bytes, rows * row_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kStageK), box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, wt.dt, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int validate_config(const moe_config* c) {
  if (c->hidden <= 0 || c->experts <= 0 || c->topk <= 0 || c->inter <= 0 ||
      c->shared_inter <= 0 || c->max_tokens <= 0 || !(c->eps >= 0.0f))
    return MOE_ERR_ARG;
  if (c->hidden % 128 || c->hidden < 256 || c->hidden > 8192) return MOE_ERR_UNSUPPORTED;
  if (c->experts % 32 || c->experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (c->topk > kMaxTopk || c->topk > c->experts) return MOE_ERR_UNSUPPORTED;
  if (c->inter % 128 || c->inter < 256 || c->inter > 8192 || c->shared_inter != c->inter)
    return MOE_ERR_UNSUPPORTED;
  if (c->max_tokens > kMaxTokens) return MOE_ERR_UNSUPPORTED;
  if (c->routed_format != MOE_ROUTED_E4M3 && c->routed_format != MOE_ROUTED_E2M1)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int validate_weights(const moe_weights* w, int routed_format) {
  const void* ptrs[] = {w->norm_w, w->gate_w, w->bias, w->w13, w->w13_s, w->w2,
                        w->w2_s,   w->sw13,   w->sw13_s, w->sw2, w->sw2_s};
  for (const void* p : ptrs) {
    if (!p) return MOE_ERR_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  }
  // the 4-bit tensor copies want 32-byte aligned bases
  if (routed_format == MOE_ROUTED_E2M1 && ((reinterpret_cast<uintptr_t>(w->w13) & 31) ||
                                           (reinterpret_cast<uintptr_t>(w->w2) & 31)))
    return MOE_ERR_ALIGN;
  return MOE_OK;
}

// Small steps run the seam inside the router kernel: every router CTA makes
// its K-slice of the normed rows (whole 32-column groups).
bool seam_fused(const moe_handle* h, int M) { return M <= kSeamFuseMaxM && h->hs % 32 == 0; }

// Makes a device current for the lifetime of the object and gives the caller
// back its own current device afterwards (host-side calls that synchronise or
// copy on the handle's device leave no trace in the calling thread's state).
class DeviceScope {
 public:
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      prev_ = -1;
    }
    ok_ = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceScope() {
    if (prev_ >= 0) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = false;
};

}  // namespace

extern "C" {

int moe_kernel_count(void) { return kNumKernels; }

int moe_step_launches(const moe_handle* h, int M) {
  if (!h || M < 1 || M > h->cfg.max_tokens) return 0;
  return seam_fused(h, M) ? kNumKernels - 1 : kNumKernels;
}

const char* moe_kernel_name(int i) {
  return (i >= 0 && i < kNumKernels) ? kKernelNames[i] : nullptr;
}

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_RANGE: return "token count outside [1, max_tokens]";
    case MOE_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_CAPTURE: return "not allowed during stream capture";
    case MOE_ERR_TIMEOUT: return "a bounded device wait expired";
    case MOE_ERR_UNSUPPORTED: return "configuration not supported";
    case MOE_ERR_DEVICE: return "device is not compute capability 10.3";
    default: return "unknown error";
  }
}

size_t moe_scratch_bytes(const moe_handle* h) { return h ? h->scratch_bytes : 0; }

int moe_scratch_region(const moe_handle* h, int region, void** ptr, size_t* bytes) {
  if (!h || !ptr || !bytes) return MOE_ERR_ARG;
  const size_t H = h->cfg.hidden, I = h->cfg.inter, K = h->cfg.topk;
  switch (region) {
    case MOE_REGION_GATHERED:
      *ptr = h->xpan;
      *bytes = static_cast<size_t>(h->cfg.experts + 1) * (H / 128) * kPanelPitch;
      return MOE_OK;
    case MOE_REGION_H8:
      *ptr = h->hpan;
      *bytes = static_cast<size_t>(h->units_max) * (I / 128) * kPanelPitch;
      return MOE_OK;
    case MOE_REGION_PARTIAL:
      *ptr = h->part;
      *bytes = static_cast<size_t>(h->rows_max) * H * 4;
      return MOE_OK;
    case MOE_REGION_ACTIVE:
      *ptr = h->act;
      *bytes = static_cast<size_t>(h->cfg.experts + 1) * sizeof(ActiveExpert);
      return MOE_OK;
    case MOE_REGION_TOKPOS:
      *ptr = h->tok_pos;
      *bytes = static_cast<size_t>(h->cfg.max_tokens) * (K + 1) * 4;
      return MOE_OK;
    default:
      return MOE_ERR_ARG;
  }
}

int moe_create(const moe_config* cfg, const moe_weights* w, int device, moe_handle** out) {
  if (!cfg || !w || !out) return MOE_ERR_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  rc = validate_weights(w, cfg->routed_format);
  if (rc) return rc;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return ndev == 0 ? MOE_ERR_CUDA : MOE_ERR_ARG;
  }
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return MOE_ERR_DEVICE;
  if (!get_encode_fn()) return MOE_ERR_CUDA;
  // one expert CTA (384 threads, 448 with MXFP4 routed experts; ~216 KB of shared
  // memory) must fit an SM
  {
    int per_sm = 0;
    const cudaError_t e =
        expert_occupancy(cfg->routed_format == MOE_ROUTED_E2M1 ? 1 : 0, &per_sm);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  }

  moe_handle* h = new (std::nothrow) moe_handle();
  if (!h) return MOE_ERR_CUDA;
  std::memset(h, 0, sizeof(*h));
  h->cfg = *cfg;
  h->w = *w;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->withhold_unit = -1;

  const int H = cfg->hidden, E = cfg->experts, K = cfg->topk, I = cfg->inter;
  const int Mx = cfg->max_tokens;
  const int ks = router_ksplit(H, E);
  h->ks = ks;
  h->hs = H / ks;
  h->rows_max = Mx * (K + 1);
  h->units_max = (E < Mx * K ? E : Mx * K) + 1;
  const int g13 = H / 128, g2 = I / 128, t13 = I / 64, t2 = H / 128;

  size_t off = 0;
  auto place = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes, 1024);
    return o;
  };
  const size_t o_ctr = place(kCtrWords * 4);
  const size_t o_act = place(static_cast<size_t>(E + 1) * sizeof(ActiveExpert));
  const size_t o_rw = place(static_cast<size_t>(Mx) * K * 4);
  const size_t o_tp = place(static_cast<size_t>(Mx) * (K + 1) * 4);
  const size_t o_sl = place(static_cast<size_t>(Mx) * K * 4);
  const size_t o_cn = place(static_cast<size_t>(E + 1) * 4);
  const size_t o_nm = place(static_cast<size_t>(Mx) * H * 2);
  const size_t o_x8 = place(static_cast<size_t>(Mx) * H);
  const size_t o_x8c = place(static_cast<size_t>(Mx) * H / 32);
  const size_t o_lp = place(static_cast<size_t>(ks) * Mx * E * 4);
  const size_t o_id = place(static_cast<size_t>(Mx) * K * 4);
  const size_t o_xp = place(static_cast<size_t>(E + 1) * g13 * kPanelPitch);  // by expert id
  const size_t o_hp = place(static_cast<size_t>(h->units_max) * g2 * kPanelPitch);
  const size_t o_pa = place(static_cast<size_t>(h->rows_max) * H * 4);
  const size_t o_a13 = place(static_cast<size_t>(E + 1) * t13 * g13 * 16);
  const size_t o_a2 = place(static_cast<size_t>(E + 1) * t2 * g2 * 16);
  const size_t o_rd = place(static_cast<size_t>(E + 1) * 4);
  const size_t o_pk = place(static_cast<size_t>(1 + kPickPrefetchMaxM * K) * 4);
  const bool fp4 = cfg->routed_format == MOE_ROUTED_E2M1;
  // MXFP4 routed experts: per-row scale images, 32 x 16 bytes per (tile, stage)
  const size_t o_i13 = fp4 ? place(static_cast<size_t>(E) * t13 * g13 * 512) : 0;
  const size_t o_i2 = fp4 ? place(static_cast<size_t>(E) * t2 * g2 * 512) : 0;
  h->scratch_bytes = off;

  cudaError_t err = cudaMalloc(&h->scratch, h->scratch_bytes);
  if (err != cudaSuccess) {
    rc = cuda_code(err);
    cudaGetLastError();
    delete h;
    return rc;
  }
  uint8_t* b = h->scratch;
  h->counters = reinterpret_cast<int*>(b + o_ctr);
  h->act = reinterpret_cast<ActiveExpert*>(b + o_act);
  h->route_w = reinterpret_cast<float*>(b + o_rw);
  h->tok_pos = reinterpret_cast<int*>(b + o_tp);
  h->slots = reinterpret_cast<int*>(b + o_sl);
  h->cnt = reinterpret_cast<int*>(b + o_cn);
  h->normed = reinterpret_cast<__nv_bfloat16*>(b + o_nm);
  h->x8 = b + o_x8;
  h->x8c = b + o_x8c;
  h->logit_part = reinterpret_cast<float*>(b + o_lp);
  h->ids = reinterpret_cast<int*>(b + o_id);
  h->xpan = b + o_xp;
  h->hpan = b + o_hp;
  h->part = reinterpret_cast<float*>(b + o_pa);
  h->sfa13 = reinterpret_cast<uint4*>(b + o_a13);
  h->sfa2 = reinterpret_cast<uint4*>(b + o_a2);
  h->ready = reinterpret_cast<int*>(b + o_rd);
  h->picks_early = reinterpret_cast<int*>(b + o_pk);
  uint4* img13 = fp4 ? reinterpret_cast<uint4*>(b + o_i13) : nullptr;
  uint4* img2 = fp4 ? reinterpret_cast<uint4*>(b + o_i2) : nullptr;

  err = cudaMemset(h->scratch, 0, h->scratch_bytes);
  if (err == cudaSuccess) err = router_setup();
  if (err == cudaSuccess) err = expert_kernel_setup();
  if (err == cudaSuccess) {
    SfaPackParams sp;
    sp.w13_s = w->w13_s;
    sp.sw13_s = w->sw13_s;
    sp.w2_s = w->w2_s;
    sp.sw2_s = w->sw2_s;
    sp.sfa13 = h->sfa13;
    sp.sfa2 = h->sfa2;
    sp.img13 = img13;
    sp.img2 = img2;
    sp.fp4 = fp4 ? 1 : 0;
    sp.E = E;
    sp.H = H;
    sp.I = I;
    err = launch_sfa_pack(sp, 0);
  }
  if (err == cudaSuccess) err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    rc = cuda_code(err);
    cudaGetLastError();
    cudaFree(h->scratch);
    delete h;
    return rc;
  }

  // the expert kernel's parameter block (fixed for the handle's lifetime)
  ExpertParams& pe = h->pe;
  pe.cnt = h->cnt;
  pe.counters = h->counters;
  pe.act = h->act;
  pe.sfa13 = h->sfa13;
  pe.sfa2 = h->sfa2;
  pe.img13 = img13;
  pe.img2 = img2;
  pe.fp4 = fp4 ? 1 : 0;
  pe.xpan = h->xpan;
  pe.hpan = h->hpan;
  pe.part = h->part;
  pe.ready = h->ready;
  pe.err = h->counters + kCtrErr;
  pe.task_ctr = h->counters + kCtrTasks;
  pe.E = E;
  pe.inter = I;
  pe.hidden = H;
  pe.t13 = t13;
  pe.g13 = g13;
  pe.t2 = t2;
  pe.g2 = g2;
  pe.units_max = h->units_max;
  pe.rows_max = h->rows_max;
  pe.withhold_unit = -1;
  // w13 as [2E halves][I rows][H]: one box = 64 gate rows over the 64 matching up rows
  const WeightType wt = fp4 ? kE2M1Map : kE4M3Map;
  bool ok = encode_planes(&pe.tm_w13, w->w13, H, I, 2ull * E, 64, 2, wt) &&
            encode_planes(&pe.tm_w13_shared, w->sw13, H, I, 2, 64, 2) &&
            encode_rows(&pe.tm_w2, w->w2, I, static_cast<uint64_t>(E) * H, kTileM, wt) &&
            encode_rows(&pe.tm_w2_shared, w->sw2, I, static_cast<uint64_t>(H), kTileM);
  if (!ok) {
    cudaFree(h->scratch);
    delete h;
    return MOE_ERR_CUDA;
  }
  *out = h;
  return MOE_OK;
}

int moe_decode_step(moe_handle* h, const void* x, int M, void* out, void* stream,
                    const moe_debug* dbg) {
  if (!h) return MOE_ERR_ARG;
  if (M < 1 || M > h->cfg.max_tokens) return MOE_ERR_RANGE;
  if (!x || !out) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(out)) return MOE_ERR_ALIGN;
  moe_debug d;
  std::memset(&d, 0, sizeof(d));
  if (dbg) d = *dbg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  const int H = h->cfg.hidden, E = h->cfg.experts, K = h->cfg.topk;
  // per-kernel events (kNumKernels + 1), or two that bracket the step
  const bool timed = h->n_events == kNumKernels + 1 || h->n_events == 2;
  cudaError_t err = cudaSuccess;
  // under stream capture a plain record only adds a dependency; an external
  // record becomes an event-record node that fires at every graph replay
  unsigned int rec_flags = cudaEventRecordDefault;
  if (timed) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    err = cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) {
    if (!timed || err != cudaSuccess) return;
    if (h->n_events == 2) {  // the step's start and end only
      if (i == 0 || i == kNumKernels) err = cudaEventRecordWithFlags(h->events[i ? 1 : 0], st, rec_flags);
      return;
    }
    err = cudaEventRecordWithFlags(h->events[i], st, rec_flags);
  };

  SeamParams sp;
  sp.x = static_cast<const __nv_bfloat16*>(x);
  sp.norm_w = static_cast<const __nv_bfloat16*>(h->w.norm_w);
  sp.normed = h->normed;
  sp.x8 = h->x8;
  sp.x8c = h->x8c;
  sp.dbg_normed = static_cast<__nv_bfloat16*>(d.normed);
  sp.dbg_x8 = d.x8;
  sp.dbg_x8c = d.x8_codes;
  sp.xpan_shared = h->xpan + static_cast<size_t>(E) * (H / 128) * kPanelPitch;
  sp.H = H;
  sp.eps = h->cfg.eps;

  // Small steps run the seam inside the router kernel (each router CTA makes
  // its K-slice of the normed rows): one kernel boundary and one pass over
  // the normed rows less on the way to the experts.
  const bool fuse_seam = seam_fused(h, M);
  RouterParams rp;
  rp.normed = h->normed;
  rp.x = fuse_seam ? sp.x : nullptr;
  rp.norm_w = sp.norm_w;
  rp.x8 = sp.x8;
  rp.x8c = sp.x8c;
  rp.xpan_shared = sp.xpan_shared;
  rp.dbg_normed = sp.dbg_normed;
  rp.dbg_x8 = sp.dbg_x8;
  rp.dbg_x8c = sp.dbg_x8c;
  rp.eps = sp.eps;
  rp.gate_w = static_cast<const __nv_bfloat16*>(h->w.gate_w);
  rp.logit_part = h->logit_part;
  rp.M = M;
  rp.H = H;
  rp.E = E;
  rp.KS = h->ks;
  rp.Hs = h->hs;
  // Small steps: the shared expert's weights go to L2 while the routing runs
  // (at larger M the prefetch slows the top-k kernel about as much as it
  // saves in the expert kernel).
  // the previous step's readers of the row counts, readiness counts and task
  // counter are done once the router's grid dependency is met
  rp.clear[0] = h->cnt;
  rp.clear_n[0] = E;
  rp.clear[1] = h->ready;
  rp.clear_n[1] = h->units_max;
  rp.clear[2] = h->counters + kCtrTasks;
  rp.clear_n[2] = 1;
  // (small steps with E4M3 routed experts; measured no gain with MXFP4 ones)
  const bool pick_pf = M <= kPickPrefetchMaxM && h->cfg.routed_format == MOE_ROUTED_E4M3;
  rp.clear[3] = pick_pf ? h->picks_early : nullptr;  // the published-picks count
  rp.clear_n[3] = 1;
  // small steps: the last round of w2 tiles runs as K-halves added into the
  // step's partial rows, which start at zero
  const int g2 = h->cfg.inter / 128;
  const bool split = M <= kW2SplitMaxM && g2 >= 4 && g2 % 2 == 0;
  rp.err = h->counters + kCtrErr;
  rp.zero_rows = split ? h->part : nullptr;
  rp.zero_n = split ? static_cast<size_t>(M) * (K + 1) * H : 0;
  const bool pf = M <= kPrefetchMaxM;
  rp.pf_ptr[0] = pf ? static_cast<const uint8_t*>(h->w.sw13) : nullptr;  // [2 I][H] e4m3
  rp.pf_bytes[0] = pf ? 2ull * h->cfg.inter * H : 0;
  rp.pf_ptr[1] = pf ? static_cast<const uint8_t*>(h->w.sw2) : nullptr;  // [H][I] e4m3
  rp.pf_bytes[1] = pf ? static_cast<uint64_t>(H) * h->cfg.inter : 0;

  TopkParams tp;
  tp.logit_part = h->logit_part;
  tp.bias = h->w.bias;
  tp.counters = h->counters;
  tp.ids = h->ids;
  tp.route_w = h->route_w;
  tp.slots = h->slots;
  tp.cnt = h->cnt;
  tp.x8 = h->x8;
  tp.x8c = h->x8c;
  tp.xpan = h->xpan;
  tp.picks_early = pick_pf ? h->picks_early : nullptr;
  tp.H = H;
  tp.dbg_ids = d.topk_ids;
  tp.dbg_w = d.topk_w;
  tp.dbg_logits = d.logits;
  tp.M = M;
  tp.E = E;
  tp.K = K;
  tp.KS = h->ks;

  CombineParams cp;
  cp.part = h->part;
  cp.route_w = h->route_w;
  cp.ids = h->ids;
  cp.slots = h->slots;
  cp.cnt = h->cnt;
  cp.tok_pos = h->tok_pos;
  cp.out = static_cast<__nv_bfloat16*>(out);
  cp.M = M;
  cp.H = H;
  cp.K = K;
  cp.E = E;

  mark(0);
  if (err == cudaSuccess && !fuse_seam) err = launch_seam(sp, M, st);
  mark(1);
  if (err == cudaSuccess) err = launch_router(rp, st);
  mark(2);
  if (err == cudaSuccess) err = launch_topk(tp, st);
  mark(3);
  ExpertParams pe = h->pe;
  pe.M = M;
  pe.K = K;
  pe.withhold_unit = h->withhold_unit;
  pe.picks_early = pick_pf ? h->picks_early : nullptr;
  pe.split_tiles = split ? h->num_sms : 0;
  if (err == cudaSuccess) err = launch_experts(pe, h->num_sms, st);
  mark(4);
  if (err == cudaSuccess) err = launch_combine(cp, st);
  mark(5);
  return cuda_code(err);
}

int moe_status(moe_handle* h) {
  if (!h) return MOE_ERR_ARG;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(h->last_stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CAPTURE;
  }
  if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_CAPTURE;
  DeviceScope scope(h->device);
  if (!scope.ok()) return MOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, h->counters + kCtrErr, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word & kErrBounds) return MOE_ERR_ARG;
  return MOE_OK;
}

int moe_clear_status(moe_handle* h) {
  if (!h) return MOE_ERR_ARG;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(h->last_stream, &cs) != cudaSuccess ||
      cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return MOE_ERR_CAPTURE;
  }
  DeviceScope scope(h->device);
  if (!scope.ok()) return MOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(h->counters + kCtrErr, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_last_unique_experts(moe_handle* h, int* unique_routed) {
  if (!h || !unique_routed) return MOE_ERR_ARG;
  DeviceScope scope(h->device);
  if (!scope.ok()) return MOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, h->counters + kCtrRouted, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  *unique_routed = v;
  return MOE_OK;
}

int moe_test_withhold_ready(moe_handle* h, int unit) {
  if (!h) return MOE_ERR_ARG;
  if (unit < -1 || unit >= h->units_max) return MOE_ERR_RANGE;
  h->withhold_unit = unit;
  return MOE_OK;
}

int moe_set_timing_events(moe_handle* h, void* const* events, int n) {
  if (!h) return MOE_ERR_ARG;
  if (!events || n == 0) {
    h->n_events = 0;
    return MOE_OK;
  }
  if (n != kNumKernels + 1 && n != 2) return MOE_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return MOE_ERR_ARG;
    h->events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  h->n_events = n;
  return MOE_OK;
}

void moe_destroy(moe_handle* h) {
  if (!h) return;
  {
    DeviceScope scope(h->device);
    if (scope.ok()) {
      cudaDeviceSynchronize();
      cudaFree(h->scratch);
    }
  }
  cudaGetLastError();
  delete h;
}

}  // extern "C"
