// Grouped-expert kernel: block-scaled E4M3 GEMMs of the active experts on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), persistent over
// the step's tasks -- first every w13 task, then every w2 task -- in one launch.
//
// "vllm.models.deepseek_v41.amd.mono.attention.device", mfma_scaled: the
// expert GEMMs are block-scaled MMAs whose operands are both MX-FP8 with one
// E8M0 per 32-K block per row. "vllm.models.deepseek_v41.amd.mono.runner",
// MonoLayerWeights: gate_up [2 inter, 5120] e4m3 with [2 inter / 32, 160]
// E8M0 (32 x 32 blocks), down [5120, inter] with [160, inter / 32].
//
// Swap-AB: the weight rows are the MMA's M (128 per tile) and the unit's
// tokens its N (rounded up to 16, at most 48), so the weights stream once
// through shared memory while the few activation rows are reused from L2.
//
//  w13 task = (unit, 64 intermediate columns): A = the 64 gate rows over the
//    matching 64 up rows of w13 (one 3D TMA box), B = the unit's MXFP8 token
//    rows (its expert's x panels, written by the top-k kernel), K = H. Epilogue: silu(g) * u,
//    requantised per token in 32-column groups (the seam's mx_code / E4M3
//    rule) straight into the unit's h panels (rows and scale images); then
//    the unit's readiness counter +1 (one device-scope release per tile).
//  w2 task = (unit, 128 hidden rows): A = w2 rows, B = the unit's h panels,
//    K = I. Its weight stages are issued at once; its activation stages wait
//    (bounded) until all w13 tiles of the unit are done. Epilogue: fp32 rows
//    of y for the combine.
// Tasks are handed out in that order from a global counter, every CTA's
// first task included. Every w13 task is handed out before any w2 task, to a
// CTA that is running and finishes it without waiting on anything, so the
// readiness waits always end, however many of the grid's CTAs are resident
// at once.
//
// Per CTA (one per SM, 384 threads; 448 with MXFP4 routed experts):
//  warp 8 lane 0, the scheduler, claims the CTA's tasks one ahead of the
//    producer (the next one when the producer has kClaimLead stages of the
//    current one left to issue, so that a w2 task is rarely claimed long
//    before its unit can be done), posts each id with its unit's table entry to a small queue
//    in shared memory, and for a w2 task waits (device scope) for the unit's
//    readiness and publishes it in shared memory. A device-scope wait in the
//    producer thread would also wait for its copies in flight.
//  lane 0 of warp 0 and warps 11 ..., the producers (two with E4M3 routed
//    experts, four with MXFP4), issue the loads into an 8-slot ring -- per
//    stage one weight box (TMA, evict-first from L2) and one contiguous bulk
//    copy of the activation panel (rows + scale image, already in the
//    swizzled layout the MMA reads, evict-last). Each slot belongs to one MMA
//    issuer (two slots each), which waits for every phase of it, and each
//    producer fills the slots of its issuers: a thread issuing TMA copies
//    spends a fixed time per copy, so several producers keep the ring full at
//    HBM speed.
//  warp 3 writes each stage's weight-scale image (the stage's 16-byte entry in
//    all 32 rows tcgen05.cp expects) as soon as the slot is free.
//  lane 0 of warps 1, 2, 9 and 10, the MMA issuers, share the stages of
//    every task: issuer h (warp 1, 2 -- which also owns the TMEM allocation
//    -- 9, 10) takes the K stages g with g mod 4 = h; each copies its stage's
//    two scale images into TMEM and issues 4 MMAs (K = 32 each, the
//    descriptor's scale-factor id picks the K block of the stage) into its
//    own accumulator, and the epilogue adds the partial sums in issuer order.
//    One thread needs ~530 cycles to issue a stage (about 100 per MMA, 55 per
//    scale copy), near the ~720 cycles per 16 KB stage at which one SM's
//    share of HBM arrives, and an MXFP4 stage carries half those bytes; the
//    issuers work concurrently at the same per-thread rate.
//  warps 4-7 drain the double-buffered accumulators (each reads its 32-lane
//    quarter).
//
// MXFP4 routed experts ("vllm.models.deepseek_v41.amd.mono.runner",
// MonoLayerWeights: w13 / w2 float4_e2m1fn_x2 with one E8M0 per row per 32
// columns): the weight box is a 4-bit tensor copy that spreads each 16 codes
// into a 16-byte shared-memory unit (8 bytes of codes, 8 of gap), the form
// kind::mxf8f6f4 reads for an E2M1 operand, so a stage has the same layout
// and descriptors as with E4M3 and only the instruction descriptor's A
// format changes. The per-row codes differ across all 128 rows of a tile, so
// each stage's scale image (lane i, cell c = row 32 c + i) is prepacked at
// creation and copied into the slot by the producer with the weights (the
// image warp only marks those slots ready). The shared expert stays E4M3.
// Every mbarrier and readiness wait is bounded; on a timeout the CTA records
// kErrTimeout, waits for its own copies and MMAs, frees TMEM and exits.
//
// Launched with programmatic dependent launch: the prologue (barriers, TMEM,
// tensor-map prefetch) runs while the top-k kernel finishes; the scheduler
// warp then waits for it (griddepcontrol.wait) -- the weights to stream depend
// on the routing it writes -- and every other role waits on the task queue.
#include "internal.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr uint32_t kABytes = kTileM * kStageK;           // 16 KB
constexpr uint32_t kImgBytes = 32 * 16;                  // scale image of one stage
constexpr uint32_t kBBytes = 7 * 1024;  // one activation panel (<= 48 rows + image), 1024-aligned
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffXchg = kOffSfa + kStages * kImgBytes;
constexpr uint32_t kOffBar = kOffXchg + 2 * kMaxTokens * 64 * 4;  // gate and up values
constexpr uint32_t kOffMisc = kOffBar + 512;
constexpr uint32_t kOffUnits = kOffMisc + 512;                     // packed unit entries
constexpr uint32_t kSmemUsed = kOffUnits + ((kMaxExperts + 1) * 4 + 15) / 16 * 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024
// MMA issuer threads per CTA: stage g of a task goes to issuer g mod kIssuers,
// each into its own accumulator, and the epilogue adds them in issuer order
// (a split that depends on g alone, so the sums are the same in every run).
// The ring's slots are owned by the issuers -- issuer h uses slots h and
// h + kIssuers in turn -- so every waiter on a slot's barriers sees each of
// its phases: with slots shared round-robin among several consumers, a
// consumer could test a slot whose previous phase it never waited for and
// take that phase's parity for the one it wants.
constexpr int kIssuers = 4;
static_assert(kStages == 2 * kIssuers, "two ring slots per issuer");
// TMA-issuing threads (producers): a thread that issues the ring's copies
// spends a fixed ~400 ns per tensor box and ~45 ns per small bulk copy
// (measured on a bare ring, whatever the box's bytes), which caps one thread
// near 3 TB/s over the GPU for the 8 KB boxes of MXFP4 weights. Measured
// there: an E4M3 stage (box + activation panel) reaches HBM speed with two
// producers, an MXFP4 stage (box + scale image + panel) only with four. Each
// producer feeds the slots of kIssuers / producers issuers. Warps: 0 the first
// producer, 1, 2, 9, 10 the issuers, 3 the scale images, 4-7 the epilogue,
// 8 the scheduler, 11 ... the other producers.
template <bool kFp4>
struct Roles {
  static constexpr int kProducers = kFp4 ? 4 : 2;
  static constexpr int kThreads = (10 + kProducers) * 32;
  static constexpr int kTaskReaders = 2 + kProducers + kIssuers;  // producers, issuers, images, epilogue
  static_assert(kIssuers % kProducers == 0, "issuers split evenly among the producers");
};
// TMEM: 2 task buffers x kIssuers issuers x 64 accumulator columns; an
// accumulator uses at most kMaxTokens columns, and ring slot s keeps its 8
// scale columns (4 for the weights, 4 for the activations) in the unused
// tail of the s-th 64-column block
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 64;
constexpr uint32_t kSfColOff = kMaxTokens;
static_assert(2 * kIssuers * kAccCols == kTmemCols, "TMEM budget");
static_assert(kSfColOff + 8 <= kAccCols, "scale columns beside the accumulator columns");
constexpr int kTaskSlots = 8;  // task-id queue from the scheduler warp to the other roles
// The producer lets the scheduler claim the next task when this many of the
// current task's stages are left to issue (the ring holds 8 more): late enough
// that a w2 task is rarely claimed before its unit can be done, early enough
// that the claim, its table read and the readiness check are over in time.
constexpr int kClaimLead = 10;

static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0, "B tiles must stay 1024-aligned");
static_assert(kBBytes >= kPanelPitch, "a panel fits its slot");
static_assert(kOffSfa % 512 == 0, "scale images alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Bars {
  uint64_t full[kStages];     // weights + activation panel landed
  uint64_t empty[kStages];    // the stage's MMAs (and scale copies) completed
  uint64_t sfa_rdy[kStages];  // the stage's weight-scale image is written
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t task_full[kTaskSlots];   // the producer posted a task id
  uint64_t task_empty[kTaskSlots];  // its readers (kTaskReaders) have taken it
};
static_assert(sizeof(Bars) <= 512, "barrier area");

struct Misc {
  int4 slot_act[kTaskSlots];  // the posted task's unit entry (expert id, first row, rows)
  int4 slot_task[kTaskSlots]; // the posted task, decoded (pack_task)
  int4 epi_act;
  int4 epi_k;
  uint32_t tmem_base;
  int abort;
  int epi_ok;
  int epi_task;
  int ready_seq;  // the last task (sequence number) whose unit's w13 tiles are all done
  int prod_seq;   // the last task (sequence number) the producer has taken
  int task_slot[kTaskSlots];
};
static_assert(sizeof(Misc) <= 512, "misc area");

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool task_valid(const int4& a, const ExpertParams& p) {
  return a.x >= 0 && a.x <= p.E && a.z >= 1 && a.z <= kMaxTokens && a.y >= 0 &&
         a.y + a.z <= p.rows_max;
}

// Lane 0 waits, the warp agrees on the outcome, then every lane observes the
// completed phase itself (returns at once) so its later reads are ordered.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = ptx::mbar_wait(bar, parity, abort, kWaitLimitNs);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok && (threadIdx.x & 31) != 0) ptx::mbar_wait(bar, parity, abort, kWaitLimitNs);
  return ok != 0;
}

// Wait used only while shutting down: bounded by time, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  int never = 0;
  ptx::mbar_wait(bar, parity, &never, kWaitLimitNs);
}

struct Task {
  int phase;   // 0: w13, 1: w2
  int u;       // unit (active expert)
  int t;       // tile within the unit
  int g0, gn;  // the task's K stages: g0 .. g0 + gn - 1
  int half;    // 1: a K-half of a w2 tile, added into rows that start at zero
};

// Task ids: every unit's w13 tiles (n13), the first w2full w2 tiles whole,
// then the remaining w2 tiles (at most one per CTA: the launch's last round)
// each as two K-halves. The halves even out the end of the launch: a CTA
// that would otherwise take one more whole tile takes half of one.
__device__ __forceinline__ Task decode_task(int task, int n13, int w2full, const ExpertParams& p) {
  Task k;
  k.g0 = 0;
  k.half = 0;
  if (task < n13) {
    k.phase = 0;
    k.u = task / p.t13;
    k.t = task - k.u * p.t13;
    k.gn = p.g13;
  } else {
    int j = task - n13;
    k.phase = 1;
    k.gn = p.g2;
    if (j >= w2full) {
      const int h = j - w2full;
      j = w2full + (h >> 1);
      k.half = 1;
      k.gn = p.g2 >> 1;
      k.g0 = (h & 1) * k.gn;
    }
    k.u = j / p.t2;
    k.t = j - k.u * p.t2;
  }
  return k;
}

// Bounded wait until *ctr >= target (acquire, device scope); then the async
// proxy (TMA) may read what the counting threads wrote.
__device__ __forceinline__ bool wait_ready(const int* ctr, int target, volatile int* abort) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  if (v < target) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
      __nanosleep(64);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if ((i & 63) == 0) {
        if (*abort) return false;
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
          *abort = 1;
          return false;
        }
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// The j-th task of this CTA: the scheduler posts its id (-1: no more tasks)
// with its unit's table entry; each reader (the producers, the issuers, the
// scale-image warp and the epilogue) takes both and frees the slot at once. A reader gets -2 when a wait gave up (the abort flag is set).
// A decoded task in 16 bytes: phase, half and tile; unit; first stage and
// stage count.
__device__ __forceinline__ int4 pack_task(const Task& k) {
  return make_int4(k.phase | (k.half << 1) | (k.t << 2), k.u, k.g0 | (k.gn << 16), 0);
}
__device__ __forceinline__ Task unpack_task(int4 v) {
  Task k;
  k.phase = v.x & 1;
  k.half = (v.x >> 1) & 1;
  k.t = v.x >> 2;
  k.u = v.y;
  k.g0 = v.z & 0xffff;
  k.gn = v.z >> 16;
  return k;
}

__device__ __forceinline__ void st_v4(volatile int4* dst, int4 v) {
  dst->x = v.x;
  dst->y = v.y;
  dst->z = v.z;
  dst->w = v.w;
}
__device__ __forceinline__ int4 ld_v4(const volatile int4* src) {
  return make_int4(src->x, src->y, src->z, src->w);
}

// The j-th task of this CTA: the scheduler posts its id (-1: no more tasks)
// with the task decoded and its unit's table entry; each of the five readers
// takes them and frees the slot at once. A reader gets -2 when a wait gave up
// (the abort flag is set).
__device__ __forceinline__ bool post_task(Bars* bars, Misc* misc, uint32_t j, int task, int4 a,
                                          int4 kt, volatile int* abort) {
  const int q = static_cast<int>(j % kTaskSlots);
  const uint32_t round = j / kTaskSlots;
  if (!ptx::mbar_wait(ptx::smem_u32(&bars->task_empty[q]), (round & 1) ^ 1, abort, kWaitLimitNs))
    return false;
  *reinterpret_cast<volatile int*>(&misc->task_slot[q]) = task;
  st_v4(&misc->slot_act[q], a);
  st_v4(&misc->slot_task[q], kt);
  ptx::mbar_arrive(ptx::smem_u32(&bars->task_full[q]));
  return true;
}

__device__ __forceinline__ int take_task(Bars* bars, Misc* misc, uint32_t j, volatile int* abort,
                                         int4* a, Task* k) {
  const int q = static_cast<int>(j % kTaskSlots);
  const uint32_t round = j / kTaskSlots;
  if (!ptx::mbar_wait(ptx::smem_u32(&bars->task_full[q]), round & 1, abort, kWaitLimitNs)) return -2;
  const int task = *reinterpret_cast<volatile int*>(&misc->task_slot[q]);
  *a = ld_v4(&misc->slot_act[q]);
  *k = unpack_task(ld_v4(&misc->slot_task[q]));
  ptx::mbar_arrive(ptx::smem_u32(&bars->task_empty[q]));
  return task;
}

__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(ptx::smem_u32(p)) : "memory");
  return v;
}

// Bounded wait until a shared-memory sequence number reaches j (the
// scheduler's readiness news, the producer's progress).
__device__ __forceinline__ bool wait_seq(const int* seq, int j, volatile int* abort) {
  if (ld_acquire_cta(seq) >= j) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(32);
    if (ld_acquire_cta(seq) >= j) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Ring slots of the stages as a role that walks every stage in order sees
// them: stage g of a task belongs to issuer h = g mod kIssuers, whose stages
// take slots h and h + kIssuers in turn; per slot, the parity of the phase to
// wait for next (its earlier uses, mod 2) and whether it was used at all.
struct SlotWalk {
  uint32_t next = 0;     // bit h: issuer h's next stage takes slot h + kIssuers
  uint32_t par = 0;      // bit s: slot s's uses so far, mod 2
  uint32_t touched = 0;  // bit s: slot s used at least once
  __device__ __forceinline__ int slot(int g) const {
    const int h = g % kIssuers;
    return h + kIssuers * static_cast<int>((next >> h) & 1u);
  }
  __device__ __forceinline__ uint32_t parity(int s) const { return (par >> s) & 1u; }
  __device__ __forceinline__ void advance(int g, int s) {
    next ^= 1u << (g % kIssuers);
    par ^= 1u << s;
    touched |= 1u << s;
  }
  // parity of the last phase armed on slot s (touched slots only)
  __device__ __forceinline__ uint32_t last_parity(int s) const { return parity(s) ^ 1u; }
};

// Small steps: the top-k kernel publishes each token's picks as soon as it has
// chosen them, while this grid is already resident and waiting for it. Lane 0
// of each epilogue warp (idle until the first accumulator is ready) waits for
// them (bounded, then gives up: only a prefetch is lost) and prefetches into
// L2 its share -- over every CTA and epilogue warp -- of the picked experts'
// first kPickPrefetchStages K stages of every w13 tile, the boxes the w13
// tasks will load first, and of their compact weight-scale entries. HBM then
// streams routed weights while the routing finishes instead of after it.
__device__ __forceinline__ void prefetch_picks(const ExpertParams& p, int q) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.picks_early) : "memory");
  if (v < p.M) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (v < p.M) {
      if (ptx::globaltimer_ns() - t0 > 20000) return;
      __nanosleep(64);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.picks_early) : "memory");
    }
  }
  const int n = p.M * p.K;
  const int S = p.g13 < kPickPrefetchStages ? p.g13 : kPickPrefetchStages;
  const int items = n * p.t13 * S;
  for (int it = static_cast<int>(blockIdx.x) * 4 + q; it < items;
       it += static_cast<int>(gridDim.x) * 4) {
    const int s = it % S, rest = it / S, t = rest % p.t13, j = rest / p.t13;
    const int e = __ldcg(p.picks_early + 1 + j);
    if (e < 0 || e >= p.E) continue;
    bool seen = false;  // an expert picked by several tokens is prefetched once
    for (int i = 0; i < j && !seen; ++i) seen = __ldcg(p.picks_early + 1 + i) == e;
    if (!seen) ptx::prefetch_tensor_3d(&p.tm_w13, s * kStageK, 64 * t, 2 * e);
  }
  // every picked expert's compact weight-scale entries (w13 and w2: one
  // contiguous range each), which the scale-image warp loads at each task's
  // start (with the weights' boxes, an HBM round trip before the first MMA of
  // a tile; on one GB300: M=1 -1.6 us, the 384-expert layer at M=1 -0.4 us):
  // pick j from CTA j
  const int j = static_cast<int>(blockIdx.x);
  if (q == 0 && j < n) {
    const int e = __ldcg(p.picks_early + 1 + j);
    bool seen = e < 0 || e >= p.E;
    for (int i = 0; i < j && !seen; ++i) seen = __ldcg(p.picks_early + 1 + i) == e;
    if (!seen) {
      const uint64_t pol = ptx::policy_evict_normal();
      const size_t n13 = static_cast<size_t>(p.t13) * p.g13, n2 = static_cast<size_t>(p.t2) * p.g2;
      ptx::prefetch_l2(p.sfa13 + e * n13, static_cast<uint32_t>(n13 * 16), pol);
      ptx::prefetch_l2(p.sfa2 + e * n2, static_cast<uint32_t>(n2 * 16), pol);
    }
  }
}

// kFp4: the routed experts are MXFP4 (E2M1 with per-row scale images); the
// E4M3 instantiation carries none of that path's code.
template <bool kFp4>
__global__ void __launch_bounds__(Roles<kFp4>::kThreads, 1)
    expert_kernel(const __grid_constant__ ExpertParams p) {
  constexpr int kProducers = Roles<kFp4>::kProducers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  volatile int* abort = &misc->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->empty[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->sfa_rdy[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&bars->tfull[a]), kIssuers);  // one commit per issuer
      ptx::mbar_init(ptx::smem_u32(&bars->tempty[a]), 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(ptx::smem_u32(&bars->drain), kIssuers);
    for (int q = 0; q < kTaskSlots; ++q) {
      ptx::mbar_init(ptx::smem_u32(&bars->task_full[q]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars->task_empty[q]), Roles<kFp4>::kTaskReaders);
    }
    misc->abort = 0;
    misc->epi_ok = 0;
    misc->epi_task = -1;
    misc->ready_seq = -1;
    misc->prod_seq = -1;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&p.tm_w13);
    ptx::prefetch_tmap(&p.tm_w13_shared);
    ptx::prefetch_tmap(&p.tm_w2);
    ptx::prefetch_tmap(&p.tm_w2_shared);
  }
  if (warp == 2) {
    ptx::tmem_alloc(ptx::smem_u32(&misc->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = misc->tmem_base;

  uint32_t* unit_s = reinterpret_cast<uint32_t*>(smem + kOffUnits);
  if (warp == 0 || warp >= 11) {
    // ------------------------------------------------------------ TMA producers
    // producer q (warp 0: q = 0, warps 11 ...: q = 1 ...) issues the stages g
    // with g mod kIssuers in [q kIssuers / kProducers, (q + 1) kIssuers /
    // kProducers), i.e. the stages of its issuers, in increasing g
    const int q = warp == 0 ? 0 : warp - 10;
    constexpr int kPerProducer = kIssuers / kProducers;
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      const uint64_t pol_x = ptx::policy_evict_last();
      SlotWalk walk;
      bool ok = true;
      // Weight stages are issued at once. A w2 task's activation stages are
      // held back (at most one ring's worth) until its unit's w13 tiles are
      // done -- which the scheduler warp finds out (a device-scope wait here
      // would also wait for this thread's copies in flight) and publishes in
      // shared memory; they go out as soon as it has.
      for (uint32_t j = 0; ok; ++j) {
        int4 a;
        Task k;
        const int task = take_task(bars, misc, j, abort, &a, &k);
        if (task < 0) break;  // -1: no more tasks; -2: a wait gave up
        const int nt = (a.z + 15) & ~15;
        const uint32_t pbytes = kPanelRows + nt * 128;  // the panel's used part
        const bool shared_e = a.x == p.E;
        // MXFP4 routed weights: a 4-bit weight box counts its global bytes
        // (two codes per byte), half of what it fills in shared memory
        const bool fp4 = kFp4 && !shared_e;
        const uint32_t bytes = (fp4 ? kABytes / 2 + kImgBytes : kABytes) + pbytes;
        const int G = k.gn;
        const int panels = k.phase ? p.g2 : p.g13;  // per unit (h) or expert (x)
        // x panels are kept per expert id (a lone token's experts all read
        // the shared expert's: its single row), h panels per unit
        const int xe = p.M == 1 ? p.E : a.x;
        const uint8_t* pan =
            (k.phase ? p.hpan + static_cast<size_t>(k.u) * panels * kPanelPitch
                     : p.xpan + static_cast<size_t>(xe) * panels * kPanelPitch) +
            static_cast<size_t>(k.g0) * kPanelPitch;
        auto issue_b = [&](int g, int s) {
          ptx::bulk_load(ptx::smem_u32(smem + kOffB + s * kBBytes), pan + g * kPanelPitch, pbytes,
                         ptx::smem_u32(&bars->full[s]), pol_x);
        };
        bool b_ok = k.phase == 0;
        int n_pending = 0;
        uint64_t pend = 0;  // held-back stages: (g << 4 | slot) in 16 bits each
        static_assert(kStages / kProducers <= 4 && kStages <= 16, "held-back stages in 64 bits");
        // MXFP4 routed weights: the stage's prepacked per-row scale image
        // (512 bytes) comes with the stage, under the same barrier
        const uint4* img_src =
            !fp4 ? nullptr
                 : (k.phase ? p.img2 + ((static_cast<size_t>(a.x) * p.t2 + k.t) * p.g2 + k.g0) * 32
                            : p.img13 + ((static_cast<size_t>(a.x) * p.t13 + k.t) * p.g13 + k.g0) * 32);
        const int claim_g = G > kClaimLead ? G - kClaimLead : 0;
        bool claimed = q != 0;  // producer 0 lets the scheduler claim the next task
        // the last stage of this producer's issuers in the task
        int g_last = -1;
        for (int g = G - 1; g >= 0 && g_last < 0; --g)
          if ((g % kIssuers) / kPerProducer == q) g_last = g;
        for (int g = 0; g < G; ++g) {
          if (!claimed && g >= claim_g) {
            st_release_cta(&misc->prod_seq, static_cast<int>(j));  // claim the next
            claimed = true;
          }
          if ((g % kIssuers) / kPerProducer != q) continue;
          const int s = walk.slot(g);
          if (!ptx::mbar_wait(ptx::smem_u32(&bars->empty[s]), walk.parity(s) ^ 1u, abort,
                              kWaitLimitNs)) {
            // the held-back activation copies of the stages already expected
            // still go out, so that each of those stages completes before exit
            for (int i = 0; i < n_pending; ++i) {
              const uint32_t e = static_cast<uint32_t>(pend >> (16 * i));
              issue_b(static_cast<int>((e >> 4) & 0xfffu), static_cast<int>(e & 15u));
            }
            ok = false;
            break;
          }
          walk.advance(g, s);
          const uint32_t full = ptx::smem_u32(&bars->full[s]);
          ptx::mbar_arrive_expect_tx(full, bytes);
          const uint32_t sa = ptx::smem_u32(smem + kOffA + s * kABytes);
          const int x = (k.g0 + g) * kStageK;
          if (k.phase == 0) {
            // one box: the 64 gate rows (half 2e) over the matching 64 up rows (half 2e + 1)
            ptx::tma_load_3d(sa, shared_e ? &p.tm_w13_shared : &p.tm_w13, x, 64 * k.t,
                             shared_e ? 0 : 2 * a.x, full, pol_w);
          } else {
            ptx::tma_load_2d(sa, shared_e ? &p.tm_w2_shared : &p.tm_w2, x,
                             (shared_e ? 0 : a.x * p.hidden) + kTileM * k.t, full, pol_w);
          }
          if (fp4)
            ptx::bulk_load(ptx::smem_u32(smem + kOffSfa + s * kImgBytes), img_src + g * 32,
                           kImgBytes, full, pol_w);
          if (b_ok) {
            issue_b(g, s);
          } else {
            if (n_pending == 0) pend = 0;
            pend |= static_cast<uint64_t>((static_cast<uint32_t>(g) << 4) | static_cast<uint32_t>(s))
                    << (16 * n_pending++);
            bool go = k.phase == 1 && ld_acquire_cta(&misc->ready_seq) >= static_cast<int>(j);
            if (!go && (n_pending == kStages / kProducers || g == g_last)) {
              // on a timeout the held-back loads still go out (their data is
              // not used), so that every issued stage completes before exit
              if (k.phase == 1 && !wait_seq(&misc->ready_seq, static_cast<int>(j), abort)) ok = false;
              go = true;
            }
            if (go) {
              if (k.phase == 1) asm volatile("fence.proxy.async.global;" ::: "memory");
              b_ok = true;
              for (int i = 0; i < n_pending; ++i) {
                const uint32_t e = static_cast<uint32_t>(pend >> (16 * i));
                issue_b(static_cast<int>((e >> 4) & 0xfffu), static_cast<int>(e & 15u));
              }
              n_pending = 0;
              if (!ok) break;
            }
          }
        }
        if (!claimed) st_release_cta(&misc->prod_seq, static_cast<int>(j));
      }
      // wait for every copy still in flight before the CTA may exit
      for (int s = 0; s < kStages; ++s)
        if ((walk.touched >> s) & 1u) drain_wait(ptx::smem_u32(&bars->full[s]), walk.last_parity(s));
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2 || warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // issuer h takes the stages g with g % kIssuers == h of every task; its
    // n-th stage overall sits in its ring slot h + kIssuers (n % 2)
    const int h = warp >= 9 ? warp - 7 : warp - 1;
    if (lane == 0) {
      uint32_t n_own = 0;
      int lt = 0;
      bool ok = true;
      for (uint32_t j = 0; ok; ++j) {
        int4 a;
        Task k;
        const int task = take_task(bars, misc, j, abort, &a, &k);
        if (task < 0) break;
        const int nt = (a.z + 15) & ~15;
        const uint32_t a_fmt = (kFp4 && a.x != p.E) ? ptx::kFmtE2M1 : ptx::kFmtE4M3;
        const int G = k.gn;  // >= 2; an issuer with no stage leaves its accumulator unused
        const int acc = lt & 1;
        const uint32_t use = static_cast<uint32_t>(lt) >> 1;
        ++lt;
        if (!ptx::mbar_wait(ptx::smem_u32(&bars->tempty[acc]), (use & 1) ^ 1, abort, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tbase + (kIssuers * acc + h) * kAccCols;
        for (int g = h; g < G; g += kIssuers, ++n_own) {
          const int s = h + kIssuers * static_cast<int>(n_own & 1u);
          const uint32_t parity = (n_own >> 1) & 1u;  // the slot's earlier uses, mod 2
          if (!ptx::mbar_wait(ptx::smem_u32(&bars->full[s]), parity, abort, kWaitLimitNs) ||
              !ptx::mbar_wait(ptx::smem_u32(&bars->sfa_rdy[s]), parity, abort, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sf_a = tbase + s * kAccCols + kSfColOff;
          const uint32_t sf_b = sf_a + 4;
          const uint32_t sa = ptx::smem_u32(smem + kOffA + s * kABytes);
          const uint32_t sp = ptx::smem_u32(smem + kOffB + s * kBBytes);  // scale image, then rows
          const uint32_t sb = sp + kPanelRows;
          ptx::tc_cp_32x128b_x4(sf_a, ptx::sdesc_rows16(ptx::smem_u32(smem + kOffSfa + s * kImgBytes)));
          ptx::tc_cp_32x128b_x4(sf_b, ptx::sdesc_rows16(sp));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            ptx::tc_mma_mxf8(d_tmem, ptx::sdesc_k128_sw128(sa + 32 * kk),
                             ptx::sdesc_k128_sw128(sb + 32 * kk), ptx::idesc_mxf8(nt, kk, a_fmt), sf_a,
                             sf_b, (g >= kIssuers) || kk != 0);
          }
          ptx::tc_commit(ptx::smem_u32(&bars->empty[s]));
        }
        if (!ok) break;
        ptx::tc_commit(ptx::smem_u32(&bars->tfull[acc]));
      }
      // every MMA / copy this thread issued has completed once drain fires
      ptx::tc_commit(ptx::smem_u32(&bars->drain));
      drain_wait(ptx::smem_u32(&bars->drain), 0);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ weight-scale images
    // Runs ahead of the MMA issuers: as soon as a ring slot is free it writes
    // the slot's 32 x 16-byte image (the stage's 16-byte entry in every row);
    // for MXFP4 routed weights the producer copies the stage's prepacked
    // per-row image with the weights and this warp only marks the slot ready.
    SlotWalk walk;
    bool ok = true;
    for (uint32_t j = 0; ok; ++j) {
      int4 a = make_int4(0, 0, 0, 0);
      Task k0 = {0, 0, 0, 0, 0, 0};
      int task = lane == 0 ? take_task(bars, misc, j, abort, &a, &k0) : 0;
      task = __shfl_sync(0xffffffffu, task, 0);
      if (task < 0) break;
      const int ex = __shfl_sync(0xffffffffu, a.x, 0);  // the unit's expert id
      Task k;
      k.phase = __shfl_sync(0xffffffffu, k0.phase, 0);
      k.u = __shfl_sync(0xffffffffu, k0.u, 0);
      k.t = __shfl_sync(0xffffffffu, k0.t, 0);
      k.g0 = __shfl_sync(0xffffffffu, k0.g0, 0);
      k.gn = __shfl_sync(0xffffffffu, k0.gn, 0);
      k.half = __shfl_sync(0xffffffffu, k0.half, 0);
      const int G = k.gn;
      // MXFP4 routed weights: the producer copies the stage's image itself
      const bool copied = kFp4 && ex != p.E;
      const uint4* sfa = (k.phase ? p.sfa2 + (static_cast<size_t>(ex) * p.t2 + k.t) * p.g2
                                  : p.sfa13 + (static_cast<size_t>(ex) * p.t13 + k.t) * p.g13) +
                         k.g0;
      const uint4 zero = make_uint4(0, 0, 0, 0);
      const uint4 e0 = !copied && lane < G ? __ldg(sfa + lane) : zero;  // stages lane, lane + 32
      const uint4 e1 = !copied && lane + 32 < G ? __ldg(sfa + lane + 32) : zero;
      for (int g = 0; g < G; ++g) {
        const int s = walk.slot(g);
        if (!warp_wait(ptx::smem_u32(&bars->empty[s]), walk.parity(s) ^ 1u, abort)) {
          ok = false;
          break;
        }
        walk.advance(g, s);
        if (copied) {
          if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->sfa_rdy[s]));
          continue;
        }
        const uint4 src = g < 32 ? e0 : e1;
        uint4 v;
        v.x = __shfl_sync(0xffffffffu, src.x, g & 31);
        v.y = __shfl_sync(0xffffffffu, src.y, g & 31);
        v.z = __shfl_sync(0xffffffffu, src.z, g & 31);
        v.w = __shfl_sync(0xffffffffu, src.w, g & 31);
        *reinterpret_cast<uint4*>(smem + kOffSfa + s * kImgBytes + lane * 16) = v;
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->sfa_rdy[s]));
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp - 4;  // TMEM lane quarter
    if (p.picks_early && lane == 0) prefetch_picks(p, q);
    __syncwarp();
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);  // [gate | up][n][64]
    int lt = 0;
    for (uint32_t j = 0;; ++j) {
      if (threadIdx.x == 128) {
        int4 ta;
        Task tk;
        misc->epi_task = take_task(bars, misc, j, abort, &ta, &tk);
        misc->epi_act = ta;
        misc->epi_k = pack_task(tk);
      }
      epi_bar();
      const int task = *reinterpret_cast<volatile int*>(&misc->epi_task);
      if (task < 0) break;
      const Task k = unpack_task(misc->epi_k);
      const int4 a = misc->epi_act;
      const int rows = a.z;
      const int nt = (rows + 15) & ~15;
      const int acc = lt & 1;
      const uint32_t use = static_cast<uint32_t>(lt) >> 1;
      ++lt;
      const uint32_t tfull = ptx::smem_u32(&bars->tfull[acc]);
      if (threadIdx.x == 128) misc->epi_ok = ptx::mbar_wait(tfull, use & 1, abort, kWaitLimitNs);
      epi_bar();
      if (!*reinterpret_cast<volatile int*>(&misc->epi_ok)) break;
      ptx::mbar_wait(tfull, use & 1, abort, kWaitLimitNs);  // completed: returns at once
      ptx::tc_fence_after();
      float v[kMaxTokens];
      // issuer 0's sums, then each later issuer's added in issuer order, 16
      // columns at a time (one 16-register buffer); an issuer that had no
      // stage in this task (fewer stages than issuers) is skipped
      const uint32_t taddr =
          tbase + (static_cast<uint32_t>(32 * q) << 16) + kIssuers * acc * kAccCols;
      ptx::tmem_ld_32x32b_x16(taddr, v);
      if (nt > 16) ptx::tmem_ld_32x32b_x16(taddr + 16, v + 16);
      if (nt > 32) ptx::tmem_ld_32x32b_x16(taddr + 32, v + 32);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int h = 1; h < kIssuers; ++h) {
        if (h >= k.gn) break;
#pragma unroll
        for (int c = 0; c < kMaxTokens / 16; ++c) {
          if (16 * c < nt) {
            float w[16];
            ptx::tmem_ld_32x32b_x16(taddr + h * kAccCols + 16 * c, w);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < 16; ++n) v[16 * c + n] += w[n];
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->tempty[acc]));

      if (k.phase == 1) {
        float* dst = p.part + static_cast<size_t>(a.y) * p.hidden + kTileM * k.t + 32 * q + lane;
        if (k.half) {
          // the two halves' reductions onto zero give the same sum in either
          // order (halves only in steps of at most kW2SplitMaxM tokens)
#pragma unroll
          for (int n = 0; n < kW2SplitMaxM; ++n)
            if (n < rows) atomicAdd(dst + static_cast<size_t>(n) * p.hidden, v[n]);
        } else {
#pragma unroll
          for (int n = 0; n < kMaxTokens; ++n)
            if (n < rows) dst[static_cast<size_t>(n) * p.hidden] = v[n];
        }
        epi_bar();
      } else {
        // gate (warps 4-5) and up (warps 6-7) values to shared memory, then
        // warp q makes h for the 32 columns 32 (q & 1) .. of rows q >> 1,
        // (q >> 1) + 2, ... in a short loop
        const int c = 32 * (q & 1) + lane;  // column within the tile
        float* gu = xchg + (q >= 2 ? kMaxTokens * 64 : 0);
#pragma unroll
        for (int n = 0; n < kMaxTokens; ++n)
          if (n < rows) gu[n * 64 + c] = v[n];
        epi_bar();
        const int i = 64 * k.t + c;  // intermediate column
        const int kb = i >> 5;       // its 32-column block
        uint8_t* panel = p.hpan + (static_cast<size_t>(k.u) * p.g2 + (i >> 7)) * kPanelPitch;
        uint8_t* img = panel + (kb & 3);
#pragma unroll 1
        for (int n = q >> 1; n < rows; n += 2) {
          const float gv = xchg[n * 64 + c];
          const float uv = xchg[(kMaxTokens + n) * 64 + c];
          const float h = (gv / (1.0f + expf(-gv))) * uv;
          float amax = fabsf(h);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
          const int code = mx_code(amax);
          panel[panel_byte(n, i & 127)] = e4m3(clamp_e4m3(h * mx_mul(code)));
          if (lane == 0) img[panel_code_byte(n)] = static_cast<uint8_t>(code);
        }
        // publish the tile's h8 columns and codes to the w2 tasks' bulk
        // copies: each writer's proxy fence, the barrier, then one release
        // count (a device-scope release orders the writes the barrier made
        // visible to the releasing thread; every device-scope fence here
        // waits for the SM's copies in flight, so there is just one)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        epi_bar();
        if (threadIdx.x == 128 && k.u != p.withhold_unit)
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.ready + k.u) : "memory");
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ scheduler
    // Every task comes from the step's counter, the first one included, so a
    // CTA that starts late (fewer SMs free than the grid has CTAs) never holds
    // back a task that a resident CTA waits for: w13 tasks precede every w2
    // task in the claim order, and a CTA only claims its next task while the
    // current one runs. The router zeroed the counter two kernels back
    // (complete once this grid runs: the top-k kernel lets it launch only
    // after its own wait), so the first claim can go out before this grid's
    // own dependency wait. The shared expert is unit 0 in every step, with the
    // fixed entry (E, first row M K, M rows), and its x panels come from the
    // seam, also two kernels back: a first claim below t13 is one of its w13
    // tiles, which needs no routing and is posted at once, so it streams while
    // the top-k kernel finishes.
    int first_task = 0;
    if (lane == 0) first_task = atomicAdd(p.task_ctr, 1);
    first_task = __shfl_sync(0xffffffffu, first_task, 0);
    const bool pre = first_task < p.t13;
    bool pre_ok = true;
    if (pre && lane == 0) {
      const Task k0 = {0, 0, first_task, 0, p.g13, 0};
      pre_ok = post_task(bars, misc, 0, first_task, make_int4(p.E, p.M * p.K, p.M, 0),
                         pack_task(k0), abort);
      if (pre_ok) st_release_cta(&misc->ready_seq, 0);
    }
    // The routing (row counts) and the routed experts' x panels come from the
    // top-k kernel: this warp alone waits for it (in the table's second pass
    // below); the other roles wait on the task queue. The next kernel may
    // start launching then: it waits for this grid before it reads anything
    // this grid writes, and may read the top-k kernel's tables at once (that
    // grid is complete).

    // ---- the step's units (pack_unit) from the per-expert row counts: lane l
    // owns the run of experts l R .. l R + R - 1 (R = ceil(E / 32)); one warp
    // exclusive scan of (rows << 16 | active experts) over the runs gives
    // each active expert its unit index (after the shared expert's 0) and
    // first row. Two passes over the same code: the first, before the grid
    // dependency wait, on counts of zero (no loads, no global writes: its
    // table is overwritten) so that the instructions are fetched while this
    // warp would only wait; the second on the top-k kernel's counts.
    int units = 0;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const bool real = pass != 0;
      if (real) {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
      }
      const int R = (p.E + 31) >> 5;
      const int e0 = lane * R;
      int n[kMaxExperts / 32];
      uint32_t mine = 0;
      bool bad = false;
#pragma unroll
      for (int r = 0; r < kMaxExperts / 32; ++r) {
        n[r] = real && r < R && e0 + r < p.E ? __ldcg(p.cnt + e0 + r) : 0;
        if (n[r] < 0 || n[r] > kMaxTokens) {
          bad = true;
          n[r] = 0;
        }
        mine += (static_cast<uint32_t>(n[r]) << 16) | (n[r] > 0 ? 1u : 0u);
      }
      uint32_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      const int routed = static_cast<int>(total & 0xffffu);
      units = routed + 1;
      if (__any_sync(0xffffffffu, bad) || units > p.units_max ||
          static_cast<int>(total >> 16) > p.M * p.K) {
        if (real && lane == 0) atomicOr(p.err, kErrBounds);
        units = 0;
      } else {
        const uint32_t excl = incl - mine;
        int u = 1 + static_cast<int>(excl & 0xffffu), first = static_cast<int>(excl >> 16);
#pragma unroll
        for (int r = 0; r < kMaxExperts / 32; ++r) {
          if (n[r] > 0) {
            unit_s[u++] = pack_unit(e0 + r, n[r], first);
            first += n[r];
          }
        }
        if (lane == 0) unit_s[0] = pack_unit(p.E, p.M, p.M * p.K);
      }
      __syncwarp();
      if (real && blockIdx.x == 0) {  // the table for diagnostics: routed units, then the shared one
        for (int i = lane; i < units; i += 32) {
          const uint32_t v = unit_s[i];
          p.act[i > 0 ? i - 1 : units - 1] =
              ActiveExpert{static_cast<int>(v & 1023u), static_cast<int>(v >> 16),
                           static_cast<int>((v >> 10) & 63u), 0};
        }
        if (lane == 0) {
          p.counters[kCtrUnits] = units;
          p.counters[kCtrRouted] = units > 0 ? units - 1 : 0;
        }
      }
    }
    const int n13 = units * p.t13;
    const int n2 = units * p.t2;
    const int w2full = n2 > p.split_tiles ? n2 - p.split_tiles : 0;  // the rest go in halves
    const int ntasks = n13 + w2full + 2 * (n2 - w2full);

    // Claims the CTA's tasks, one ahead of the producer: each after the first
    // once the producer has taken the previous one. It posts each with its
    // unit's entry, then -- for a w2 task -- waits (device scope) until the
    // unit's w13 tiles are all done and publishes that for the producer, so
    // the check runs while the producer still streams the previous task.
    if (lane == 0 && pre_ok) {
      int task = first_task;
      uint32_t j = 0;
      bool ok = true;
      if (pre) {  // the first task is posted: claim the next once the producer has taken it
        j = 1;
        ok = wait_seq(&misc->prod_seq, 0, abort);
        task = atomicAdd(p.task_ctr, 1);
      }
      for (; ok; ++j) {
        Task k = {0, 0, 0, 0, 0, 0};
        int4 a = make_int4(0, 0, 0, 0);
        for (; task < ntasks; task = atomicAdd(p.task_ctr, 1)) {  // only valid tasks are posted
          k = decode_task(task, n13, w2full, p);
          const uint32_t v = unit_s[k.u];  // (expert id, first row, rows)
          a = make_int4(static_cast<int>(v & 1023u), static_cast<int>(v >> 16),
                        static_cast<int>((v >> 10) & 63u), 0);
          if (task_valid(a, p)) break;
        }
        const bool last = task >= ntasks;
        if (!post_task(bars, misc, j, last ? -1 : task, a, pack_task(k), abort) || last) break;
        if (k.phase == 1 && !wait_ready(p.ready + k.u, p.t13, abort)) break;
        st_release_cta(&misc->ready_seq, static_cast<int>(j));
        if (!wait_seq(&misc->prod_seq, static_cast<int>(j), abort)) break;
        task = atomicAdd(p.task_ctr, 1);
      }
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, kTmemCols);
  }
  if (threadIdx.x == 0 && misc->abort) atomicOr(p.err, kErrTimeout);
}

}  // namespace

size_t expert_smem_bytes(int) { return kSmemBytes; }

cudaError_t expert_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(expert_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expert_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
  return e;
}

cudaError_t expert_occupancy(int fp4, int* per_sm) {
  cudaError_t e = expert_kernel_setup();
  if (e != cudaSuccess) return e;
  return fp4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                   per_sm, expert_kernel<true>, Roles<true>::kThreads, kSmemBytes)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                   per_sm, expert_kernel<false>, Roles<false>::kThreads, kSmemBytes);
}

cudaError_t launch_experts(const ExpertParams& p, int grid, cudaStream_t s) {
  return p.fp4 ? launch_pdl(expert_kernel<true>, dim3(grid), dim3(Roles<true>::kThreads),
                            kSmemBytes, s, p)
               : launch_pdl(expert_kernel<false>, dim3(grid), dim3(Roles<false>::kThreads),
                            kSmemBytes, s, p);
}

}  // namespace moe
