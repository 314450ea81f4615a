/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) MXFP8 MoE decode step.
 *
 * One call computes the FFN half of one MoE decode step for M <= max_tokens
 * token rows, on one GPU, unsharded:
 *
 *   normed = bf16(RMSNorm(x) * norm_w)                      (FFN seam)
 *   x8, c  = MXFP8(normed): E4M3 bytes + one E8M0 code / 32  (seam quant)
 *   s      = sigmoid(normed . gate_w^T); ids = top-k(s + bias); w = s[ids]/sum
 *   y_e    = MX-GEMM(requant(silu(g) * u), w2_e),  [g; u] = MX-GEMM(x8, w13_e)
 *   out    = bf16(sum_j w_j * y_{ids_j} + y_shared)
 *
 * Sources (the pages this library restates):
 *  - "vllm.models.deepseek_v41.amd.mono.runner": DSV41MonoLayer.ffn (one launch
 *    from the FFN seam to the MoE output; every argument a device pointer so
 *    the launch can be captured in a graph), DSV41MonoLayer.supports
 *    (1 <= tokens <= MAX_TOKENS = 48), DSV41MonoLayer.scratch (scratch
 *    allocated up front, never inside a capture), MonoLayerWeights and its
 *    check (tensor shapes: gate_w [E, 5120] bf16, bias [E] f32, shared
 *    gate_up [2 inter, 5120] e4m3 with [2 inter/32, 160] E8M0, shared down
 *    [5120, inter] e4m3 with [160, inter/32]), _check_tensors (shape / dtype /
 *    contiguity are validated because the kernels' loads are unbounded).
 *  - "vllm.models.deepseek_v41.amd.mono.layer": run_ffn (stage order: norm ->
 *    bf16 MoE input row -> MoE), store_normed, store_x8 (MXFP8 of 32-groups).
 *  - "vllm.models.deepseek_v41.amd.mono.attention.device": mx_code, ceil_exp,
 *    div_rn, mx_mul, fp8_pack4 (E4M3 RNE), mfma_scaled (block-scaled MMA).
 *
 * Conventions shared by every entry point:
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code; nothing throws.
 *  - Pointers named "device" are CUDA device pointers on the handle's device;
 *    "host" pointers are ordinary process memory.
 *  - Ownership: the caller owns every buffer it passes (weights, inputs,
 *    outputs, debug buffers) and keeps the weights alive and unchanged for the
 *    lifetime of the handle. The library owns its scratch and frees it in
 *    moe_destroy.
 *  - Streams are passed as void* holding a cudaStream_t (NULL = the legacy
 *    default stream).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MOE_OK 0
#define MOE_ERR_ARG (-1)         /* null or inconsistent argument */
#define MOE_ERR_RANGE (-2)       /* M outside [1, max_tokens] */
#define MOE_ERR_ALIGN (-3)       /* a device pointer is not 16-byte aligned */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime / driver call failed */
#define MOE_ERR_CAPTURE (-5)     /* not allowed while the stream is being captured */
#define MOE_ERR_TIMEOUT (-6)     /* a bounded device-side wait expired (moe_status) */
#define MOE_ERR_UNSUPPORTED (-7) /* configuration outside what the kernels implement */
#define MOE_ERR_DEVICE (-8)      /* the device is not a compute capability 10.3 GPU */

/*
 * Layer dimensions.
 *  hidden        H: multiple of 128, 256..8192.
 *  experts       E: routed experts, multiple of 32, 32..512.
 *  topk          k: 1..16 and <= E.
 *  inter         I: routed expert intermediate size, multiple of 128, in [256, 8192].
 *  shared_inter  the shared expert's intermediate size; must equal inter.
 *  max_tokens    largest M a step may use, 1..48 (the pages' MAX_TOKENS).
 *  eps           RMSNorm epsilon (1e-6 for the pages' layer).
 *  routed_format MOE_ROUTED_E4M3 (0): routed experts in E4M3 with one E8M0
 *                code per 32 x 32 block; MOE_ROUTED_E2M1 (1): routed experts
 *                in MXFP4 ("vllm.models.deepseek_v41.amd.mono.runner",
 *                MonoLayerWeights: w13 / w2 float4_e2m1fn_x2 with one E8M0
 *                code per row per 32 columns), read by the tensor cores as
 *                E2M1 against the E4M3 activations. The shared expert is E4M3
 *                with 32 x 32 blocks in both.
 */
#define MOE_ROUTED_E4M3 0
#define MOE_ROUTED_E2M1 1
typedef struct moe_config {
  int hidden;
  int experts;
  int topk;
  int inter;
  int shared_inter;
  int max_tokens;
  float eps;
  int routed_format;
} moe_config;

/*
 * Weights: device pointers, row-major, contiguous, 16-byte aligned, read by
 * every step (the E8M0 weight scales are also packed once by moe_create into
 * the kernels' tile order, so changing them later needs a new handle).
 *  norm_w  bf16 [H]                      RMSNorm weight, used as given
 *  gate_w  bf16 [E, H]                   router gate
 *  bias    f32  [E]                      e_score_correction_bias (selection only)
 *  w13     e4m3 [E, 2I, H]               rows [0, I) gate, rows [I, 2I) up
 *  w13_s   u8   [E, 2I/32, H/32]         E8M0 code of each 32 x 32 block
 *  w2      e4m3 [E, H, I]                down projection
 *  w2_s    u8   [E, H/32, I/32]
 *  sw13, sw13_s, sw2, sw2_s              the shared expert, same layouts
 *                                        without the E axis
 * With routed_format MOE_ROUTED_E2M1 the routed tensors are instead
 *  w13     e2m1x2 [E, 2I, H/2]           two E2M1 codes per byte, column 2j in
 *                                        the low nibble of byte j; 32-byte aligned
 *  w13_s   u8   [E, 2I, H/32]            E8M0 code per row per 32 columns
 *  w2      e2m1x2 [E, H, I/2]            32-byte aligned
 *  w2_s    u8   [E, H, I/32]
 * (the pages store them in AITER's shuffled orders; these are row-major).
 */
typedef struct moe_weights {
  const void* norm_w;
  const void* gate_w;
  const float* bias;
  const uint8_t* w13;
  const uint8_t* w13_s;
  const uint8_t* w2;
  const uint8_t* w2_s;
  const uint8_t* sw13;
  const uint8_t* sw13_s;
  const uint8_t* sw2;
  const uint8_t* sw2_s;
} moe_weights;

/*
 * Optional per-step outputs for checking the intermediate steps (device
 * pointers; any may be NULL; each must hold M rows of the given width):
 *  normed    bf16 [M, H]     the MoE input row (FFN seam output)
 *  x8        u8   [M, H]     its E4M3 bytes
 *  x8_codes  u8   [M, H/32]  its E8M0 codes
 *  topk_ids  i32  [M, k]     chosen experts, decreasing score + bias
 *  topk_w    f32  [M, k]     their normalised weights
 *  logits    f32  [M, E]     router logits
 */
typedef struct moe_debug {
  void* normed;
  uint8_t* x8;
  uint8_t* x8_codes;
  int32_t* topk_ids;
  float* topk_w;
  float* logits;
} moe_debug;

typedef struct moe_handle moe_handle;

/*
 * Validates cfg and the weight pointers, makes `device` current, allocates the
 * step's scratch for cfg->max_tokens rows (all of it, up front), packs the
 * weight scales, encodes the TMA descriptors, and synchronises the device.
 * On success *out holds a new handle. Errors: MOE_ERR_ARG (null / bad dims),
 * MOE_ERR_UNSUPPORTED (dims or routed_format outside the limits above),
 * MOE_ERR_ALIGN (a weight pointer not 16-byte aligned, or with
 * MOE_ROUTED_E2M1 the routed w13 / w2 not 32-byte aligned), MOE_ERR_DEVICE,
 * MOE_ERR_CUDA, MOE_ERR_CAPTURE (the legacy stream of `device` is being
 * captured: creation allocates and synchronises), and MOE_ERR_UNSUPPORTED
 * also when one CTA of the expert kernel (384 threads, 448 with
 * MOE_ROUTED_E2M1; about 216 KB of shared memory) cannot be resident on an SM
 * of this device. With MOE_ROUTED_E2M1 the
 * handle also holds the routed experts' per-row scale codes regrouped for the
 * tensor cores (as many bytes as w13_s and w2_s).
 *
 * The expert kernel launches one CTA per SM of the device and hands its tasks
 * out in order from a counter: its progress does not depend on how many of
 * those CTAs are resident at once, so kernels running beside it, or a context
 * limited to fewer SMs, make a step slower but never stall it.
 */
int moe_create(const moe_config* cfg, const moe_weights* w, int device, moe_handle** out);

/*
 * Enqueues one decode step on `stream` (the handle's device must be current):
 * x bf16 [M, H] device -> out bf16 [M, H] device (the MoE output only; no
 * residual is added). Kernel launches only: no allocation, no host
 * synchronisation, so the call may be captured into a CUDA graph. Steps on
 * one handle share its scratch, so they must not run concurrently (enqueue
 * them on one stream). Errors are checked before anything is enqueued:
 * MOE_ERR_RANGE (M < 1 or M > max_tokens), MOE_ERR_ARG, MOE_ERR_ALIGN,
 * MOE_ERR_CUDA (a launch failed). A device-side failure (a bounded wait that
 * expired) is reported later by moe_status. A row holding NaN or infinite
 * values is routed to k distinct valid experts and raises no error; its own
 * output row is unspecified, every other row is as without it.
 */
int moe_decode_step(moe_handle* h, const void* x, int M, void* out, void* stream,
                    const moe_debug* dbg);

/*
 * Synchronises the handle's device and returns MOE_OK, MOE_ERR_TIMEOUT if a
 * step's kernel gave up a bounded wait since the last moe_clear_status,
 * MOE_ERR_ARG if a kernel found a pick or a per-expert row count out of range
 * (a defensive check: top-k always picks k distinct valid experts, even from
 * non-finite scores, so only corrupted scratch sets it), or MOE_ERR_CUDA if
 * the device reported an error. Not allowed during capture (MOE_ERR_CAPTURE).
 */
int moe_status(moe_handle* h);

/* Resets the device-side error word (synchronous). MOE_ERR_CAPTURE during capture.
 * moe_status, moe_clear_status, moe_last_unique_experts and moe_destroy work on
 * the handle's device and leave the calling thread's current device as it was. */
int moe_clear_status(moe_handle* h);

/*
 * Test hook for the device-side timeout path (off by default; the source
 * pages have no counterpart). While unit >= 0, the steps enqueued on this
 * handle never report the w13 tiles of the expert kernel's unit `unit` as
 * done (unit 0 is the shared expert, present in every step), so each w2 task
 * of that unit waits until its bounded wait (1 s) expires: the CTA records
 * MOE_ERR_TIMEOUT in the error word, lets its copies and MMAs in flight
 * complete, frees its tensor memory and exits, and the step's output is
 * unspecified. No memory fault and no hang: the stream completes. unit = -1
 * turns the hook off. Errors: MOE_ERR_ARG (null handle), MOE_ERR_RANGE (unit
 * < -1 or beyond the handle's unit capacity).
 */
int moe_test_withhold_ready(moe_handle* h, int unit);

/*
 * Number of distinct routed experts the last completed step used (synchronous
 * read of the device routing table into *unique_routed). For byte accounting.
 */
int moe_last_unique_experts(moe_handle* h, int* unique_routed);

/*
 * Timing hooks for profiling: while set, every step records events[i]
 * (cudaEvent_t values, caller-owned) on its stream just before kernel i and
 * events[n_kernels] after the last kernel; n must equal moe_kernel_count()+1.
 * With n = 2, events[0] is recorded just before the step's first kernel and
 * events[1] after its last, and nothing in between (the kernels keep
 * overlapping through programmatic dependent launch).
 * Pass events = NULL, n = 0 to turn it off. Inside a stream capture the
 * records become event-record nodes of the graph: the events must then outlive
 * every graph (and graph exec) captured with them.
 */
int moe_set_timing_events(moe_handle* h, void* const* events, int n);

/* The kernels a step can launch, in order, and the name of kernel i (static
 * string). A step of at most 4 tokens runs the seam inside the router kernel
 * and launches the others only (its seam events are recorded back to back). */
int moe_kernel_count(void);
const char* moe_kernel_name(int i);

/* Number of kernels a step of M tokens launches on this handle (0 if h is
 * null or M is out of range). */
int moe_step_launches(const moe_handle* h, int M);

/*
 * Diagnostics: device address and size of one region of the handle's scratch,
 * valid until moe_destroy; contents are those of the last completed step.
 * Regions (layouts are internal and may change):
 *  MOE_REGION_GATHERED  u8  [E + 1][H / 128][7168] activation panels by
 *      expert id (E = the shared expert): panel (e, g) holds, for K columns
 *      [128 g, 128 g + 128), a 32 x 16-byte scale image at byte 0 (row r,
 *      byte 4 j + b = E8M0 code of K block b of the expert's row 32 j + r),
 *      then from byte 1024 the expert's MXFP8 token rows: row r, column c at
 *      byte 1024 + 128 r + 16 ((c / 16) xor (r % 8)) + c % 16. Row r of a
 *      routed expert is the token that took slot r (any order); rows of the
 *      shared expert are the tokens in order. Rows >= the expert's token
 *      count, and experts no token picked, are unspecified; at M = 1 no
 *      routed panel is written (every unit reads the shared expert's).
 *  MOE_REGION_H8        u8  [units][I / 128][7168] the same layout for the
 *      requantised silu(g) * u rows, by the expert kernel's unit index: the
 *      shared expert first, then the routed experts of MOE_REGION_ACTIVE in
 *      its order
 *  MOE_REGION_PARTIAL   f32 [rows][H]  expert output rows y
 *  MOE_REGION_ACTIVE    i32 [E + 1][4] active experts: expert, first row, rows, 0
 *  MOE_REGION_TOKPOS    i32 [M][k + 1] row of (token, pick); pick k = shared expert
 * rows = M * (k + 1) for the step's M: each active routed expert (increasing
 * id) owns a run of rows, its tokens in slot order, then the shared expert's M
 * rows in token order; units = the active experts, at most
 * min(E, max_tokens * k) + 1.
 */
#define MOE_REGION_GATHERED 0
#define MOE_REGION_H8 1
#define MOE_REGION_PARTIAL 2
#define MOE_REGION_ACTIVE 3
#define MOE_REGION_TOKPOS 4
int moe_scratch_region(const moe_handle* h, int region, void** ptr, size_t* bytes);

/* Bytes of device scratch the handle holds. */
size_t moe_scratch_bytes(const moe_handle* h);

/* Static description of an error code. */
const char* moe_strerror(int code);

/* Frees the handle's scratch and the handle (NULL is allowed). */
void moe_destroy(moe_handle* h);

/*
 * Allocation-free routing. The source pages have no counterpart to this entry
 * point; it is an addition of this library for callers that may not allocate
 * device memory when they route: an engine whose memory is all handed out by
 * its own pool (or planned before it starts) cannot have a library call
 * cudaMalloc behind its back, code running inside a CUDA graph capture cannot
 * call cudaMalloc at all, and a caller that only needs routing decisions for
 * rows it already normalised should not need a moe_create handle (which
 * allocates the whole step's scratch).
 *
 * Computes, for M bf16 rows `normed` [M, hidden] (device), the router of
 * moe_decode_step: logits against gate_w bf16 [experts, hidden] (device),
 * scores sigmoid(logit), the topk experts of score + bias (bias f32
 * [experts], device; ties to the lower index) in decreasing order into
 * topk_ids i32 [M, topk] (device), and their scores over the chosen scores'
 * sum into topk_w f32 [M, topk] (device). The caller owns every buffer;
 * nothing is allocated: the kernel's scratch is one fixed device array of
 * MOE_ROUTE_STATIC_SCRATCH_BYTES inside the library, held by every GPU that
 * loads the library until the process exits.
 *
 * Limits: 1 <= M <= 48; hidden a multiple of 128 in [256, 8192]; experts a
 * multiple of 32 in [32, 512]; 1 <= topk <= 16. A problem whose scratch
 * (partial logits, 4 * KS * experts * M bytes with KS the router's K-split,
 * about 1024 / experts and at least hidden / 1536, plus small routing tables)
 * would not fit the array is refused with MOE_ERR_UNSUPPORTED before anything
 * is enqueued (e.g. experts = 512 with hidden > 3072). Other errors:
 * MOE_ERR_ARG (null pointer), MOE_ERR_ALIGN (normed / gate_w not 16-byte
 * aligned, the others not 4-byte aligned), MOE_ERR_RANGE (M), MOE_ERR_CUDA.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address and sets the kernel's shared-memory limit; make that first
 * call before any stream capture. The address is kept until the process
 * exits: calls after a cudaDeviceReset of that device are not supported. Each
 * call enqueues a memset of the array's counters and two kernels on `stream`
 * (void* holding a cudaStream_t). All calls share the one array, which keeps
 * the last call's contents: calls whose work overlaps on the GPU (different
 * streams, or concurrent host threads without ordering) race on it and must
 * be serialised by the caller.
 *
 * Device-side errors are not returned by the call (it only enqueues): read
 * them with moe_route_static_status. Rows whose scores are not finite (NaN or
 * infinite inputs) give k distinct valid but unspecified ids and NaN weights,
 * and no error.
 */
#define MOE_ROUTE_STATIC_SCRATCH_BYTES (256 * 1024)
int moe_route_static(const void* normed, const void* gate_w, const float* bias, int M,
                     int hidden, int experts, int topk, int32_t* topk_ids, float* topk_w,
                     void* stream);

/*
 * Device-side status of the moe_route_static calls enqueued on the current
 * device (void* stream holding a cudaStream_t): waits for `stream`, then
 * reads the array's error word, which each moe_route_static call clears when
 * it starts. Returns MOE_OK, MOE_ERR_TIMEOUT (a kernel gave up a bounded wait:
 * that call's outputs are unspecified), MOE_ERR_CAPTURE (the stream is being
 * captured: this call synchronises), MOE_ERR_CUDA, or MOE_OK if no call has
 * run on the device yet. Allocates nothing.
 */
int moe_route_static_status(void* stream);

/*
 * Attention-seam MXFP8 ("vllm.models.deepseek_v41.amd.mono.layer", store_x8:
 * the attention seam's fp32 norm output -> the attention's input quant).
 *
 * For M bf16 rows x [M, hidden] (device) and the attention norm weight
 * norm_w bf16 [hidden] (device): ys = x * (mean(x^2) + eps)^(-1/2) * norm_w
 * computed in fp32 (the sum of squares in the FFN seam's fixed order), then
 * per 32 columns the E8M0 code of the fp32 values' amax (the same code as the
 * FFN seam: clamp(ceil(log2(fp32(amax / 448))) + 127, 0, 254), amax floored
 * at FLT_MIN) into x8_codes u8 [M, hidden/32], and the E4M3 bytes (round to
 * nearest even) of clamp(ys * 2^(127 - code), -448, 448) into x8 u8
 * [M, hidden]. Unlike moe_decode_step's seam, the quant reads the fp32 norm
 * outputs, not their bf16 rounding. If ys is not null the fp32 norm outputs
 * also go to ys f32 [M, hidden] (device).
 *
 * The caller owns every buffer; nothing is allocated and nothing synchronises:
 * one kernel is enqueued on `stream` (void* holding a cudaStream_t; capture
 * safe). Limits: 1 <= M <= 48; hidden a multiple of 32 in [32, 8192].
 * Errors: MOE_ERR_ARG (a null required pointer, eps < 0 or NaN), MOE_ERR_ALIGN
 * (x, norm_w, x8 or ys not 16-byte aligned), MOE_ERR_RANGE (M),
 * MOE_ERR_UNSUPPORTED (hidden), MOE_ERR_CUDA (the launch failed).
 */
int moe_attn_seam_x8(const void* x, const void* norm_w, int M, int hidden, float eps,
                     uint8_t* x8, uint8_t* x8_codes, float* ys, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
