/*
 * moe.h -- C ABI of one routed mixture-of-experts layer forward pass on a
 * single NVIDIA GB300 GPU (sm_103a).
 *
 * What the layer is.  FreeToken ("FreeToken：把 284B MoE 塞进游戏 PC",
 * zhichai.net, §二 "Decode: q⋆ = m·B_P/B_H" and "LRU 为什么赢" paragraphs)
 * serves MoE models whose routed experts live in a GPU-resident LRU expert
 * cache; experts that miss are loaded into it from host memory.  Its formats
 * are MXFP4 and NVFP4 (same page §五; juejin.cn overview §五).  The pages give
 * no formula for the layer; this library computes the standard one:
 *
 *   logits = x W_r^T (+ b);  top-k per token (ties -> lower expert id);
 *   gates  = softmax over the k selected logits (or full-softmax probs);
 *   y[t]   = sum_j gate[t,j] * FFN_{e_j}(x[t]) (+ FFN_shared(x[t]));
 *   FFN(x) = W_d (SiLU(W_g x) * (W_u x)),  weights block-scaled FP4.
 *
 * Every call returns an int status: MOE_OK (0) or a negative MOE_ERR_*.
 * Nothing throws across this boundary.  moe_last_error(layer) gives the text
 * of the last failure on that layer, moe_status_string(code) a fixed text.
 *
 * Memory.  The library owns, and allocates with cudaMalloc at create time,
 * the slot pool (n_slots experts), the shared-expert copy, the router weights,
 * the slot table and all per-step workspaces.  The caller owns x, y, the
 * host expert pool and the streams it passes.  Device pointers are CUDA
 * device addresses on the layer's device (the device current at create).
 * A layer is not thread-safe; calls on one layer must not overlap.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK                 0
#define MOE_ERR_ARG           -1  /* bad shape, index or pointer            */
#define MOE_ERR_NOT_INSTALLED -2  /* a miss has no registered host source   */
#define MOE_ERR_OOM           -3  /* cudaMalloc / pinned allocation failed  */
#define MOE_ERR_FILL          -4  /* a host->slot copy could not be issued  */
#define MOE_ERR_TIMEOUT       -5  /* a bounded device wait gave up          */
#define MOE_ERR_CUDA          -6  /* a CUDA runtime call failed             */
#define MOE_ERR_STATE         -7  /* call made in the wrong state           */
#define MOE_ERR_UNSUPPORTED   -8  /* valid request this build cannot serve  */

/* ---- weight formats ----------------------------------------------------
 * The engine runs MXFP4, NVFP4, FP8 and BF16 checkpoints (juejin.cn overview,
 * §五 模型生态与硬件支持; zhichai.net §五 for the FP4 ones). */
#define MOE_MXFP4 0  /* E2M1 codes, one E8M0 scale per 32 along K            */
#define MOE_NVFP4 1  /* E2M1 codes, one E4M3 scale per 16 along K, fp32/tensor */
#define MOE_MXFP8 2  /* E4M3 codes (one byte each), one E8M0 scale per 32    */
#define MOE_BF16  3  /* bf16 elements, no scales                             */

/* ---- regimes -----------------------------------------------------------
 * Decode: the weights x bf16-class activations (A16), a GEMV.  Prefill: a
 * tensor-core grouped GEMM whose activations take the weight's element type:
 * FP4 x FP4 (MXFP4 / NVFP4), MXFP8 x MXFP8 (W8A8), bf16 x bf16 (W16A16). */
#define MOE_REGIME_AUTO    0  /* decode for N <= 64, prefill otherwise       */
#define MOE_REGIME_DECODE  1  /* weights x bf16 activations, GEMV            */
#define MOE_REGIME_PREFILL 2  /* weights x activations of their type, GEMM   */

typedef struct moe_layer* moe_layer_t;
typedef struct moe_stack* moe_stack_t;

/* Layer descriptor.  E experts, top-k, d_model, d_ff, n_slots cache slots. */
typedef struct {
    int E;            /* routed experts, 1..1024                              */
    int k;            /* experts per token, 1..min(E, 32)                     */
    int d_model;      /* multiple of 128 (of 256 for the prefill regime)      */
    int d_ff;         /* multiple of 128 (of 256 for the prefill regime)      */
    int n_slots;      /* GPU expert-cache slots, 1..E (a stack: 1..min(L E, 1024)) */
    int fmt;          /* MOE_MXFP4, MOE_NVFP4, MOE_MXFP8 or MOE_BF16          */
    int has_shared;   /* 1: one always-on shared expert, weight 1, resident   */
    int norm_topk;    /* 1: gates renormalised over the k selected            */
    int has_bias;     /* 1: per-expert router bias added to the logits        */
    int max_tokens;   /* largest N of one moe_forward (sizes the workspaces)  */
    float act_scale_x;/* NVFP4 prefill: static fp32 scale of x (power of 2)   */
    float act_scale_h;/* NVFP4 prefill: static fp32 scale of h (power of 2)   */
    int prefill_act_bits; /* activations of the prefill regime: 0 (or the
                       * weights' own code bits: 4, 8, 16) = the weights' own
                       * format; 8 on MOE_MXFP4 weights = MXFP8 activations,
                       * W4A8 (x and h quantised to MXFP8; tcgen05
                       * kind::mxf8f6f4 with E4M3 x E2M1 operands).  The
                       * FreeToken engine serves MXFP4, NVFP4, FP8 and BF16
                       * precisions (juejin.cn overview, §五 "模型生态与硬件支持");
                       * FP4 weights under FP8 activations pair two of them.
                       * Other values: MOE_ERR_ARG.                          */
} moe_layer_desc;

/* Byte layout of one expert (identical in the host pool and in a slot).
 * Matrices are K-contiguous: gate [d_ff, d_model], up [d_ff, d_model],
 * down [d_model, d_ff].  Codes: two E2M1 per byte, low nibble = even K
 * (MXFP4, NVFP4); one E4M3 byte per element (MXFP8); bf16 elements as
 * little-endian byte pairs (BF16).  Scales: row-major [rows, K/32] E8M0 (MXFP4,
 * MXFP8) or [rows, K/16] E4M3 (NVFP4); none for BF16 (the scale offsets then
 * coincide).  tensor_scales: three fp32 (gate, up, down; 1.0 except NVFP4).  All offsets
 * are multiples of 256 bytes; `bytes` is the padded size of one expert. */
typedef struct {
    size_t bytes;
    size_t gate_codes, up_codes, down_codes;
    size_t gate_scales, up_scales, down_scales;
    size_t tensor_scales;
} moe_expert_layout;

/* Filled by moe_forward when `info` is not NULL. */
typedef struct {
    int regime;        /* regime actually run                                 */
    int n_tokens;
    int n_distinct;    /* |U|: distinct routed experts this step              */
    int n_hits;
    int n_misses;
    int n_waves;       /* ceil(|U| / n_slots)                                 */
    size_t fill_bytes; /* bytes copied host -> slots this step                */
    int host_synced;   /* 1 if the call waited for the routing on the host    */
    int n_launches;    /* kernels this call launched                          */
    int fused_step;    /* 1 if the step ran as one fused launch               */
} moe_forward_info;

/* Kernel classes of moe_profile_read. */
#define MOE_PROF_ROUTER      0
#define MOE_PROF_PERMUTE     1  /* permutation (and the LRU step, fused, N<=128) */
#define MOE_PROF_LRU         2
#define MOE_PROF_GATEUP      3  /* expert FFN phase 1: W_g, W_u, SiLU * mul
                                   (decode GEMV or prefill grouped GEMM)       */
#define MOE_PROF_DOWN        4  /* expert FFN phase 2: W_d                      */
#define MOE_PROF_COMBINE     5
#define MOE_PROF_FILL        6  /* host -> slot copies on the fill stream       */
#define MOE_PROF_PREFILL     7  /* prefill: activation gather + FP4 quantiser   */
#define MOE_PROF_COMMIT      8  /* no launches: later-wave misses are remapped,
                                   not copied (kept for the class numbering)   */
#define MOE_PROF_STEP        9  /* the fused decode step (one launch)           */
#define MOE_PROF_KINDS      10

/* Layout of one expert for a descriptor (no GPU work). */
int moe_expert_layout_for(const moe_layer_desc* desc, moe_expert_layout* out);

/* Create a layer on the current device: validates the descriptor, allocates
 * the slot pool, table and workspaces, creates the fill stream.  The cache
 * starts empty (every slot free).  The arguments are the layer's shape (E
 * routed experts, top-k, d_model, d_ff: the MoE layer the FreeToken pages
 * serve, "FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二 "Decode"
 * paragraph: per token only a few of many experts run) and the number of
 * GPU expert-cache slots (the same page's LRU expert cache, §二 "LRU 为什么赢";
 * juejin.cn overview, §二 "全局 LRU 专家缓存"), plus the weight format (MXFP4
 * or NVFP4 checkpoints, zhichai.net §五) and the optional shared expert
 * (ananclaw.com explainer, §核心方法 4, shared experts as an architecture
 * axis).  MOE_ERR_ARG on an invalid descriptor,
 * MOE_ERR_UNSUPPORTED when d_model or d_ff exceeds 8192 (the decode kernels
 * stage one token group's activations in shared memory), MOE_ERR_OOM when
 * device memory runs out (nothing is leaked). */
int moe_layer_create(const moe_layer_desc* desc, moe_layer_t* out);
int moe_layer_destroy(moe_layer_t layer);

/* Router weights W_r fp32 [E, d_model] row-major and, when has_bias, the
 * fp32 bias [E] (NULL otherwise).  Host or device pointers; copied
 * synchronously. */
int moe_set_router(moe_layer_t layer, const float* W_r, const float* bias);

/* Register the caller's host expert pool: E experts back to back, expert e
 * at byte offset e * layout.bytes.  Must be pinned (page-locked) host memory
 * of at least E * layout.bytes bytes; it stays owned by the caller and must
 * outlive the layer's use of it.  It is the source of every cache fill. */
int moe_register_host_experts(moe_layer_t layer, const void* pool, size_t bytes);

/* Copy the shared expert (layout.bytes, same layout; host or device pointer)
 * into its resident buffer.  MOE_ERR_STATE if the layer has no shared one. */
int moe_set_shared_expert(moe_layer_t layer, const void* weights);

/* Install expert `expert` into slot `slot` from the host pool, as most
 * recently used, ordered on `stream` (NULL = legacy default stream).  An
 * expert previously in that slot is evicted; if `expert` was resident in
 * another slot that slot becomes free.  MOE_ERR_NOT_INSTALLED if no host pool
 * is registered.  (The expert cache of the zhichai.net page, §二.) */
int moe_cache_install(moe_layer_t layer, int expert, int slot, void* stream);

/* Apply one step's accesses to the device slot table, as moe_forward does
 * (the per-step update of the LRU expert cache: "FreeToken：把 284B MoE 塞进游戏
 * PC", zhichai.net, §二 "LRU 为什么赢" -- recently routed experts stay on the
 * GPU, misses are loaded from host memory; the per-step access order below is
 * this library's reading, the pages leave it open):
 * the distinct experts of experts[0..n) are accessed hits first (ascending
 * id), then misses (ascending id); a miss takes the lowest free slot, else
 * evicts the least recently used expert.  Misses are filled from the host
 * pool when one is registered.  Outputs (host arrays, any may be NULL):
 * slot_of_out[i] = slot that experts[i] was served from this step;
 * miss_experts_out / miss_slots_out = the misses in access order (capacity
 * n); *n_miss_out = their count.  Synchronous: returns after the table and
 * fills are complete. */
int moe_lru_touch(moe_layer_t layer, const int* experts, int n, int* slot_of_out,
                  int* miss_experts_out, int* miss_slots_out, int* n_miss_out,
                  void* stream);

/* Change the number of GPU expert-cache slots between steps, without
 * reloading any expert from host memory (the pages' elastic expert cache:
 * "FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二 "弹性显存" -- the cache
 * is a runtime variable, rebuilt at scheduler safe points).  The
 * min(n_slots, resident) most recently used experts stay, with their recency
 * stamps, in slots 0, 1, ... in the order of their old slots; the other
 * slots are free; the clock is unchanged.  The slot pool is reallocated to
 * the new size (n_slots + 1 + spare buffers) and the kept experts and the
 * shared expert are copied into it on the device, so device memory is given
 * back when the cache shrinks.  Synchronizes the device (a step boundary).
 * MOE_ERR_ARG unless 1 <= n_slots <= E; MOE_ERR_OOM (cache unchanged) if the
 * new pool cannot be allocated. */
int moe_cache_resize(moe_layer_t layer, int n_slots, void* stream);

/* Read / replace the slot table (host arrays of n_slots entries; expert -1 =
 * free slot; stamps are recency counters, larger = more recent; *clock is
 * the last stamp issued).  set_state does not move weights: the caller
 * must make each slot's contents match (e.g. with moe_cache_install). */
int moe_lru_get_state(moe_layer_t layer, int* expert_of_slot, uint64_t* stamp,
                      uint64_t* clock);
int moe_lru_set_state(moe_layer_t layer, const int* expert_of_slot,
                      const uint64_t* stamp, uint64_t clock);

/* One forward pass: x bf16 [N, d_model] -> y bf16 [N, d_model], ordered on
 * `stream`.  One step of the pages' MoE layer: route each token to k experts,
 * serve the routed experts from the GPU expert cache (hits) or load them from
 * host memory first (misses), run them and combine ("FreeToken：把 284B MoE
 * 塞进游戏 PC", zhichai.net, §二 "Decode" for a decode step, "Prefill：把计算
 * 藏进传输" for a prefill chunk; the layer formula is the standard one given at
 * the top of this file, since the pages print none).  x and y may be device pointers or host pointers (then staged
 * through the layer's workspace, and the call returns after y is written).
 * N == 0 is a no-op; 0 < N <= max_tokens.  With misses (possible unless
 * every expert is resident) the call waits on the host for the step's routing
 * record, which the LRU kernel writes into mapped pinned memory (polled,
 * bounded: MOE_ERR_STATE if the routing finished and no record arrived,
 * MOE_ERR_TIMEOUT after 30 s), and then issues the slot fills on the layer's
 * fill stream; otherwise it returns without waiting.  Misses beyond
 * the first n_slots accesses of a step are filled into spare buffers at once,
 * and a spare whose expert keeps its LRU slot becomes that slot's buffer (no
 * copy), so the cache state after the call is the LRU's either way.  regime:
 * MOE_REGIME_*.  MOE_ERR_NOT_INSTALLED if a miss has no host source. */
int moe_forward(moe_layer_t layer, const void* x, int N, void* y, void* stream,
                int regime, moe_forward_info* info);

/* How misses reach their slots.  Registering the host pool selects
 * MOE_FILL_AUTO when the device can address the pool (pinned memory under
 * unified addressing) and MOE_FILL_MEMCPY otherwise, unless a mode was set
 * here before; a pool the device cannot address always turns the mode to
 * MOE_FILL_MEMCPY.  MOE_FILL_MEMCPY: the host reads
 * the step's routing record and issues cudaMemcpyAsync from the pinned pool on
 * the layer's fill stream (a run of consecutive experts bound for consecutive
 * slots is one copy) while the hits compute; a long miss list runs its expert
 * FFN in chunks, each after its own copies.
 * MOE_FILL_DEVICE: a copy kernel on a side stream reads the record on the GPU
 * and pulls the missed experts from the pinned pool itself (unified
 * addressing over the host link), so moe_forward never waits on the host;
 * moe_forward_info then reports n_distinct / n_hits = -1 (see moe_stats).
 * MOE_FILL_KERNEL: the copies are made by a copy kernel on 12 SMs that the
 * decode expert GEMV leaves free, queued on the fill stream (created with the
 * highest stream priority) behind the routing, one launch per chunk of the
 * miss list, each reading its part of the list from the record on the device;
 * the host still reads the record to launch the misses' expert FFN, so the
 * copies start as soon as the routing ends and pay no per-copy cost of the
 * copy engine.  The prefill regime fills with cudaMemcpyAsync in this mode,
 * since its GEMM takes every SM, and so does a GPU of at most 24 SMs.
 * MOE_FILL_FUSED: no separate copy: one decode expert-FFN launch covers the
 * step's hits and misses, reading each miss's weights from the pinned pool
 * over the host link (the pool must be device-addressable) and writing them
 * on to the miss's slot as it computes; the host never waits (as with
 * MOE_FILL_DEVICE, moe_forward_info reports -1 counts).  The prefill regime
 * fills with cudaMemcpyAsync in this mode.
 * MOE_FILL_AUTO: per decode call, MOE_FILL_FUSED while min(E, N k) <= n_slots
 * (no access can need a spare buffer), else MOE_FILL_KERNEL.
 * MOE_ERR_STATE if the registered pool is not device-addressable (every mode
 * but MOE_FILL_MEMCPY). */
#define MOE_FILL_MEMCPY 0
#define MOE_FILL_DEVICE 1
#define MOE_FILL_KERNEL 2
#define MOE_FILL_FUSED 3
#define MOE_FILL_AUTO 4
int moe_set_fill_mode(moe_layer_t layer, int mode);

/* How a decode step runs.  MOE_DECODE_AUTO (default): as one fused,
 * cooperative launch -- routing, LRU step, expert FFN over hits and misses,
 * shared expert and combine, one CTA per SM meeting at grid barriers --
 * for small steps (N * k <= 32) of a layer that holds every expert or of a
 * stack's layer, else as the chain of launches.  The fused launch takes steps of at most 16 tokens with
 * N * k <= 256, E <= 640,
 * d_model a multiple of 128, whose misses (if any) are filled by the expert
 * FFN itself (every expert resident, or MOE_FILL_FUSED, or MOE_FILL_AUTO
 * choosing it).  Both paths compute the same values bit for bit.
 * MOE_DECODE_CHAIN: always the chain.  MOE_DECODE_STEP: always fused;
 * moe_forward returns MOE_ERR_UNSUPPORTED for a step that cannot be. */
#define MOE_DECODE_AUTO  0
#define MOE_DECODE_CHAIN 1
#define MOE_DECODE_STEP  2
int moe_set_decode_path(moe_layer_t layer, int path);

/* Totals since create, accumulated on the device by the LRU step of every
 * moe_forward: out4 = {steps, distinct experts, hits, misses}.  Synchronizes
 * the device. */
int moe_stats(moe_layer_t layer, uint64_t* out4);

/* Kernel timing.  moe_profile(layer, 1) resets the counters and from then
 * on brackets every launch of the layer with CUDA events on the stream it runs
 * on (at most 32768 launches are timed); moe_profile(layer, 0) stops.
 * moe_profile_read synchronizes the device and returns, per MOE_PROF_* class,
 * the summed device milliseconds and the launch count (arrays of
 * MOE_PROF_KINDS entries, either may be NULL).  Timing adds one event record
 * per launch edge and nothing else. */
int moe_profile(moe_layer_t layer, int enable);
int moe_profile_read(moe_layer_t layer, double* ms, int* launches);

const char* moe_last_error(moe_layer_t layer);
const char* moe_status_string(int status);

/* ---- test hooks: each runs one step of moe_forward's path in isolation.
 * All pointers are device pointers; work is ordered on `stream`. ---------- */

/* Router: idx int32 [N, k] ascending expert id, gates fp32 [N, k], logits fp32
 * [N, E] (may be NULL). */
int moe_debug_router(moe_layer_t layer, const void* x, int N, int* idx,
                     float* gates, float* logits, void* stream);

/* Permutation of idx int32 [N, k]: counts [E], offsets [E+1], row_of [N*k]
 * (row of (t, j) at t*k + j), tok_of [N*k]. */
int moe_debug_permute(moe_layer_t layer, const int* idx, int N, int* counts,
                      int* offsets, int* row_of, int* tok_of, void* stream);

/* What the last moe_forward on this layer decided, copied from the layer's
 * workspaces into caller device arrays (any may be NULL), ordered on
 * `stream`: idx int32 [N, k] and gates fp32 [N, k] of its router, counts
 * [E], offsets [E+1], row_of [N*k] and tok_of [N*k] of its permutation (the
 * arrays the expert FFN and the combine of that call used), N = that call's
 * token count (*n_out, may be NULL).  MOE_ERR_STATE before the first
 * moe_forward. */
int moe_debug_last_step(moe_layer_t layer, int* idx, float* gates, int* counts, int* offsets,
                        int* row_of, int* tok_of, int* n_out, void* stream);

/* The expert FFN's intermediate values of the last moe_forward, copied into
 * caller device arrays (any may be NULL), ordered on `stream`; rows =
 * N*k permuted rows (+ N shared-expert rows, token order, when the layer has
 * one).  After a decode call: h fp32 [rows, 2*d_ff] = W_g x | W_u x of each
 * row (block scales and tensor scales applied).  After a prefill call:
 * hq_codes and hq_scales, the codes and block scales of h = SiLU(W_g x) *
 * (W_u x) that the down GEMM consumed, in the prefill activation format:
 * FP4 [rows, d_ff/2] + [rows, d_ff/block]; MXFP8 [rows, d_ff] + [rows,
 * d_ff/32]; bf16 [rows, 2 d_ff] bytes, no scales.
 * MOE_ERR_STATE when the requested arrays were not produced by that call. */
int moe_debug_last_hidden(moe_layer_t layer, float* h, uint8_t* hq_codes, uint8_t* hq_scales,
                          void* stream);

/* Error-path hooks for tests.  They act on the host only: nothing makes the
 * GPU fault, trap or wait without bound.
 * MOE_INJECT_FILL: the next host-issued fill of this layer (moe_forward in
 * MOE_FILL_MEMCPY mode, moe_lru_touch, moe_cache_install) fails before its
 * cudaMemcpyAsync is issued.  The call returns MOE_ERR_FILL; a forward or
 * touch step's misses are then dropped from the cache (their slots become
 * free, so a later step fills them again) and y is not written.
 * MOE_INJECT_WAIT_LIMIT: the bounded device waits of the next moe_forward's
 * decode expert-FFN launches give up after `arg` SM clock cycles (instead of
 * about 2 s); a launch whose wait gives up sets the layer's error word,
 * finishes without further work, and the next moe_forward returns
 * MOE_ERR_TIMEOUT (the slot table, updated before the expert FFN, stays
 * consistent).  MOE_INJECT_NONE clears both. */
#define MOE_INJECT_NONE 0
#define MOE_INJECT_FILL 1
#define MOE_INJECT_WAIT_LIMIT 2
int moe_debug_inject(moe_layer_t layer, int what, long long arg);

/* Process-wide test hook: the nth device or pinned-host allocation the
 * library makes from now on fails without being attempted (1 = the next one,
 * 0 = none), as if the memory had run out.  live_out (2 entries, may be NULL)
 * receives the number of device and pinned-host allocations the library holds
 * at the time of the call, for leak checks. */
int moe_debug_alloc_fault(long long nth, long long* live_out);

/* Timeline of the last fused decode step run while kernel timing
 * (moe_profile) was on: per CTA, 11 global-timer stamps (ns) -- kernel
 * start, logits written, grid barrier 1 passed, top-k done, permutation
 * done, access table built, phase-1 (gate/up) outputs written, barrier 2
 * passed, phase-2 (down) outputs written, barrier 3 passed, combine done
 * (marks a CTA does not reach stay from an earlier step) -- then the SM clock
 * counter at the first and at the last stamp, then the global timer when the
 * CTA's first phase-1 weight stage had landed and when its last one was
 * consumed, the same two for phase 2, and when the CTA's first phase-2
 * activation block was staged (18 entries per CTA).  out: host array of at least
 * n_cta * n_marks entries, CTA-major; *n_cta, *n_marks (may be NULL) get the
 * sizes.  MOE_ERR_STATE if no such step ran. */
int moe_debug_step_trace(moe_layer_t layer, uint64_t* out, int cap, int* n_cta, int* n_marks);

/* Dequantised fp32 weights of matrix m (0 gate, 1 up, 2 down) of the expert
 * in slot `slot` (slot -1: the shared expert), written row-major to out. */
int moe_debug_dequant(moe_layer_t layer, int slot, int m, float* out, void* stream);

/* Activation quantiser of the prefill regime (the layer's prefill activation
 * format) on fp32 rows v [rows, K]: FP4 packed codes [rows, K/2] + scale
 * bytes [rows, K/block]; MXFP8 codes [rows, K] + E8M0 bytes [rows, K/32];
 * bf16 [rows, 2K] bytes (scales untouched).  `which` 0 uses act_scale_x, 1
 * act_scale_h (NVFP4 only). */
int moe_debug_actquant(moe_layer_t layer, const float* v, int rows, int K,
                       uint8_t* codes, uint8_t* scales, int which, void* stream);

/* ---- multi-layer stacks --------------------------------------------------
 * A stack is L layers of one descriptor that share ONE GPU expert cache: one
 * slot pool of desc->n_slots slots and one LRU table over all layers' experts
 * (key l * E + e for expert e of layer l), as FreeToken keeps one global LRU
 * expert cache across layers ("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net,
 * §二, "LRU 为什么赢" paragraph; juejin.cn overview, §二 "全局 LRU 专家缓存").
 * Every layer has its own router, host expert pool and shared expert, set
 * through its member handle (moe_stack_layer) with the per-layer calls above.
 * A member's step record, statistics and errors are its own; moe_lru_get_state
 * and moe_lru_set_state on any member read or write the shared table, whose
 * expert_of entries are keys; moe_cache_install(member l, e, slot) installs key
 * l E + e.  Members cannot be resized (moe_cache_resize returns
 * MOE_ERR_UNSUPPORTED) or destroyed on their own (MOE_ERR_STATE).  Members
 * share their workspaces, so moe_debug_last_step / moe_debug_last_hidden on a
 * member read what the stack's latest forward of any member left there.
 *
 * moe_stack_forward runs the layers in order, the output of layer l (bf16,
 * [N, d_model]) being the input of layer l + 1 (the MoE sublayers of a
 * transformer with the rest of each block left out).  Decode: each layer's step
 * is moe_forward on the shared cache.  Prefill (whole-layer streaming, the
 * pages' "Prefill: hide the compute in the transfer", zhichai.net §二
 * "Prefill：把计算藏进传输"; juejin.cn §二 "全层双缓冲预填充"): before layer l's
 * step, every expert of layer l is accessed as one table step (hits first,
 * misses ascending) and its misses are copied from the layer's host pool, so
 * the layer's own step finds every routed expert resident.  Prefetch modes:
 *   MOE_PREFETCH_NONE     no prefetch: each layer's step fills its own misses;
 *   MOE_PREFETCH_SERIAL   layer l + 1's prefetch after layer l (n_slots >= E);
 *   MOE_PREFETCH_OVERLAP  layer l + 1's prefetch right after layer l's table
 *                         step, its copies on a few SMs while layer l's GEMMs
 *                         run on the others (n_slots >= 2 E: layer l's experts
 *                         are then never the victims);
 *   MOE_PREFETCH_AUTO     (default) OVERLAP when n_slots >= 2 E, else SERIAL
 *                         when n_slots >= E, else NONE.
 * The table ends in the same state in every mode that prefetches (the same
 * sequence of steps). */
#define MOE_PREFETCH_AUTO    0
#define MOE_PREFETCH_NONE    1
#define MOE_PREFETCH_SERIAL  2
#define MOE_PREFETCH_OVERLAP 3

/* Create a stack of n_layers (1..4096) layers of descriptor desc, sharing
 * desc->n_slots cache slots (1..min(n_layers E, 1024)), on the current device.
 * Returns MOE_ERR_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_OOM / MOE_ERR_CUDA as
 * moe_layer_create. */
int moe_stack_create(const moe_layer_desc* desc, int n_layers, moe_stack_t* out);
/* Synchronises the device, then frees every member and the shared storage. */
int moe_stack_destroy(moe_stack_t stack);
/* Member handle of layer l (owned by the stack). */
int moe_stack_layer(moe_stack_t stack, int l, moe_layer_t* out);
/* Prefetch mode of later prefill forwards; MOE_ERR_UNSUPPORTED when n_slots
 * is too small for the mode. */
int moe_stack_set_prefetch(moe_stack_t stack, int mode);
/* One forward through every layer: x [N, d_model] bf16 -> y [N, d_model] bf16
 * (device or pinned host memory, as moe_forward; the hidden states between
 * layers stay on the device).  regime as moe_forward, one regime for every
 * layer.  A member's error is returned with its message in
 * moe_stack_last_error.  info (may be NULL): regime, n_tokens, n_launches
 * (all layers and prefetches), fused_step (layers run as one fused launch);
 * the per-step counts are -1 (read each member's statistics instead). */
int moe_stack_forward(moe_stack_t stack, const void* x, int N, void* y, void* stream, int regime,
                      moe_forward_info* info);
/* How prefetched experts are copied: MOE_FILL_MEMCPY (default; AUTO means
 * it) -- the host reads the prefetch's step record (mapped pinned memory,
 * polled, bounded) and issues cudaMemcpyAsync per run of consecutive experts
 * on the prefetch's stream (the fill stream when overlapped), so the GEMMs
 * keep every SM; MOE_FILL_KERNEL -- copy kernels on 12 SMs read the step
 * record on the device (no host wait), and an overlapped prefill GEMM leaves
 * those SMs free.  MOE_ERR_ARG for other values. */
int moe_stack_set_prefetch_copy(moe_stack_t stack, int fill);
/* Accumulated prefetch counters: steps, keys accessed, hits, misses
 * (synchronises the device). */
int moe_stack_prefetch_stats(moe_stack_t stack, uint64_t* out4);
/* The last stack call's error message. */
const char* moe_stack_last_error(moe_stack_t stack);

/* ---- allocation-free permutation ----------------------------------------
 * The FreeToken pages have no counterpart to this entry point.  It is for
 * callers that cannot allocate GPU memory themselves: code embedded in a host
 * framework that owns every device allocation, code running under a fixed
 * memory budget, or code that must not call cudaMalloc because that call can
 * synchronise the whole device.  It computes what moe_debug_permute computes
 * (counts [E], offsets [E+1], row_of [N*k], tok_of [N*k] from the sorted top-k
 * ids idx [N, k]; all device pointers, owned by the caller) without a layer
 * handle and without allocating anything: its scratch is one fixed 2 MiB array
 * in the library's device memory, held on every GPU that loads the library
 * until the process exits.  Each row of idx must hold k distinct ids in
 * [0, E), ascending; ids outside [0, E) are skipped (their row_of entry is -1)
 * and duplicate ids in a row give an unspecified permutation, but neither
 * makes the kernels read or write outside the caller's arrays.  Limits:
 * 1 <= E <= 1024, 1 <= k <= min(E, 32),
 * N * k <= 262144 and ceil(N / 128) * E <= 262144; a larger request returns
 * MOE_ERR_ARG and, when errbuf is not NULL, the reason as text in the caller's
 * errbuf (errbuf_len bytes, NUL-terminated).  The first call on a device (and
 * the first after that device's context was destroyed and re-created, e.g. by
 * cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress);
 * make that first call before any stream capture.  Every call shares the one array and finds the
 * previous call's contents in it (each entry a call reads, that call has
 * written first, so nothing needs clearing); calls that overlap on the GPU --
 * on different streams or from different threads -- race, so the caller must
 * order them.  N == 0 is a no-op.  Work is ordered on `stream`. */
int moe_permute_noalloc(const int* idx, int N, int k, int E, int* counts, int* offsets,
                        int* row_of, int* tok_of, void* stream, char* errbuf,
                        size_t errbuf_len);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
