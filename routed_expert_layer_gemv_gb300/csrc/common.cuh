// Internal declarations shared by the CUDA translation units of the layer.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------- dependent launch
// A kernel started with launch_pdl may begin while its predecessor on the
// stream still runs (programmatic dependent launch): it must call pdl_wait()
// before it reads anything the predecessor (or an earlier kernel) writes, and
// it may only write what no running kernel reads.  pdl_trigger() lets the
// successor start early; a kernel whose successor reads anything before its
// own pdl_wait() triggers only after its own pdl_wait(), so those reads see
// the finished work of every kernel before it.  Both are no-ops for kernels
// launched normally.
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  Function attributes are per device, so this is done once
// per (kernel, device) pair -- a process that drives several GPUs sets them on
// each -- under a lock, so concurrent first launches from several threads are
// safe.  Defined in api.cu.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kPrefillTileRows = 128;   // rows of one prefill GEMM tile (its MMA M): the padded-block unit
constexpr int kWarp = 32;

// ---------------------------------------------------------------- formats
// E8M0 scale byte -> 2^(x-127) (x = 0 is the fp32 subnormal 2^-127).
MOE_DEV float e8m0_to_f32(uint32_t x) {
  return x == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(x << 23);
}

// E4M3 (fn) byte -> fp32: bias 7 -> fp32 bias 127; exponent 0 is subnormal.
MOE_DEV float e4m3_to_f32(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v = e == 0 ? (float)m * (1.0f / 512.0f) : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -v : v;
}

// Two E2M1 codes (one byte, low nibble first) -> f16x2, exact.
MOE_DEV uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(out) : "r"(byte));
  return out;
}

// ---------------------------------------------------------------- step record
// What one step's routing and LRU update decided; written by the LRU kernel,
// copied to pinned host memory for the fill issue.  Arrays hold |U| entries
// in access order (hits ascending id, then misses ascending id).  acc_slot is
// the LRU slot an access ends up in (logical); acc_buf the buffer of the slot
// pool it is computed from and, for a miss, filled into (physical).
struct StepRecord {
  int U;        // distinct routed experts
  int n_hit;
  int n_miss;
  int S;        // slots (wave length)
  unsigned long long seq;   // host copy only: step number, written last
  int pad[2];
  // followed by int acc_expert[E], acc_slot[E], acc_evicted[E], acc_buf[E]
};
__host__ __device__ inline int* rec_expert(StepRecord* r) { return reinterpret_cast<int*>(r + 1); }
__host__ __device__ inline int* rec_slot(StepRecord* r, int E) { return rec_expert(r) + E; }
__host__ __device__ inline int* rec_evicted(StepRecord* r, int E) { return rec_expert(r) + 2 * E; }
__host__ __device__ inline int* rec_buf(StepRecord* r, int E) { return rec_expert(r) + 3 * E; }
// bytes the host reads back (header and the four access arrays)
inline size_t rec_bytes(int E) { return sizeof(StepRecord) + 4 * sizeof(int) * (size_t)E; }
// Device-only tail: per access i, {buffer (acc_buf, -1 when the record is
// inconsistent), first permuted row, rows, tokens}, so a kernel
// finds an access's weights and tokens with one 16-byte load.  tokens = the
// first row's token (low 16 bits; 0xffff in the high half when it is not
// known).
__host__ __device__ inline int4* rec_entry(StepRecord* r, int E) {
  const size_t off = (sizeof(StepRecord) + 4 * sizeof(int) * (size_t)E + 15) & ~size_t(15);
  return reinterpret_cast<int4*>(reinterpret_cast<char*>(r) + off);
}
inline size_t rec_dev_bytes(int E) { return ((rec_bytes(E) + 15) & ~size_t(15)) + sizeof(int4) * (size_t)E; }

// ---------------------------------------------------------------- formats
// Bits per weight element and the K elements one block scale covers (0: the
// format has no block scales).  The prefill regime's activations take the
// same element type and block (FP4 x FP4, MXFP8 x MXFP8, bf16 x bf16).
__host__ __device__ constexpr int fmt_code_bits(int fmt) {
  return fmt == MOE_MXFP8 ? 8 : fmt == MOE_BF16 ? 16 : 4;
}
__host__ __device__ constexpr int fmt_block(int fmt) {
  return fmt == MOE_NVFP4 ? 16 : fmt == MOE_BF16 ? 0 : 32;
}
// Scale bytes of a K-long row (0 without block scales).
__host__ __device__ constexpr int fmt_scale_row(int fmt, int K) {
  return fmt_block(fmt) ? K / fmt_block(fmt) : 0;
}

// ---------------------------------------------------------------- layer geometry
struct Geo {
  int E, k, d, f, S, fmt, has_shared, norm_topk, has_bias;
  int afmt;                    // activation format of the prefill regime (fmt, or MXFP8 on MXFP4: W4A8)
  int X;                       // spare buffers: the pool holds S + 1 + X (the shared expert's is S)
  // The slot table is keyed: key = key0 + expert.  A lone layer has key0 = 0
  // and keys = E; layer l of a stack of L layers sharing one pool and one
  // table has key0 = l E and keys = L E (slot_of has `keys` entries,
  // expert_of holds keys).
  int key0, keys;
  int shb;                     // the pool buffer of this layer's shared expert (S for a lone layer)
  int nbuf;                    // buffers in the pool (S + 1 + X, plus one per further stack layer)
  int blk;                     // 32 (MXFP4) or 16 (NVFP4)
  size_t ebytes;               // padded bytes of one expert
  size_t off_codes[3], off_scales[3], off_tscale;
};

// Work-range selectors of the expert FFN launches (resolved on the device
// from the StepRecord so a launch needs no host round trip): the step's
// hits, its misses, or every access (with GemvArgs::host_pool set, the misses
// are then read from the host pool and written on to their slots).
enum RangeMode : int { kRangeHits = 0, kRangeMisses = 1, kRangeAll = 2 };

// Buffers of the slot pool.  The pool holds S + 1 + X expert buffers (the
// shared expert's is buffer S); LRU slot s lives in buffer buf[s] and
// buf[S .. S + X) lists the spare ones (buf, S + X ints, kept by the LRU
// kernel, initially s and S + 1 + j).  Misses of the first wave (access index
// i < S) are filled into their LRU slot's buffer (a free or stale one); a
// later miss would evict a slot the same step still reads, so it is filled
// into spare buf[S + (i - S)], and when it keeps that slot at the end of the
// step the LRU kernel swaps the two buffers: the slot's old buffer becomes
// the spare.  No expert is ever copied within the pool.

// A long miss list is cut into chunks, each filled and then computed on its
// own so its expert FFN runs while later fills are still in flight: up to
// kMissChunks chunks of at least kMissesPerChunk misses.  The last chunk takes
// kMissesPerChunk misses (its expert FFN, which runs after the last fill, is
// the step's tail) and the others share the rest equally.  Chunk c of nch over
// m misses is [lo, hi) (offsets from the first miss); host and device use this
// one split.
constexpr int kMissChunks = 4;
constexpr int kMissesPerChunk = 3;
__host__ __device__ inline int miss_chunks(int m) {
  const int n = m / kMissesPerChunk;
  return n < 1 ? 1 : n > kMissChunks ? kMissChunks : n;
}
__host__ __device__ inline void miss_chunk(int m, int c, int nch, int* lo, int* hi) {
  if (nch <= 1) {
    *lo = 0;
    *hi = m;
    return;
  }
  const int rest = m - (m < kMissesPerChunk ? m : kMissesPerChunk);
  if (c >= nch - 1) {
    *lo = rest;
    *hi = m;
    return;
  }
  *lo = (int)((long long)rest * c / (nch - 1));
  *hi = (int)((long long)rest * (c + 1) / (nch - 1));
}

// ---------------------------------------------------------------- launchers
// router.cu
// counter: kRouterCounterBytes of zeroed device memory (one word per token
// tile of the one-launch path for N <= 64), left zeroed
constexpr size_t kRouterCounterBytes = 64;
// Whl (may be null): W_r split into three bf16 parts [3][E][d]
// (launch_router_split); with it, batches over 64 tokens take the tensor-core
// logits kernel
// (xexp may be null when no decode GEMV follows; err: the layer's device
// error word, set when a bounded wait of the tcgen05 logits kernel runs out)
cudaError_t launch_router(const Geo& g, const __nv_bfloat16* x, int N, const float* Wr,
                          const __nv_bfloat16* Whl, const float* bias, float* logits, int* idx,
                          float* gates, int* xexp, unsigned int* counter, int* err, float* part2,
                          cudaStream_t st);
// router_tc.cu: logits of batches over 64 tokens on tcgen05 (E a multiple of
// 16 up to 256, d a multiple of 64; cudaErrorNotSupported otherwise), then
// xexp when asked.  part2 (may be null; [N, E]): room for the second K half's
// partial sums; *split = 2 when they were written (the logits then hold the
// first half's, without the bias), else 1
bool router_tc5_shape_ok(const Geo& g);
cudaError_t launch_router_tc5(const Geo& g, const __nv_bfloat16* x, int N, const __nv_bfloat16* Whl,
                              const float* bias, float* logits, float* part2, int* split, int* xexp, int* err,
                              cudaStream_t st);
cudaError_t launch_router_split(const Geo& g, const float* Wr, __nv_bfloat16* Whl, cudaStream_t st);
// permute.cu
size_t permute_scratch_bytes(const Geo& g, int max_tokens);
cudaError_t launch_permute(const Geo& g, const int* idx, int N, int* counts, int* offsets,
                           int* row_of, int* tok_of, void* scratch, cudaStream_t st);
// its first and last launches for N > 128 (block histograms and in-block
// ranks into scratch; rows from them and the offsets), for a caller that
// runs the scan itself (launch_scan_lru)
cudaError_t launch_perm_hist(const Geo& g, const int* idx, int N, void* scratch, cudaStream_t st);
cudaError_t launch_perm_scatter(const Geo& g, const int* idx, int N, const int* offsets, void* scratch,
                                int* row_of, int* tok_of, cudaStream_t st);
// lru.cu
// stats (may be null): steps, distinct experts, hits, misses, accumulated
// offsets (may be null: entries then get no rows) = the permutation's
// expert row offsets, for the record's entry table
// host_rec (may be null): mapped pinned copy of the record, written by the
// kernel itself, seq last, so the host can poll it instead of a copy + event
// buf: the slot -> buffer map and spare list (S + X ints, updated in place)
cudaError_t launch_lru_step(const Geo& g, const int* counts, const int* offsets, int* slot_of,
                            int* expert_of, unsigned long long* stamp, unsigned long long* clock,
                            int* buf, StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                            unsigned long long seq, cudaStream_t st);
// N > 128: the permutation's scan (after launch_perm_hist), the prefill's
// padded blocks (pbase, may be null: E + 2 ints, as launch_gather_quant
// writes them) and the LRU step, in one launch; with pbase and tiles (the
// prefill tile workspace, prefill_tile_bytes; n_tiles its counts) also the
// tile list of the step's hits and shared expert, as launch_prefill_gemms
// builds it for its first range
cudaError_t launch_scan_lru(const Geo& g, int N, void* perm_scratch, int* counts, int* offsets, int* pbase,
                            int* slot_of, int* expert_of, unsigned long long* stamp, unsigned long long* clock,
                            int* buf, StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                            unsigned long long seq, void* tiles, int* n_tiles, cudaStream_t st);
cudaError_t launch_lru_install(const Geo& g, int expert, int slot, int* slot_of, int* expert_of,
                               unsigned long long* stamp, unsigned long long* clock,
                               cudaStream_t st);
// Drop the misses of the step in `rec` from the table (their slots become
// free): the recovery of a step whose fills could not be issued.
cudaError_t launch_lru_drop_misses(const Geo& g, const StepRecord* rec, int* slot_of, int* expert_of,
                                   cudaStream_t st);
// permutation + LRU step in one CTA, for N <= 128 tokens
cudaError_t launch_route_tail(const Geo& g, const int* idx, int N, int* counts, int* offsets,
                              int* row_of, int* tok_of, int* slot_of, int* expert_of,
                              unsigned long long* stamp, unsigned long long* clock, int* buf,
                              StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                              unsigned long long seq, cudaStream_t st);
cudaError_t launch_counts_from_list(const Geo& g, const int* experts, int n, int* counts,
                                    cudaStream_t st);
// gemv.cu
struct GemvArgs {
  const uint8_t* slots;        // slot pool base
  const uint8_t* shared_w;     // shared expert (or null)
  const StepRecord* rec;
  const int* offsets;          // [E+1]
  const int* tok_of;           // [N*k]
  int N;
  int mode;                    // RangeMode
  int chunk, n_chunks;         // kRangeMisses: chunk `chunk` of n_chunks (miss_chunk) of the misses
  const uint8_t* host_pool;    // kRangeAll: device address of the pinned host pool the misses stream from
  int with_shared;             // also run the shared expert (rows N*k .. N*k+N)
  int* err;                    // set to 1 when a bounded wait gives up
  float* hmax;                 // [rows][2][d_ff / 64]: max |W_g x|, |W_u x| per 64 columns
  long long wait_cycles;       // limit of the launch's bounded waits (SM clock cycles; <= 0: ~2 s)
};
struct GemvPlan;               // tensor maps of the slot pool's weight codes
bool gemv_shape_ok(const Geo& g);
GemvPlan* gemv_plan_create(const Geo& g, const uint8_t* slots);
void gemv_plan_destroy(GemvPlan* pl);
bool gemv_plan_ready(const GemvPlan* pl);
// x must be 16-byte aligned; h holds 2 * d_ff floats per row (phase 1
// writes W_g x and W_u x, phase 2 forms SiLU(a) * u from them).  ev (may be
// null): 4 events recorded before/after phase 1 and phase 2.  phases: 1, 2 or
// 3 (both) -- the phases a call launches; num_sms: the SMs the grids may use
cudaError_t launch_gemv_decode(const Geo& g, const GemvPlan* pl, const GemvArgs& a,
                               const __nv_bfloat16* x, const int* xexp, float* h, float* O,
                               int n_ent_max, int num_sms, cudaStream_t st, const cudaEvent_t* ev,
                               int phases);
// prefill.cu
struct PrefillPlan;
bool prefill_shape_ok(const Geo& g);
PrefillPlan* prefill_plan_create(const Geo& g, const uint8_t* slots, const uint8_t* xq_codes,
                                 size_t xq_rows, const uint8_t* hq_codes);
void prefill_plan_destroy(PrefillPlan* pl);
bool prefill_plan_ready(const PrefillPlan* pl);
size_t prefill_tile_bytes(const Geo& g, int N);            // tiles, then the launch's entries
int prefill_max_tiles(const Geo& g, int N);                // tiles of one launch at most (its entries follow)
size_t prefill_act_scale_bytes(const Geo& g, int N, int K);  // x (K = d) or h (K = f) block scales
size_t prefill_wscale_bytes(const Geo& g);                   // interleaved weight scales, per pool buffer
size_t prefill_wtag_ints(const Geo& g);                      // their tags (ints, -1 = none) and counts (0)
// Activations of the prefill regime: pbase (E + 2 ints) <- the padded
// 128-row blocks of each expert's rows (from counts), then x quantised into
// its permuted rows (row_of [N, k], ids idx [N, k]) with its block scales by
// padded block (the tcgen05.cp layout)
cudaError_t launch_gather_quant(const Geo& g, const __nv_bfloat16* x, const int* idx, const int* row_of,
                                const int* counts, const int* offsets, int N, float gx, int* pbase,
                                bool pbase_ready, uint8_t* codes, uint8_t* scales, cudaStream_t st);
// ev (may be null): 4 events around phase 1 and phase 2; wsf: prefill_wscale_bytes,
// wtag: prefill_wtag_ints (a buffer whose weights are those its scales were
// laid out for, and that this step did not refill, keeps them)
cudaError_t launch_prefill_gemms(const Geo& g, const PrefillPlan* pl, const StepRecord* rec,
                                 const int* offsets, const int* pbase, int N, int mode, int with_shared,
                                 void* tiles, int* n_tiles, const uint8_t* slots,
                                 const uint8_t* xq_scales, uint8_t* hq_codes, uint8_t* hq_scales, uint8_t* wsf,
                                 int* wtag, float* O, float gx, float gh, int* err, int num_sms, cudaStream_t st,
                                 const cudaEvent_t* ev, bool tiles_ready = false);
// h's block scales of the last prefill call back to rows [rows][f / block]
cudaError_t launch_untile_hscales(const Geo& g, const uint8_t* tiled, const int* offsets, const int* pbase, int N,
                                  uint8_t* out, cudaStream_t st);
// fill.cu: copy every miss of the step from the (device-addressable) host pool
// into the buffer the record names (acc_buf)
cudaError_t launch_fill_copy(const Geo& g, const StepRecord* rec, int max_misses,
                             const uint8_t* pool_dev, uint8_t* slots, cudaStream_t st);
// the same copy by kFillSms CTAs, one per SM, for chunk `chunk` of the miss
// list (miss_chunk); the decode expert GEMV leaves those SMs free
constexpr int kFillSms = 12;
cudaError_t launch_fill_sm(const Geo& g, const StepRecord* rec, int chunk, const uint8_t* pool_dev,
                           uint8_t* slots, cudaStream_t st);
// dst <- src (bytes a multiple of 16, 16-byte aligned; src may be mapped host memory)
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t st);
// combine.cu
// The prefill GEMM writes O as f16 rows [rows][d] in the first half of the
// O buffer, each row's 128-column blocks scaled by 2^-s; the exponents s
// (int8, [rows][d / 128]) follow the f16 rows.
inline int8_t* prefill_o_exp(const Geo& g, const float* O, int N) {
  const size_t rows = (size_t)N * g.k + (g.has_shared ? N : 0);
  return reinterpret_cast<int8_t*>(const_cast<float*>(O)) + rows * g.d * 2;
}
// O: fp32 rows, or (o_f16) the prefill GEMM's scaled f16 rows
cudaError_t launch_combine(const Geo& g, const float* O, bool o_f16, const float* gates, const int* row_of,
                           int N, __nv_bfloat16* y, cudaStream_t st);
// debug.cu
cudaError_t launch_dequant(const Geo& g, const uint8_t* expert, int m, float* out, cudaStream_t st);
cudaError_t launch_actquant(const Geo& g, const float* v, int rows, int K, uint8_t* codes,
                            uint8_t* scales, float gscale, cudaStream_t st);

}  // namespace moe
