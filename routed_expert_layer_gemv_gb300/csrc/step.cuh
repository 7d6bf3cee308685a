// Host interface of the fused decode step (step.cu): one cooperative launch
// per decode step of a small batch.
#pragma once
#include "common.cuh"
#include "gemv_dev.cuh"

namespace moe {

constexpr int kStepMaxTokens = 16;        // tokens of one fused step
constexpr int kStepMaxE = gv::kThreads;   // experts: one per thread of a CTA in the routing and the LRU step
constexpr int kStepMaxPairs = 256;        // N * k (so also the step's distinct experts)
constexpr int kStepSmemMax = 232448 - 2048;   // dynamic shared memory (227 KB less the static part)
constexpr int kStepAutoPairs = 32;        // MOE_DECODE_AUTO fuses steps of at most this many (token, expert) pairs

// Buffers of one fused step (device pointers unless noted).
struct StepArgs {
  const __nv_bfloat16* x;      // [N, d] (16-byte aligned)
  const float* Wr;             // [E, d]
  const float* bias;           // [E] or null
  float* logits;               // [N, E] workspace (every CTA writes its experts', every CTA reads all)
  int *idx, *counts, *offsets, *row_of, *tok_of;   // the step's routing, as the chained path writes it
  float* gates;
  int *slot_of, *expert_of, *buf;                 // the slot table (updated by CTA 0)
  unsigned long long *stamp, *clock;
  StepRecord* rec;             // the step record (CTA 0's LRU step writes it)
  unsigned long long* stats;
  unsigned long long* ready;   // publication word of the misses' buffers
  unsigned long long seq;      // this step's value of it
  unsigned long long* gbar;    // the three grid barriers' arrival counters
  unsigned long long gbar_base;   // their value when the launch starts (the launch adds G to each)
  float* h;                    // [rows, 2 d_ff] phase-1 outputs
  float* O;                    // [rows, d] phase-2 outputs
  __nv_bfloat16* y;            // [N, d] (device or mapped pinned host memory)
  unsigned long long* trace;   // [G][kStepMarks] global-timer stamps per CTA, or null
  int ctl_off;                 // set by launch_step
};

// Marks of the per-CTA timeline (moe_debug_step_trace): kernel start, logits
// written, barrier 1 passed, top-k done, permutation done, access table
// built, phase-1 outputs written, barrier 2 passed, phase-2 outputs written,
// barrier 3 passed, done (global timer, ns); then the SM clock (clock64) at
// the first and the last mark, which give the clock rate the step ran at;
// then (global timer) the first phase-1 stage landed and the last consumed,
// as compute warp 0 saw them, the same for phase 2, and the first phase-2
// activation block staged by the epilogue (left from an earlier step when the
// CTA had no such work).
constexpr int kStepMarks = 18;

struct StepPlan {
  gv::SG p1, p2;   // the two phases' geometry, sharing one ring layout
  int ctl_off;     // offset of the routing copy in the aligned dynamic shared memory
  int smem;        // dynamic shared memory bytes
};

// Whether a decode step of N tokens fits the fused launch (and its plan).
bool step_plan(const Geo& g, int N, StepPlan* out);

// One fused step on `grid` CTAs (the SM count: one per SM, all resident).
// a: the expert-FFN arguments (slots, N, err, hmax, host pool for fused
// fills, wait limit); the launch adds `grid` to each barrier counter.
cudaError_t launch_step(const Geo& g, const GemvPlan* pl, const GemvArgs& a, StepArgs s, const StepPlan& P,
                        int grid, cudaStream_t st);

}  // namespace moe
