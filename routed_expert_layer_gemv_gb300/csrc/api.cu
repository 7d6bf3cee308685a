// Host side of the C ABI (include/moe.h): validation, device buffers, the
// per-step launch sequence, and the host->slot fills of cache misses.
//
// One step of moe_forward (decode regime; the prefill regime quantises the
// permuted activations to FP4 first and runs the tcgen05 grouped GEMM in place
// of the GEMV):
//   caller stream: router -> permute -> LRU step -> [record copy to host]
//                  -> expert GEMV over the hits (+ shared expert)
//   host:          wait for the record, then for every miss at once:
//   fill stream:   cudaMemcpyAsync pinned host expert -> its slot's buffer
//                  (first wave of n_slots accesses) or a spare buffer (later
//                  accesses, whose LRU slots this step still reads; the LRU
//                  kernel makes the spare the slot's buffer for later steps)
//   caller stream: wait for the fills -> expert GEMV over all misses
//                  -> combine -> y
// The hits are computed while the host reads the record and the fills are in
// flight.  When every expert is resident (n_slots >= E, all installed) no
// miss can happen and the step runs without any host wait.
//
// The fill design follows the pages' decode path: misses are loaded into the
// GPU's LRU expert cache from host memory ("FreeToken：把 284B MoE 塞进游戏
// PC", zhichai.net, §二 "Decode" paragraph).  The pages' alternative of
// running some misses on the CPU (their q* split) is not part of this library.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <chrono>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"
#include "step.cuh"

using namespace moe;

namespace moe {

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;   // (kernel, device) -> limit set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

}  // namespace moe

constexpr size_t kDirectHostBytes = 256 * 1024;   // host x / y read and written in place up to this size
constexpr int kMaxStackLayers = 4096;

struct moe_layer {
  moe_layer_desc desc{};
  Geo g{};
  moe_expert_layout lay{};
  int device = 0;
  int num_sms = 0;
  std::vector<void*> dev_allocs;
  void* pinned_rec = nullptr;
  // device buffers
  uint8_t* slots = nullptr;
  uint8_t* shared_w = nullptr;
  float* Wr = nullptr;
  __nv_bfloat16* Wr_hl = nullptr;   // W_r as three bf16 parts summing to it (tensor-core router)
  float* bias = nullptr;
  int* slot_of = nullptr;
  int* expert_of = nullptr;
  unsigned long long* stamp = nullptr;
  int* buf = nullptr;                // slot -> pool buffer map, then the spare buffers (S + X)
  unsigned long long* clock = nullptr;
  float* logits2 = nullptr;     // second K half's partial logits (large batches)
  float* logits = nullptr;
  int* idx = nullptr;
  float* gates = nullptr;
  int* xexp = nullptr;
  int* counts = nullptr;
  int* offsets = nullptr;
  int* row_of = nullptr;
  int* tok_of = nullptr;
  void* perm_scratch = nullptr;
  StepRecord* rec = nullptr;
  StepRecord* rec_host = nullptr;
  StepRecord* rec_host_dev = nullptr;         // rec_host as the device sees it (mapped)
  unsigned long long step_seq = 0;            // sequence number of the last polled record
  float* h = nullptr;
  float* hmax = nullptr;          // decode: per-row maxima of phase 1 per 64 columns
  float* O = nullptr;
  __nv_bfloat16* x_stage = nullptr;
  __nv_bfloat16* y_stage = nullptr;
  int* list_dev = nullptr;
  int list_cap = 0;
  // prefill regime
  uint8_t* xq_codes = nullptr;   // permuted FP4 activations [(rows + 128), d/2]
  uint8_t* xq_scales = nullptr;
  uint8_t* hq_codes = nullptr;   // FP4 h [(rows + 128), f/2]
  uint8_t* hq_scales = nullptr;
  int* pbase = nullptr;          // padded 128-row block of each expert's rows (E + 2)
  uint8_t* wsf = nullptr;        // the pool buffers' weight scales, interleaved for tcgen05.cp
  int* wtag = nullptr;           // per buffer: key of the weights wsf holds scales for (-1: none), then counts
  void* tiles = nullptr;
  int* n_tiles = nullptr;
  PrefillPlan* plan = nullptr;
  GemvPlan* gplan = nullptr;
  unsigned int* rcounter = nullptr;  // CTA counters of the one-launch router (one per token tile)
  int* err_host = nullptr;       // kernels' timeout flag (mapped pinned memory)
  int* err_dev = nullptr;
  // host state
  const uint8_t* host_pool = nullptr;
  size_t host_pool_bytes = 0;
  bool router_set = false;
  bool shared_set = false;
  cudaStream_t fill = nullptr;                // miss fills: one copy queue (more add no bandwidth on the host link)
  cudaEvent_t ev_chunk[kMissChunks] = {};     // the fills of each miss chunk have landed
  cudaEvent_t ev_route = nullptr, ev_fill = nullptr;
  int fill_mode = MOE_FILL_MEMCPY;    // set by the pool's registration unless the caller chose one
  bool fill_mode_chosen = false;
  const uint8_t* pool_dev = nullptr;          // device address of the host pool
  unsigned long long* stats = nullptr;        // steps, distinct, hits, misses
  std::vector<int> mirror_own;   // key per slot as far as the host knows (the pool owner's)
  std::vector<int>* mir = nullptr;   // the mirror of the table this layer uses (its own, or its stack's)
  // stack membership: layer `index` of a stack whose pool, slot table and
  // workspaces belong to its layer 0 (owner = false for the others)
  moe_stack* stack = nullptr;
  int index = 0;
  bool owner = true;
  bool assume_resident = false;        // set by the stack around a forward whose experts it prefetched
  cudaEvent_t ev_after_route = nullptr;   // set by the stack: recorded after the step's LRU update
  int gemm_sms = 0;                    // set by the stack: SMs the prefill GEMM may use (0: all)
  std::string err;
  // kernel timing (moe_profile)
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_pool;
  size_t prof_used = 0;
  std::vector<int> prof_kind;          // one entry per timed launch (pair of events)
  int launches = 0;                    // kernels launched by the current call
  int last_N = 0;                      // tokens of the last moe_forward (0: none yet)
  // fused decode step
  int decode_path = MOE_DECODE_AUTO;
  bool step_failed = false;            // a cooperative launch was refused once: use the chain
  unsigned long long* gbar = nullptr;  // arrival counters of the fused step's three grid barriers (device)
  unsigned long long gbar_base = 0;    // its value before the next fused step
  unsigned long long* ready = nullptr; // publication word of a fused step's miss buffers (device)
  unsigned long long* step_trace = nullptr;   // per-CTA timeline of the last fused step (device, under moe_profile)
  int step_trace_grid = 0;
  unsigned long long ready_seq = 0;
  bool inject_fill = false;            // test hook: the next host-issued fill fails before its copy
  long long inject_wait = 0;           // test hook: wait limit (cycles) of the next forward's expert FFN
  bool last_prefill = false;           // regime of the last moe_forward
};

// A stack of layers of one geometry that share one slot pool and one LRU
// table keyed by (layer, expert).
struct moe_stack {
  std::vector<moe_layer*> layers;
  int prefetch = MOE_PREFETCH_AUTO;
  int prefetch_copy = MOE_FILL_MEMCPY;           // how prefetched experts are copied (MOE_FILL_MEMCPY / KERNEL)
  __nv_bfloat16* hid[2] = {nullptr, nullptr};   // hidden states between layers [max_tokens, d]
  int* ones = nullptr;                           // [E] ones: a whole layer as a step's counts
  unsigned long long* pf_stats = nullptr;        // prefetch steps, keys, hits, misses
  cudaEvent_t ev_pf = nullptr, ev_in = nullptr, ev_route = nullptr;
  std::string err;
};

namespace {

// Test hooks of the error paths (moe_debug_alloc_fault): the nth allocation
// from now fails without being attempted; live counts of what the library
// holds, for leak checks.
std::atomic<long long> g_alloc_countdown{0};
std::atomic<long long> g_live_dev{0}, g_live_host{0};

bool alloc_fault_due() {
  long long c = g_alloc_countdown.load();
  while (c > 0)
    if (g_alloc_countdown.compare_exchange_weak(c, c - 1)) return c == 1;
  return false;
}

int fail(moe_layer* L, int code, const char* fmt, ...) {
  if (L) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    L->err = buf;
  }
  return code;
}

int cuda_fail(moe_layer* L, cudaError_t e, const char* what) {
  return fail(L, MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(L, call)                                   \
  do {                                                      \
    cudaError_t e_ = (call);                                \
    if (e_ != cudaSuccess) return cuda_fail((L), e_, #call); \
  } while (0)

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool is_pow2_float(float v) {
  if (!(v > 0.f) || !std::isfinite(v)) return false;
  int ex;
  return std::frexp(v, &ex) == 0.5f;
}

int check_desc(const moe_layer_desc* d, std::string* why, int max_slots) {
  char buf[256];
  auto bad = [&](const char* m) { *why = m; return MOE_ERR_ARG; };
  if (!d) return bad("descriptor is NULL");
  if (d->E < 1 || d->E > kMaxE) return bad("E must be in [1, 1024]");
  if (d->k < 1 || d->k > d->E || d->k > kMaxK) return bad("k must be in [1, min(E, 32)]");
  if (d->d_model <= 0 || d->d_model % 128) return bad("d_model must be a positive multiple of 128");
  if (d->d_ff <= 0 || d->d_ff % 128) return bad("d_ff must be a positive multiple of 128");
  if (d->n_slots < 1 || d->n_slots > max_slots) {
    snprintf(buf, sizeof buf, "n_slots must be in [1, %d]", max_slots);
    *why = buf;
    return MOE_ERR_ARG;
  }
  if (d->fmt != MOE_MXFP4 && d->fmt != MOE_NVFP4 && d->fmt != MOE_MXFP8 && d->fmt != MOE_BF16)
    return bad("fmt must be MOE_MXFP4, MOE_NVFP4, MOE_MXFP8 or MOE_BF16");
  if (d->prefill_act_bits != 0 && d->prefill_act_bits != fmt_code_bits(d->fmt) &&
      !(d->fmt == MOE_MXFP4 && d->prefill_act_bits == 8))
    return bad("prefill_act_bits must be 0, the weights' code bits, or 8 on MOE_MXFP4 weights");
  if (d->max_tokens < 1) return bad("max_tokens must be >= 1");
  if ((long long)d->max_tokens * (d->k + 1) > (1LL << 30)) return bad("max_tokens * (k+1) too large");
  if (d->fmt == MOE_NVFP4 && (!is_pow2_float(d->act_scale_x) || !is_pow2_float(d->act_scale_h))) {
    snprintf(buf, sizeof buf, "NVFP4 act_scale_x/act_scale_h must be positive powers of two");
    *why = buf;
    return MOE_ERR_ARG;
  }
  return MOE_OK;
}

void fill_layout(const moe_layer_desc* d, moe_expert_layout* l) {
  const size_t D = d->d_model, F = d->d_ff;
  const size_t blk = fmt_block(d->fmt);          // 0: no scales
  const size_t cb2 = fmt_code_bits(d->fmt);      // bits per element
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  l->gate_codes = take(F * D * cb2 / 8);
  l->up_codes = take(F * D * cb2 / 8);
  l->down_codes = take(D * F * cb2 / 8);
  l->gate_scales = take(blk ? F * D / blk : 0);
  l->up_scales = take(blk ? F * D / blk : 0);
  l->down_scales = take(blk ? D * F / blk : 0);
  l->tensor_scales = take(16);
  l->bytes = off;
}

Geo make_geo(const moe_layer_desc* d, const moe_expert_layout* l) {
  Geo g{};
  g.E = d->E; g.k = d->k; g.d = d->d_model; g.f = d->d_ff; g.S = d->n_slots; g.fmt = d->fmt;
  g.afmt = d->fmt == MOE_MXFP4 && d->prefill_act_bits == 8 ? MOE_MXFP8 : d->fmt;
  g.has_shared = d->has_shared ? 1 : 0; g.norm_topk = d->norm_topk ? 1 : 0;
  g.has_bias = d->has_bias ? 1 : 0;
  g.blk = fmt_block(d->fmt);
  g.ebytes = l->bytes;
  g.off_codes[0] = l->gate_codes; g.off_codes[1] = l->up_codes; g.off_codes[2] = l->down_codes;
  g.off_scales[0] = l->gate_scales; g.off_scales[1] = l->up_scales; g.off_scales[2] = l->down_scales;
  g.off_tscale = l->tensor_scales;
  g.key0 = 0;
  g.keys = g.E;
  g.shb = g.S;
  g.nbuf = g.S + 1;   // + X once known
  return g;
}

template <class T>
int dalloc(moe_layer* L, T** p, size_t bytes) {
  void* q = nullptr;
  if (alloc_fault_due()) return fail(L, MOE_ERR_OOM, "cudaMalloc(%zu) failed: injected by the test hook", bytes);
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(L, MOE_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  L->dev_allocs.push_back(q);
  g_live_dev++;
  *p = static_cast<T*>(q);
  return MOE_OK;
}

// Mapped pinned host memory (the device address is looked up by the caller).
int halloc(moe_layer* L, void** p, size_t bytes) {
  *p = nullptr;
  if (alloc_fault_due()) return fail(L, MOE_ERR_OOM, "cudaHostAlloc(%zu) failed: injected by the test hook", bytes);
  if (cudaHostAlloc(p, bytes, cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return fail(L, MOE_ERR_OOM, "cudaHostAlloc(%zu) failed", bytes);
  }
  g_live_host++;
  return MOE_OK;
}

void hfree(void* p) {
  if (p) {
    cudaFreeHost(p);
    g_live_host--;
  }
}

void release(moe_layer* L) {
  for (cudaEvent_t e : L->prof_pool) cudaEventDestroy(e);
  L->prof_pool.clear();
  for (void* p : L->dev_allocs) {
    cudaFree(p);
    g_live_dev--;
  }
  L->dev_allocs.clear();
  hfree(L->pinned_rec);
  L->pinned_rec = nullptr;
  hfree(L->err_host);
  L->err_host = nullptr;
  if (!L->owner) return;   // the rest belongs to the stack's layer 0
  if (L->plan) prefill_plan_destroy(L->plan);
  L->plan = nullptr;
  if (L->gplan) gemv_plan_destroy(L->gplan);
  L->gplan = nullptr;
  if (L->ev_route) cudaEventDestroy(L->ev_route);
  if (L->ev_fill) cudaEventDestroy(L->ev_fill);
  for (int i = 0; i < kMissChunks; ++i) {
    if (L->ev_chunk[i]) cudaEventDestroy(L->ev_chunk[i]);
    L->ev_chunk[i] = nullptr;
  }
  if (L->fill) cudaStreamDestroy(L->fill);
  L->fill = nullptr;
  L->ev_route = L->ev_fill = nullptr;
}

// Where p lives: device memory of `device` (*on_device), or host memory;
// *mapped = the device address of pinned host memory the device can reach
// through unified addressing (null for pageable memory).
int pointer_kind(const void* p, bool* on_device, int device, const void** mapped) {
  cudaPointerAttributes a{};
  *mapped = nullptr;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *on_device = false;
    return MOE_OK;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    if (a.device != device) return MOE_ERR_ARG;
    *on_device = true;
  } else {
    *on_device = false;
    if (a.type == cudaMemoryTypeHost) *mapped = a.devicePointer;
  }
  return MOE_OK;
}

// Every key of the table resident: then no step can miss or evict (the
// host mirror is exact while nothing can be evicted; with fewer slots than
// keys, device-side steps may evict without the host knowing, so the answer
// is no).
bool all_resident(const moe_layer* L) {
  if (L->g.S < L->g.keys) return false;
  int n = 0;
  for (int e : *L->mir) n += e >= 0 ? 1 : 0;
  return n == L->g.keys;
}

// Apply a step record to the host mirror of the slot table.
void mirror_apply(moe_layer* L, const StepRecord* r) {
  const int U = r->U, S = r->S, E = L->g.E;
  const int* ae = rec_expert(const_cast<StepRecord*>(r));
  const int* as = rec_slot(const_cast<StepRecord*>(r), E);
  for (int i = std::max(0, U - S); i < U; ++i) (*L->mir)[as[i]] = L->g.key0 + ae[i];
}

// A miss of record r left the cache again (its fill failed).
void mirror_drop_misses(moe_layer* L, const StepRecord* r) {
  const int E = L->g.E;
  const int* ae = rec_expert(const_cast<StepRecord*>(r));
  const int* as = rec_slot(const_cast<StepRecord*>(r), E);
  for (int q = r->n_hit; q < r->U; ++q)
    if ((*L->mir)[as[q]] == L->g.key0 + ae[q]) (*L->mir)[as[q]] = -1;
}

constexpr size_t kProfPairs = 16384;

// Two events bracketing one launch of class `kind` (null when timing is off
// or the pool is used up); the start event is recorded on `st` here.
cudaEvent_t* prof_begin(moe_layer* L, int kind, cudaStream_t st) {
  if (!L->prof_on || L->prof_used + 2 > L->prof_pool.size()) return nullptr;
  cudaEvent_t* e = &L->prof_pool[L->prof_used];
  L->prof_used += 2;
  L->prof_kind.push_back(kind);
  cudaEventRecord(e[0], st);
  return e;
}

void prof_end(cudaEvent_t* e, cudaStream_t st) {
  if (e) cudaEventRecord(e[1], st);
}

// A buffer a fill may write: an LRU slot's or a spare, never the shared expert's.
bool buf_ok(const Geo& g, int b) { return b >= 0 && b <= g.S + g.X && b != g.S; }

// Forget every buffer's laid-out weight scales (the next prefill call lays
// them out again): after any call that writes weights into the pool, moves
// them between buffers or registers another host pool.  Ordered on `st`.
cudaError_t forget_wscales(moe_layer* L, cudaStream_t st) {
  if (!L->wtag) return cudaSuccess;
  const size_t n = prefill_wtag_ints(L->g) / 2;
  cudaError_t e = cudaMemsetAsync(L->wtag, 0xff, n * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(L->wtag + n, 0, n * 4, st);
  return e;
}

// The pool buffer LRU slot `slot` lives in, read once the device is idle (a
// step's LRU kernel may remap slots).
int slot_buffer(moe_layer* L, int slot, int* b) {
  MOE_CUDA(L, cudaDeviceSynchronize());
  MOE_CUDA(L, cudaMemcpy(b, L->buf + slot, 4, cudaMemcpyDeviceToHost));
  if (!buf_ok(L->g, *b)) return fail(L, MOE_ERR_STATE, "slot %d maps to buffer %d", slot, *b);
  return MOE_OK;
}

int n_ent_cap(const moe_layer* L, int N) {
  long long routed = (long long)N * L->g.k;
  return (int)std::min<long long>(std::min(L->g.S, L->g.E), routed);
}

}  // namespace

extern "C" {

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_NOT_INSTALLED: return "expert has no host source";
    case MOE_ERR_OOM: return "out of memory";
    case MOE_ERR_FILL: return "cache fill failed";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_STATE: return "invalid state";
    case MOE_ERR_UNSUPPORTED: return "unsupported by this build";
    default: return "unknown status";
  }
}

const char* moe_last_error(moe_layer_t L) { return L ? L->err.c_str() : "null layer"; }

int moe_expert_layout_for(const moe_layer_desc* desc, moe_expert_layout* out) {
  std::string why;
  if (!out) return MOE_ERR_ARG;
  int rc = check_desc(desc, &why, desc ? desc->E : 1);
  if (rc) return rc;
  fill_layout(desc, out);
  return MOE_OK;
}

// Layer `index` of `n_layers` sharing one pool and one slot table (a lone
// layer: index 0 of 1).  base: the stack's layer 0, whose pool, table,
// workspaces, plans, fill stream and events the others use; null for layer 0.
int create_layer(const moe_layer_desc* desc, moe_layer* base, int index, int n_layers, moe_layer** out) {
  *out = nullptr;
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OOM;
  L->desc = *desc;
  fill_layout(desc, &L->lay);
  L->g = make_geo(desc, &L->lay);
  if (!gemv_shape_ok(L->g)) {
    delete L;
    return MOE_ERR_UNSUPPORTED;
  }
  if (cudaGetDevice(&L->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device) != cudaSuccess) {
    cudaGetLastError();
    delete L;
    return MOE_ERR_CUDA;
  }
  const size_t Nm = desc->max_tokens;
  // spare buffers: one per miss a step can have beyond the first wave of n_slots
  L->g.X = (int)std::max<long long>(0, std::min<long long>(L->g.E, (long long)Nm * L->g.k) - L->g.S);
  // pool buffers: the S slots' (slot s starts in buffer s), layer 0's shared
  // expert (S), the X spares, then the other layers' shared experts
  L->g.key0 = index * L->g.E;
  L->g.keys = n_layers * L->g.E;
  L->g.shb = index == 0 ? L->g.S : L->g.S + L->g.X + index;
  L->g.nbuf = L->g.S + 1 + L->g.X + (n_layers - 1);
  L->index = index;
  const Geo& g = L->g;
  const size_t rows = Nm * g.k + (g.has_shared ? Nm : 0);
  int rc = MOE_OK;
  const bool prefill_ok = prefill_shape_ok(g);
  const size_t prows = Nm * g.k + Nm + 128;   // permuted rows (+ shared) + one tile of padding
#define MOE_ALLOC(ptr, bytes) \
  if (rc == MOE_OK) rc = dalloc(L, &L->ptr, (bytes))
  // this layer's own: router, step record, fused-step words, counters
  MOE_ALLOC(Wr, (size_t)g.E * g.d * 4);
  MOE_ALLOC(Wr_hl, (size_t)g.E * g.d * 6);
  MOE_ALLOC(bias, (size_t)g.E * 4);
  MOE_ALLOC(rec, rec_dev_bytes(g.E));
  MOE_ALLOC(gbar, 24);
  MOE_ALLOC(ready, 8);
  MOE_ALLOC(stats, 64);
  if (base) {
    // the pool, table and workspaces of the stack's layer 0
    L->owner = false;
    L->mir = base->mir;
    L->slots = base->slots;
    L->slot_of = base->slot_of;
    L->expert_of = base->expert_of;
    L->stamp = base->stamp;
    L->buf = base->buf;
    L->clock = base->clock;
    L->logits = base->logits;
    L->logits2 = base->logits2;
    L->idx = base->idx;
    L->gates = base->gates;
    L->xexp = base->xexp;
    L->counts = base->counts;
    L->offsets = base->offsets;
    L->row_of = base->row_of;
    L->tok_of = base->tok_of;
    L->perm_scratch = base->perm_scratch;
    L->h = base->h;
    L->hmax = base->hmax;
    L->O = base->O;
    L->x_stage = base->x_stage;
    L->y_stage = base->y_stage;
    L->list_cap = base->list_cap;
    L->list_dev = base->list_dev;
    L->rcounter = base->rcounter;
    L->step_trace = base->step_trace;
    L->xq_codes = base->xq_codes;
    L->xq_scales = base->xq_scales;
    L->hq_codes = base->hq_codes;
    L->hq_scales = base->hq_scales;
    L->pbase = base->pbase;
    L->wsf = base->wsf;
    L->wtag = base->wtag;
    L->tiles = base->tiles;
    L->n_tiles = base->n_tiles;
    L->gplan = base->gplan;
    L->plan = base->plan;
    L->fill = base->fill;
    for (int i = 0; i < kMissChunks; ++i) L->ev_chunk[i] = base->ev_chunk[i];
    L->ev_route = base->ev_route;
    L->ev_fill = base->ev_fill;
  }
  if (rc == MOE_OK && !base) {
  // buffers of the n_slots LRU slots, the shared experts (resident, not LRU), the spares
  MOE_ALLOC(slots, (size_t)g.nbuf * g.ebytes);
  MOE_ALLOC(slot_of, (size_t)g.keys * 4);
  MOE_ALLOC(expert_of, (size_t)g.S * 4);
  MOE_ALLOC(stamp, (size_t)g.S * 8);
  MOE_ALLOC(buf, (size_t)(g.S + g.X) * 4);
  MOE_ALLOC(clock, 8);
  MOE_ALLOC(logits, Nm * g.E * 4);
  MOE_ALLOC(logits2, Nm > 64 ? Nm * g.E * 4 : 16);   // the second K half of the large-batch router
  MOE_ALLOC(idx, Nm * g.k * 4);
  MOE_ALLOC(gates, Nm * g.k * 4);
  MOE_ALLOC(xexp, Nm * 4);
  MOE_ALLOC(counts, (size_t)g.E * 4);
  MOE_ALLOC(offsets, (size_t)(g.E + 1) * 4);
  MOE_ALLOC(row_of, Nm * g.k * 4);
  MOE_ALLOC(tok_of, Nm * g.k * 4);
  MOE_ALLOC(perm_scratch, permute_scratch_bytes(g, (int)Nm));
  MOE_ALLOC(h, rows * g.f * 8);   // decode: scaled W_g x and W_u x per row
  MOE_ALLOC(hmax, rows * (g.f / 64) * 8);
  MOE_ALLOC(O, rows * g.d * 4);
  MOE_ALLOC(x_stage, Nm * g.d * 2);
  MOE_ALLOC(y_stage, Nm * g.d * 2);
  L->list_cap = (int)std::max<size_t>(Nm * g.k, (size_t)g.E);
  MOE_ALLOC(list_dev, (size_t)L->list_cap * 4);
  MOE_ALLOC(rcounter, kRouterCounterBytes);
  MOE_ALLOC(step_trace, (size_t)std::max(L->num_sms, 1) * kStepMarks * 8);
  if (prefill_ok) {
    // prefill activations in their format (the weights' own, or MXFP8 for
    // W4A8): codes, then block scales
    MOE_ALLOC(xq_codes, prows * g.d * fmt_code_bits(g.afmt) / 8);
    MOE_ALLOC(xq_scales, prefill_act_scale_bytes(g, (int)Nm, g.d));
    MOE_ALLOC(hq_codes, prows * g.f * fmt_code_bits(g.afmt) / 8);
    MOE_ALLOC(hq_scales, prefill_act_scale_bytes(g, (int)Nm, g.f));
    MOE_ALLOC(pbase, (size_t)(g.E + 2) * 4);
    MOE_ALLOC(wsf, prefill_wscale_bytes(g));
    MOE_ALLOC(wtag, prefill_wtag_ints(g) * 4);
    MOE_ALLOC(tiles, prefill_tile_bytes(g, (int)Nm));
    MOE_ALLOC(n_tiles, 16);
  }
  }
#undef MOE_ALLOC
  if (rc == MOE_OK) L->shared_w = L->slots + (size_t)g.shb * g.ebytes;
  if (rc == MOE_OK) {
    void* eh = nullptr;
    rc = halloc(L, &eh, 16);
    L->err_host = static_cast<int*>(eh);
    if (rc == MOE_OK && cudaHostGetDevicePointer(reinterpret_cast<void**>(&L->err_dev), L->err_host, 0) != cudaSuccess) {
      cudaGetLastError();
      rc = MOE_ERR_CUDA;
    }
    if (rc == MOE_OK) *L->err_host = 0;
  }
  if (rc == MOE_OK && !base) {
    L->gplan = gemv_plan_create(g, L->slots);
    if (!gemv_plan_ready(L->gplan)) rc = MOE_ERR_CUDA;   // tensor-map encoding failed
  }
  if (rc == MOE_OK && prefill_ok && !base) {
    L->plan = prefill_plan_create(g, L->slots, L->xq_codes, prows, L->hq_codes);
    if (!prefill_plan_ready(L->plan)) {
      prefill_plan_destroy(L->plan);
      L->plan = nullptr;   // prefill regime unavailable (tensor-map encoding failed)
    }
  }
  if (rc == MOE_OK) rc = halloc(L, &L->pinned_rec, rec_bytes(g.E));
  if (rc == MOE_OK) {
    L->rec_host = static_cast<StepRecord*>(L->pinned_rec);
    std::memset(L->pinned_rec, 0, rec_bytes(g.E));
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, L->pinned_rec, 0) != cudaSuccess) {
      cudaGetLastError();
      rc = MOE_ERR_CUDA;
    }
    L->rec_host_dev = static_cast<StepRecord*>(dp);
  }
  if (rc == MOE_OK && !base) {
    bool sok = true;
    // the fill stream has the highest priority: a fill kernel's CTAs are
    // dispatched before expert-GEMV CTAs waiting for SMs
    int prio_lo = 0, prio_hi = 0;
    sok = sok && cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi) == cudaSuccess;
    sok = sok && cudaStreamCreateWithPriority(&L->fill, cudaStreamNonBlocking, prio_hi) == cudaSuccess;
    for (int i = 0; i < kMissChunks; ++i)
      sok = sok && cudaEventCreateWithFlags(&L->ev_chunk[i], cudaEventDisableTiming) == cudaSuccess;
    if (!sok ||
        cudaEventCreateWithFlags(&L->ev_route, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&L->ev_fill, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      rc = MOE_ERR_CUDA;
    }
  }
  if (rc == MOE_OK) {
    // zero bias, empty record and counters; the owner: empty cache
    bool ok = cudaMemset(L->bias, 0, (size_t)g.E * 4) == cudaSuccess &&
              cudaMemset(L->rec, 0, rec_dev_bytes(g.E)) == cudaSuccess &&
              cudaMemset(L->gbar, 0, 24) == cudaSuccess &&
              cudaMemset(L->ready, 0, 8) == cudaSuccess &&
              cudaMemset(L->stats, 0, 64) == cudaSuccess;
    if (!base) {
      ok = ok && cudaMemset(L->slot_of, 0xff, (size_t)g.keys * 4) == cudaSuccess &&
           cudaMemset(L->expert_of, 0xff, (size_t)g.S * 4) == cudaSuccess &&
           cudaMemset(L->stamp, 0, (size_t)g.S * 8) == cudaSuccess &&
           cudaMemset(L->clock, 0, 8) == cudaSuccess &&
           cudaMemset(L->rcounter, 0, kRouterCounterBytes) == cudaSuccess &&
           forget_wscales(L, nullptr) == cudaSuccess;
      // slot s in buffer s; the spares after the shared expert's buffer S
      std::vector<int> b0(g.S + g.X);
      for (int s = 0; s < g.S; ++s) b0[s] = s;
      for (int j = 0; j < g.X; ++j) b0[g.S + j] = g.S + 1 + j;
      ok = ok && (b0.empty() || cudaMemcpy(L->buf, b0.data(), b0.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess);
    }
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      rc = MOE_ERR_CUDA;
    }
  }
  if (rc != MOE_OK) {
    release(L);
    delete L;
    return rc;
  }
  if (!base) {
    L->mirror_own.assign(g.S, -1);
    L->mir = &L->mirror_own;
  }
  *out = L;
  return MOE_OK;
}

int moe_layer_create(const moe_layer_desc* desc, moe_layer_t* out) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  std::string why;
  const int rc = check_desc(desc, &why, desc ? desc->E : 1);
  if (rc) return rc;
  return create_layer(desc, nullptr, 0, 1, out);
}

int moe_layer_destroy(moe_layer_t L) {
  if (!L) return MOE_ERR_ARG;
  if (L->stack) return fail(L, MOE_ERR_STATE, "layer %d belongs to a stack: destroy the stack", L->index);
  cudaDeviceSynchronize();
  release(L);
  delete L;
  return MOE_OK;
}

int moe_set_router(moe_layer_t L, const float* W_r, const float* bias) {
  if (!L) return MOE_ERR_ARG;
  if (!W_r) return fail(L, MOE_ERR_ARG, "W_r is NULL");
  if (L->g.has_bias && !bias) return fail(L, MOE_ERR_ARG, "layer has a bias but bias is NULL");
  MOE_CUDA(L, cudaMemcpy(L->Wr, W_r, (size_t)L->g.E * L->g.d * 4, cudaMemcpyDefault));
  MOE_CUDA(L, launch_router_split(L->g, L->Wr, L->Wr_hl, nullptr));
  MOE_CUDA(L, cudaDeviceSynchronize());
  if (L->g.has_bias) MOE_CUDA(L, cudaMemcpy(L->bias, bias, (size_t)L->g.E * 4, cudaMemcpyDefault));
  L->router_set = true;
  return MOE_OK;
}

int moe_register_host_experts(moe_layer_t L, const void* pool, size_t bytes) {
  if (!L) return MOE_ERR_ARG;
  if (!pool) return fail(L, MOE_ERR_ARG, "pool is NULL");
  if (bytes < (size_t)L->g.E * L->g.ebytes)
    return fail(L, MOE_ERR_ARG, "pool holds %zu bytes, need E * layout.bytes = %zu", bytes,
                (size_t)L->g.E * L->g.ebytes);
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, pool) != cudaSuccess || a.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(L, MOE_ERR_ARG, "pool must be pinned (page-locked) host memory");
  }
  MOE_CUDA(L, forget_wscales(L, nullptr));
  MOE_CUDA(L, cudaDeviceSynchronize());
  L->host_pool = static_cast<const uint8_t*>(pool);
  L->host_pool_bytes = bytes;
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, const_cast<void*>(pool), 0) == cudaSuccess) {
    L->pool_dev = static_cast<const uint8_t*>(dp);
  } else {
    cudaGetLastError();
    L->pool_dev = nullptr;   // device-driven fills unavailable for this pool
  }
  // the automatic choice by default; the copy engine when the device cannot
  // address the pool
  if (!L->pool_dev) L->fill_mode = MOE_FILL_MEMCPY;
  else if (!L->fill_mode_chosen) L->fill_mode = MOE_FILL_AUTO;
  return MOE_OK;
}

int moe_set_shared_expert(moe_layer_t L, const void* weights) {
  if (!L) return MOE_ERR_ARG;
  if (!L->g.has_shared) return fail(L, MOE_ERR_STATE, "layer has no shared expert");
  if (!weights) return fail(L, MOE_ERR_ARG, "weights is NULL");
  MOE_CUDA(L, cudaMemcpy(L->shared_w, weights, L->g.ebytes, cudaMemcpyDefault));
  MOE_CUDA(L, forget_wscales(L, nullptr));
  MOE_CUDA(L, cudaDeviceSynchronize());
  L->shared_set = true;
  return MOE_OK;
}

int moe_cache_install(moe_layer_t L, int expert, int slot, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (expert < 0 || expert >= L->g.E) return fail(L, MOE_ERR_ARG, "expert %d out of range", expert);
  if (slot < 0 || slot >= L->g.S) return fail(L, MOE_ERR_ARG, "slot %d out of range", slot);
  if (!L->host_pool) return fail(L, MOE_ERR_NOT_INSTALLED, "no host expert pool registered");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int b = -1;
  int rc = slot_buffer(L, slot, &b);
  if (rc) return rc;
  if (L->inject_fill) {
    L->inject_fill = false;
    return fail(L, MOE_ERR_FILL, "fill of expert %d could not be issued (injected by the test hook); the "
                "table is unchanged", expert);
  }
  MOE_CUDA(L, cudaMemcpyAsync(L->slots + (size_t)b * L->g.ebytes,
                              L->host_pool + (size_t)expert * L->g.ebytes, L->g.ebytes,
                              cudaMemcpyHostToDevice, st));
  MOE_CUDA(L, forget_wscales(L, st));
  MOE_CUDA(L, launch_lru_install(L->g, expert, slot, L->slot_of, L->expert_of, L->stamp, L->clock, st));
  const int key = L->g.key0 + expert;
  for (int s = 0; s < L->g.S; ++s)
    if ((*L->mir)[s] == key) (*L->mir)[s] = -1;
  (*L->mir)[slot] = key;
  return MOE_OK;
}

int moe_lru_get_state(moe_layer_t L, int* expert_of_slot, uint64_t* stamp, uint64_t* clock) {
  if (!L) return MOE_ERR_ARG;
  MOE_CUDA(L, cudaDeviceSynchronize());
  if (expert_of_slot)
    MOE_CUDA(L, cudaMemcpy(expert_of_slot, L->expert_of, (size_t)L->g.S * 4, cudaMemcpyDeviceToHost));
  if (stamp) MOE_CUDA(L, cudaMemcpy(stamp, L->stamp, (size_t)L->g.S * 8, cudaMemcpyDeviceToHost));
  if (clock) MOE_CUDA(L, cudaMemcpy(clock, L->clock, 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

int moe_cache_resize(moe_layer_t L, int n_slots, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (L->stack) return fail(L, MOE_ERR_UNSUPPORTED, "a stack's shared pool is not resized through one layer");
  const Geo g0 = L->g;
  if (n_slots < 1 || n_slots > g0.E) return fail(L, MOE_ERR_ARG, "n_slots must be in [1, E = %d]", g0.E);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a step boundary: nothing of an earlier call may still read the pool
  MOE_CUDA(L, cudaDeviceSynchronize());
  const int S0 = g0.S, S1 = n_slots;
  std::vector<int> eo(S0), bufm(S0 + g0.X);
  std::vector<unsigned long long> stp(S0);
  MOE_CUDA(L, cudaMemcpy(eo.data(), L->expert_of, (size_t)S0 * 4, cudaMemcpyDeviceToHost));
  MOE_CUDA(L, cudaMemcpy(stp.data(), L->stamp, (size_t)S0 * 8, cudaMemcpyDeviceToHost));
  if (!bufm.empty()) MOE_CUDA(L, cudaMemcpy(bufm.data(), L->buf, bufm.size() * 4, cudaMemcpyDeviceToHost));
  // the S1 most recently used experts stay, in the order of their old slots
  std::vector<int> occ;
  for (int s = 0; s < S0; ++s)
    if (eo[s] >= 0 && eo[s] < g0.E) occ.push_back(s);
  std::vector<int> by_stamp = occ;
  std::sort(by_stamp.begin(), by_stamp.end(), [&](int a, int b) { return stp[a] > stp[b]; });
  if ((int)by_stamp.size() > S1) by_stamp.resize(S1);
  std::vector<int> keep = by_stamp;
  std::sort(keep.begin(), keep.end());
  for (int s : keep)
    if (!buf_ok(g0, bufm[s])) return fail(L, MOE_ERR_STATE, "slot %d maps to buffer %d", s, bufm[s]);
  // the new geometry and its buffers: slot i in buffer i, the shared expert
  // in buffer S1, the spares after it
  Geo g1 = g0;
  g1.S = S1;
  g1.X = (int)std::max<long long>(0, std::min<long long>(g1.E, (long long)L->desc.max_tokens * g1.k) - S1);
  g1.shb = S1;
  g1.nbuf = S1 + 1 + g1.X;
  const size_t nb1 = (size_t)g1.nbuf;
  uint8_t* pool = nullptr;
  int *eo_d = nullptr, *buf_d = nullptr;
  unsigned long long* st_d = nullptr;
  auto undo = [&]() {
    if (pool) cudaFree(pool);
    if (eo_d) cudaFree(eo_d);
    if (buf_d) cudaFree(buf_d);
    if (st_d) cudaFree(st_d);
    cudaGetLastError();
  };
  if (alloc_fault_due() || cudaMalloc(&pool, nb1 * g1.ebytes) != cudaSuccess ||
      cudaMalloc(&eo_d, (size_t)S1 * 4) != cudaSuccess || cudaMalloc(&st_d, (size_t)S1 * 8) != cudaSuccess ||
      cudaMalloc(&buf_d, std::max<size_t>(16, (size_t)(S1 + g1.X) * 4)) != cudaSuccess) {
    undo();
    return fail(L, MOE_ERR_OOM, "resizing the expert cache to %d slots: out of device memory (cache unchanged)", S1);
  }
  // kept experts and the shared expert move buffer to buffer on the device
  cudaError_t ce = cudaSuccess;
  for (size_t i = 0; i < keep.size() && ce == cudaSuccess; ++i)
    ce = cudaMemcpyAsync(pool + i * g1.ebytes, L->slots + (size_t)bufm[keep[i]] * g0.ebytes, g0.ebytes,
                         cudaMemcpyDeviceToDevice, st);
  if (ce == cudaSuccess && g1.has_shared)
    ce = cudaMemcpyAsync(pool + (size_t)S1 * g1.ebytes, L->slots + (size_t)S0 * g0.ebytes, g0.ebytes,
                         cudaMemcpyDeviceToDevice, st);
  std::vector<int> eo1(S1, -1), buf1(S1 + g1.X), so1(g1.E, -1);
  std::vector<unsigned long long> st1(S1, 0);
  for (size_t i = 0; i < keep.size(); ++i) {
    eo1[i] = eo[keep[i]];
    st1[i] = stp[keep[i]];
    so1[eo1[i]] = (int)i;
  }
  for (int s = 0; s < S1; ++s) buf1[s] = s;
  for (int j = 0; j < g1.X; ++j) buf1[S1 + j] = S1 + 1 + j;
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(eo_d, eo1.data(), (size_t)S1 * 4, cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(st_d, st1.data(), (size_t)S1 * 8, cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess && !buf1.empty())
    ce = cudaMemcpyAsync(buf_d, buf1.data(), buf1.size() * 4, cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(L->slot_of, so1.data(), (size_t)g1.E * 4, cudaMemcpyHostToDevice, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  GemvPlan* gp = ce == cudaSuccess ? gemv_plan_create(g1, pool) : nullptr;
  if (ce != cudaSuccess || !gemv_plan_ready(gp)) {
    if (gp) gemv_plan_destroy(gp);
    undo();
    // slot_of may already hold the new table: put the old one back
    std::vector<int> so0(g0.E, -1);
    for (int s = 0; s < S0; ++s)
      if (eo[s] >= 0 && eo[s] < g0.E) so0[eo[s]] = s;
    cudaMemcpy(L->slot_of, so0.data(), (size_t)g0.E * 4, cudaMemcpyHostToDevice);
    return ce != cudaSuccess ? cuda_fail(L, ce, "resizing the expert cache") :
                               fail(L, MOE_ERR_CUDA, "tensor maps of the resized pool could not be encoded");
  }
  // swap in the new pool and table
  auto swap_alloc = [&](void* old_p, void* new_p) {
    for (auto& p : L->dev_allocs)
      if (p == old_p) {
        cudaFree(old_p);
        p = new_p;
        return;
      }
  };
  swap_alloc(L->slots, pool);
  swap_alloc(L->expert_of, eo_d);
  swap_alloc(L->stamp, st_d);
  swap_alloc(L->buf, buf_d);
  L->slots = pool;
  L->shared_w = pool + (size_t)S1 * g1.ebytes;
  L->expert_of = eo_d;
  L->stamp = st_d;
  L->buf = buf_d;
  gemv_plan_destroy(L->gplan);
  L->gplan = gp;
  L->g = g1;
  L->desc.n_slots = S1;
  if (L->plan) {
    prefill_plan_destroy(L->plan);
    const size_t Nm = L->desc.max_tokens;
    L->plan = prefill_plan_create(g1, L->slots, L->xq_codes, Nm * g1.k + Nm + 128, L->hq_codes);
    if (!prefill_plan_ready(L->plan)) {
      prefill_plan_destroy(L->plan);
      L->plan = nullptr;
    }
  }
  *L->mir = eo1;
  MOE_CUDA(L, forget_wscales(L, nullptr));
  MOE_CUDA(L, cudaDeviceSynchronize());
  return MOE_OK;
}

int moe_lru_set_state(moe_layer_t L, const int* expert_of_slot, const uint64_t* stamp, uint64_t clock) {
  if (!L) return MOE_ERR_ARG;
  if (!expert_of_slot || !stamp) return fail(L, MOE_ERR_ARG, "NULL state array");
  const int E = L->g.keys, S = L->g.S;   // a stack's table holds keys l E + e
  std::vector<int> slot_of(E, -1);
  for (int s = 0; s < S; ++s) {
    const int e = expert_of_slot[s];
    if (e < -1 || e >= E) return fail(L, MOE_ERR_ARG, "expert %d in slot %d out of range", e, s);
    if (e >= 0) {
      if (slot_of[e] >= 0) return fail(L, MOE_ERR_ARG, "expert %d in two slots", e);
      if (stamp[s] > clock) return fail(L, MOE_ERR_ARG, "stamp of slot %d exceeds clock", s);
      slot_of[e] = s;
    }
  }
  MOE_CUDA(L, cudaDeviceSynchronize());
  MOE_CUDA(L, cudaMemcpy(L->expert_of, expert_of_slot, (size_t)S * 4, cudaMemcpyHostToDevice));
  MOE_CUDA(L, cudaMemcpy(L->slot_of, slot_of.data(), (size_t)E * 4, cudaMemcpyHostToDevice));
  MOE_CUDA(L, cudaMemcpy(L->stamp, stamp, (size_t)S * 8, cudaMemcpyHostToDevice));
  MOE_CUDA(L, cudaMemcpy(L->clock, &clock, 8, cudaMemcpyHostToDevice));
  MOE_CUDA(L, forget_wscales(L, nullptr));
  MOE_CUDA(L, cudaDeviceSynchronize());
  L->mir->assign(expert_of_slot, expert_of_slot + S);
  return MOE_OK;
}

int moe_lru_touch(moe_layer_t L, const int* experts, int n, int* slot_of_out, int* miss_experts_out,
                  int* miss_slots_out, int* n_miss_out, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (n < 0 || n > L->list_cap) return fail(L, MOE_ERR_ARG, "n must be in [0, %d]", L->list_cap);
  if (n > 0 && !experts) return fail(L, MOE_ERR_ARG, "experts is NULL");
  for (int i = 0; i < n; ++i)
    if (experts[i] < 0 || experts[i] >= L->g.E) return fail(L, MOE_ERR_ARG, "expert %d out of range", experts[i]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Geo& g = L->g;
  if (n > 0) MOE_CUDA(L, cudaMemcpyAsync(L->list_dev, experts, (size_t)n * 4, cudaMemcpyHostToDevice, st));
  MOE_CUDA(L, launch_counts_from_list(g, L->list_dev, n, L->counts, st));
  MOE_CUDA(L, launch_lru_step(g, L->counts, nullptr, L->slot_of, L->expert_of, L->stamp, L->clock, L->buf,
                              L->rec, nullptr, nullptr, 0, st));
  MOE_CUDA(L, cudaMemcpyAsync(L->rec_host, L->rec, rec_bytes(g.E), cudaMemcpyDeviceToHost, st));
  MOE_CUDA(L, cudaStreamSynchronize(st));
  const StepRecord* r = L->rec_host;
  const int* ae = rec_expert(const_cast<StepRecord*>(r));
  const int* as = rec_slot(const_cast<StepRecord*>(r), g.E);
  const int* ab = rec_buf(const_cast<StepRecord*>(r), g.E);
  if (r->U < 0 || r->U > g.E || r->n_hit < 0 || r->n_hit > r->U)
    return fail(L, MOE_ERR_STATE, "step record is inconsistent");
  for (int i = 0; i < r->U; ++i)
    if (ae[i] < 0 || ae[i] >= g.E || as[i] < 0 || as[i] >= g.S || !buf_ok(g, ab[i]))
      return fail(L, MOE_ERR_STATE, "step record entry %d is out of range", i);
  if (L->host_pool) {
    // every miss into the buffer the step gave it (a later-wave miss's spare
    // became its slot's buffer at the end of the step)
    for (int i = r->n_hit; i < r->U; ++i) {
      cudaError_t ce = cudaSuccess;
      if (L->inject_fill) {
        L->inject_fill = false;
        ce = cudaErrorInvalidValue;
      } else {
        ce = cudaMemcpyAsync(L->slots + (size_t)ab[i] * g.ebytes, L->host_pool + (size_t)ae[i] * g.ebytes,
                             g.ebytes, cudaMemcpyHostToDevice, st);
      }
      if (ce != cudaSuccess) {
        cudaGetLastError();
        mirror_apply(L, r);
        mirror_drop_misses(L, r);
        MOE_CUDA(L, launch_lru_drop_misses(g, L->rec, L->slot_of, L->expert_of, st));
        MOE_CUDA(L, cudaStreamSynchronize(st));
        return fail(L, MOE_ERR_FILL, "fill of expert %d could not be issued (%s); the %d misses were dropped "
                    "from the cache", ae[i], cudaGetErrorString(ce), r->U - r->n_hit);
      }
    }
    MOE_CUDA(L, cudaStreamSynchronize(st));
  }
  mirror_apply(L, r);
  if (slot_of_out) {
    std::vector<int> where(g.E, -1);
    for (int i = 0; i < r->U; ++i) where[ae[i]] = as[i];
    for (int i = 0; i < n; ++i) slot_of_out[i] = where[experts[i]];
  }
  for (int i = r->n_hit, m = 0; i < r->U; ++i, ++m) {
    if (miss_experts_out) miss_experts_out[m] = ae[i];
    if (miss_slots_out) miss_slots_out[m] = as[i];
  }
  if (n_miss_out) *n_miss_out = r->n_miss;
  return MOE_OK;
}

// Wait for the LRU kernel's host copy of step `seq` (bounded).  Fails on an
// error of the routing launches or when the record is not there well after
// they finished.
static int poll_record(moe_layer_t L, unsigned long long seq) {
  using clk = std::chrono::steady_clock;
  const clk::time_point t0 = clk::now();
  clk::time_point done_at{};
  bool done = false;
  for (unsigned it = 1;; ++it) {
    if (__atomic_load_n(&L->rec_host->seq, __ATOMIC_ACQUIRE) == seq) return MOE_OK;
    if ((it & 255) == 0) {
      const cudaError_t q = cudaEventQuery(L->ev_route);
      if (q != cudaSuccess && q != cudaErrorNotReady) return cuda_fail(L, q, "routing");
      if (q == cudaSuccess && !done) {
        done = true;
        done_at = clk::now();
      }
      if (done && clk::now() - done_at > std::chrono::milliseconds(200))
        return fail(L, MOE_ERR_STATE, "the routing finished but step record %llu never reached the host", seq);
      if (clk::now() - t0 > std::chrono::seconds(30))
        return fail(L, MOE_ERR_TIMEOUT, "step record %llu did not arrive within 30 s", seq);
    }
  }
}

int moe_forward(moe_layer_t L, const void* x, int N, void* y, void* stream, int regime,
                moe_forward_info* info) {
  if (!L) return MOE_ERR_ARG;
  const Geo& g = L->g;
  if (info) {
    std::memset(info, 0, sizeof *info);
    info->n_tokens = N;
  }
  if (N < 0 || N > L->desc.max_tokens)
    return fail(L, MOE_ERR_ARG, "N = %d outside [0, max_tokens = %d]", N, L->desc.max_tokens);
  if (N == 0) return MOE_OK;
  if (!x || !y) return fail(L, MOE_ERR_ARG, "x or y is NULL");
  if (!L->router_set) return fail(L, MOE_ERR_STATE, "router weights not set");
  if (g.has_shared && !L->shared_set) return fail(L, MOE_ERR_STATE, "shared expert not set");
  if (regime != MOE_REGIME_AUTO && regime != MOE_REGIME_DECODE && regime != MOE_REGIME_PREFILL)
    return fail(L, MOE_ERR_ARG, "unknown regime %d", regime);
  if (regime == MOE_REGIME_PREFILL && !L->plan)
    return fail(L, MOE_ERR_UNSUPPORTED, "the prefill regime needs d_model and d_ff multiples of 256");
  const bool prefill = regime == MOE_REGIME_PREFILL || (regime == MOE_REGIME_AUTO && N > 64 && L->plan);
  if (*L->err_host) {
    *L->err_host = 0;
    // a fused step that gave up may have left its barrier counter short:
    // start it again from zero, after every launch already queued
    cudaStream_t st0 = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(L->gbar, 0, 24, st0) != cudaSuccess) cudaGetLastError();
    L->gbar_base = 0;
    return fail(L, MOE_ERR_TIMEOUT, "a wait inside an earlier step's kernel timed out; its output is invalid");
  }
  // assume_resident: a stack prefetched every expert of this layer just before
  const bool resident = L->assume_resident || all_resident(L);
  if (!resident && !L->host_pool)
    return fail(L, MOE_ERR_NOT_INSTALLED, "not every expert is resident and no host pool is registered");
  bool x_dev = false, y_dev = false;
  const void* x_map = nullptr;
  const void* y_map = nullptr;
  if (pointer_kind(x, &x_dev, L->device, &x_map) || pointer_kind(y, &y_dev, L->device, &y_map))
    return fail(L, MOE_ERR_ARG, "x or y is device memory of another device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xbytes = (size_t)N * g.d * 2;
  const __nv_bfloat16* xd = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* yd = static_cast<__nv_bfloat16*>(y);
  // decode-sized batches in pinned host buffers go through unified
  // addressing: a copy kernel stages x (no DMA set-up on the critical path)
  // and the combine writes y straight into the host buffer
  const bool small = !prefill && xbytes <= kDirectHostBytes;
  const bool x_direct = !x_dev && small && x_map && reinterpret_cast<uintptr_t>(x_map) % 16 == 0;
  const bool y_direct = !y_dev && small && y_map && reinterpret_cast<uintptr_t>(y_map) % 16 == 0;
  if (x_direct) {
    MOE_CUDA(L, launch_copy16(L->x_stage, x_map, xbytes, st));
    xd = L->x_stage;
  } else if (!x_dev) {
    MOE_CUDA(L, cudaMemcpyAsync(L->x_stage, x, xbytes, cudaMemcpyHostToDevice, st));
    xd = L->x_stage;
  } else if (reinterpret_cast<uintptr_t>(x) % 16) {
    // the kernels read x in 16-byte vectors
    MOE_CUDA(L, cudaMemcpyAsync(L->x_stage, x, xbytes, cudaMemcpyDeviceToDevice, st));
    xd = L->x_stage;
  }
  if (y_direct) yd = static_cast<__nv_bfloat16*>(const_cast<void*>(y_map));
  else if (!y_dev) yd = L->y_stage;

  L->launches = x_direct ? 1 : 0;
  {
    // the whole decode step as one launch (step.cu), when every expert is
    // resident or misses are filled by the expert FFN itself
    int fm = L->fill_mode;
    if (fm == MOE_FILL_AUTO) fm = std::min(g.E, N * g.k) <= g.S ? MOE_FILL_FUSED : MOE_FILL_KERNEL;
    const bool fused_fill = !resident && fm == MOE_FILL_FUSED && L->pool_dev;
    StepPlan plan{};
    // AUTO takes the fused launch for steps of at most kStepAutoPairs (token,
    // expert) pairs (measured on GB300): with every expert resident it is the
    // faster path (batch 1 and 4 of the 35B-A3B-shaped layer, batch 1 of the
    // 284B-A13B-shaped one; larger steps keep pace on the chain); with misses,
    // a lone layer is faster on the chain with fused fills (58.5 vs 64.3 us at
    // batch 1, 121 vs 131 us at batch 4, 35B-A3B layer, 47 slots, miss rate
    // 0.16-0.2), a stack's layers -- with twice the miss rate on the shared
    // pool -- in the fused launch (76 vs 111 us per layer step at batch 1, 150
    // vs 177 at batch 4: the chain's two expert-FFN launches each pay the host
    // link's latency for the misses)
    const bool want = !prefill && L->decode_path != MOE_DECODE_CHAIN && !L->step_failed && L->num_sms >= 2 &&
                      (L->decode_path == MOE_DECODE_STEP ||
                       (N * g.k <= kStepAutoPairs && (resident || L->stack != nullptr)));
    const bool can = want && (resident || fused_fill) && step_plan(g, N, &plan);
    if (L->decode_path == MOE_DECODE_STEP && !can)
      return fail(L, MOE_ERR_UNSUPPORTED, "this step cannot run as one fused launch (N = %d, fill mode %d)", N, fm);
    if (can) {
      GemvArgs a{};
      a.slots = L->slots;
      a.shared_w = L->shared_w;
      a.rec = L->rec;
      a.N = N;
      a.mode = kRangeAll;
      a.host_pool = fused_fill ? L->pool_dev : nullptr;
      a.with_shared = g.has_shared;
      a.err = L->err_dev;
      a.hmax = L->hmax;
      a.wait_cycles = L->inject_wait;
      L->inject_wait = 0;
      StepArgs sa{};
      sa.x = xd;
      sa.Wr = L->Wr;
      sa.bias = g.has_bias ? L->bias : nullptr;
      sa.logits = L->logits;
      sa.idx = L->idx;
      sa.gates = L->gates;
      sa.counts = L->counts;
      sa.offsets = L->offsets;
      sa.row_of = L->row_of;
      sa.tok_of = L->tok_of;
      sa.slot_of = L->slot_of;
      sa.expert_of = L->expert_of;
      sa.buf = L->buf;
      sa.stamp = L->stamp;
      sa.clock = L->clock;
      sa.rec = L->rec;
      sa.stats = L->stats;
      sa.ready = L->ready;
      sa.seq = ++L->ready_seq;
      sa.gbar = L->gbar;
      sa.gbar_base = L->gbar_base;
      sa.h = L->h;
      sa.O = L->O;
      sa.y = yd;
      sa.trace = L->prof_on ? L->step_trace : nullptr;
      if (sa.trace) L->step_trace_grid = L->num_sms;
      cudaEvent_t* ps = prof_begin(L, MOE_PROF_STEP, st);
      const cudaError_t ce = launch_step(g, L->gplan, a, sa, plan, L->num_sms, st);
      prof_end(ps, st);
      if (ce == cudaSuccess) {
        L->gbar_base += (unsigned long long)L->num_sms;
        L->launches += 1;
        if (!y_dev) {
          if (!y_direct) MOE_CUDA(L, cudaMemcpyAsync(y, yd, xbytes, cudaMemcpyDeviceToHost, st));
          MOE_CUDA(L, cudaStreamSynchronize(st));
        }
        L->last_N = N;
        L->last_prefill = false;
        if (info) {
          info->regime = MOE_REGIME_DECODE;
          info->n_distinct = info->n_hits = -1;
          info->n_misses = resident ? 0 : -1;
          info->n_waves = 1;
          info->fill_bytes = 0;
          info->host_synced = 0;
          info->n_launches = L->launches;
          info->fused_step = 1;
        }
        return MOE_OK;
      }
      // a device that cannot hold the cooperative grid: the chained launches from now on
      cudaGetLastError();
      if (L->decode_path == MOE_DECODE_STEP) return cuda_fail(L, ce, "launch_step");
      L->step_failed = true;
    }
  }
  cudaEvent_t* pe = prof_begin(L, MOE_PROF_ROUTER, st);
  MOE_CUDA(L, launch_router(g, xd, N, L->Wr, L->Wr_hl, g.has_bias ? L->bias : nullptr, L->logits, L->idx,
                            L->gates, prefill ? nullptr : L->xexp, L->rcounter, L->err_dev, L->logits2, st));
  prof_end(pe, st);
  L->launches += N <= 64 ? 1 : 2;
  // memcpy fills: the LRU kernel also writes the step record into mapped
  // pinned host memory, sequence number last, and the host polls it
  // the automatic choice: fused fills while no access of the step can need a
  // spare buffer, SM-copy fills beyond
  int fmode = L->fill_mode;
  if (fmode == MOE_FILL_AUTO) fmode = std::min(g.E, N * g.k) <= g.S ? MOE_FILL_FUSED : MOE_FILL_KERNEL;
  // SM fills need the GPU to keep most of its SMs for the expert GEMV
  if (fmode == MOE_FILL_KERNEL && L->num_sms <= 2 * kFillSms) fmode = MOE_FILL_MEMCPY;
  // fused fills (decode): one expert-FFN launch covers every access and reads
  // the misses' weights from the host pool itself, writing them on to their
  // slots, so no separate copy and no host round trip
  const bool fused = !resident && !prefill && fmode == MOE_FILL_FUSED;
  const bool host_poll = !resident && fmode != MOE_FILL_DEVICE && !fused;
  StepRecord* hrec = host_poll ? L->rec_host_dev : nullptr;
  bool tiles_built = false;   // the prefill tiles of the hits came with the routing (N > 128)
  const unsigned long long seq = host_poll ? ++L->step_seq : 0ull;
  if (N <= 128) {
    // permutation and LRU step in one CTA
    pe = prof_begin(L, MOE_PROF_PERMUTE, st);
    MOE_CUDA(L, launch_route_tail(g, L->idx, N, L->counts, L->offsets, L->row_of, L->tok_of,
                                  L->slot_of, L->expert_of, L->stamp, L->clock, L->buf, L->rec, L->stats,
                                  hrec, seq, st));
    prof_end(pe, st);
    L->launches += 1;
    if (L->ev_after_route) MOE_CUDA(L, cudaEventRecord(L->ev_after_route, st));
  } else {
    // permutation (histograms; scan + the prefill's padded blocks + LRU step
    // in one CTA; scatter of the rows)
    pe = prof_begin(L, MOE_PROF_PERMUTE, st);
    MOE_CUDA(L, launch_perm_hist(g, L->idx, N, L->perm_scratch, st));
    MOE_CUDA(L, launch_scan_lru(g, N, L->perm_scratch, L->counts, L->offsets, prefill ? L->pbase : nullptr,
                                L->slot_of, L->expert_of, L->stamp, L->clock, L->buf, L->rec, L->stats, hrec, seq,
                                prefill ? L->tiles : nullptr, L->n_tiles, st));
    tiles_built = prefill;
    MOE_CUDA(L, launch_perm_scatter(g, L->idx, N, L->offsets, L->perm_scratch, L->row_of, L->tok_of, st));
    prof_end(pe, st);
    L->launches += 3;
    if (L->ev_after_route) MOE_CUDA(L, cudaEventRecord(L->ev_after_route, st));
  }
  const bool dev_fill = !resident && fmode == MOE_FILL_DEVICE;
  if (!resident) MOE_CUDA(L, cudaEventRecord(L->ev_route, st));
  GemvArgs a{};
  a.slots = L->slots;
  a.shared_w = L->shared_w;
  a.rec = L->rec;
  a.offsets = L->offsets;
  a.tok_of = L->tok_of;
  a.N = N;
  a.mode = fused ? kRangeAll : kRangeHits;
  a.host_pool = fused ? L->pool_dev : nullptr;
  a.chunk = 0;
  a.n_chunks = 1;
  a.with_shared = g.has_shared;
  a.err = L->err_dev;
  a.hmax = L->hmax;
  a.wait_cycles = L->inject_wait;   // 0: the default limit
  L->inject_wait = 0;
  const int cap = n_ent_cap(L, N);
  const float gx = g.fmt == MOE_NVFP4 ? L->desc.act_scale_x : 1.0f;
  const float gh = g.fmt == MOE_NVFP4 ? L->desc.act_scale_h : 1.0f;
  if (prefill) {
    pe = prof_begin(L, MOE_PROF_PREFILL, st);
    // the padded blocks came with the LRU step when N > 128
    MOE_CUDA(L, launch_gather_quant(g, xd, L->idx, L->row_of, L->counts, L->offsets, N, gx, L->pbase, N > 128,
                                    L->xq_codes, L->xq_scales, st));
    prof_end(pe, st);
    L->launches += N > 128 ? 1 : 2;
  }
  // SM fills (decode): kFillSms SMs copy the misses, the expert GEMV takes
  // the others, and the hits' phase 2 is launched after the host has read the
  // record, so that its waiting CTAs cannot take the SMs the fills need
  const bool sm_fill = !resident && !prefill && fmode == MOE_FILL_KERNEL;
  const int gemv_sms = sm_fill ? L->num_sms - kFillSms : L->num_sms;
  auto gemv = [&](int n_ent, int phases) -> int {
    cudaEvent_t ev[4] = {};
    const bool room = L->prof_used + 4 <= L->prof_pool.size();
    cudaEvent_t* p1 = room && (phases & 1) ? prof_begin(L, MOE_PROF_GATEUP, st) : nullptr;
    cudaEvent_t* p2 = room && (phases & 2) ? prof_begin(L, MOE_PROF_DOWN, st) : nullptr;
    const cudaEvent_t* evp = nullptr;
    if ((p1 || p2) && (p1 || !(phases & 1)) && (p2 || !(phases & 2))) {
      if (p1) { ev[0] = p1[0]; ev[1] = p1[1]; }
      if (p2) { ev[2] = p2[0]; ev[3] = p2[1]; }
      evp = ev;
    }
    cudaError_t ce;
    if (prefill) {
      // the first range (the hits and the shared expert) may come with its
      // tiles already built by the routing CTA
      const bool ready = tiles_built && a.mode == kRangeHits && a.with_shared == g.has_shared;
      tiles_built = false;
      ce = launch_prefill_gemms(g, L->plan, L->rec, L->offsets, L->pbase, N, a.mode, a.with_shared,
                                L->tiles, L->n_tiles, L->slots, L->xq_scales, L->hq_codes,
                                L->hq_scales, L->wsf, L->wtag, L->O, gx, gh, L->err_dev,
                                L->gemm_sms > 0 ? L->gemm_sms : L->num_sms, st, evp, ready);
      L->launches += (fmt_block(g.afmt) ? 4 : 3) - (ready ? 1 : 0);
    } else {
      ce = launch_gemv_decode(g, L->gplan, a, xd, L->xexp, L->h, L->O, n_ent, gemv_sms, st, evp, phases);
      L->launches += (phases & 1) + (phases >> 1 & 1);
    }
    if (ce != cudaSuccess) return cuda_fail(L, ce, prefill ? "launch_prefill_gemms" : "launch_gemv_decode");
    return MOE_OK;
  };
  int grc = gemv((fused ? std::min(g.E, N * g.k) : cap) + (g.has_shared ? 1 : 0), sm_fill ? 1 : 3);
  if (grc) return grc;
  if (sm_fill) {
    // every fill chunk a step can have is queued behind the routing (after the
    // hits' phase 1, whose early start must not wait for these launches); each
    // finds its part of the miss list in the record on the device, so the
    // copies start when the routing ends, not after the host has read it
    const int max_pre = miss_chunks(std::min(g.E, N * g.k));
    cudaStream_t fs = L->fill;
    MOE_CUDA(L, cudaStreamWaitEvent(fs, L->ev_route, 0));
    cudaEvent_t* pf = prof_begin(L, MOE_PROF_FILL, fs);
    for (int c = 0; c < max_pre; ++c) {
      MOE_CUDA(L, launch_fill_sm(g, L->rec, c, L->pool_dev, L->slots, fs));
      MOE_CUDA(L, cudaEventRecord(L->ev_chunk[c], fs));
    }
    prof_end(pf, fs);
    // every chunk launch, including those this step's miss list leaves
    // without work, reads the step record: the step ends (and the next one
    // may rewrite the record and the buffer map) only after all of them
    MOE_CUDA(L, cudaEventRecord(L->ev_fill, fs));
    L->launches += max_pre;
  }

  // Misses.  Every fill starts as soon as the routing is known: first-wave
  // misses go straight into their (free or stale) LRU slots' buffers, later
  // ones into spare buffers, since their LRU slots are still read by this
  // step (the record names each access's buffer); expert-FFN launches over
  // the misses follow their fills.
  size_t fill_bytes = 0;
  int U = -1, n_hit = -1, n_miss = 0, waves = 1, n_chunks = 0;
  const int max_miss = std::min(g.E, N * g.k);
  bool any_miss = true;
  if (dev_fill) {
    cudaStream_t fs = L->fill;
    MOE_CUDA(L, cudaStreamWaitEvent(fs, L->ev_route, 0));
    cudaEvent_t* pf = prof_begin(L, MOE_PROF_FILL, fs);
    MOE_CUDA(L, launch_fill_copy(g, L->rec, max_miss, L->pool_dev, L->slots, fs));
    prof_end(pf, fs);
    L->launches += 1;
    MOE_CUDA(L, cudaEventRecord(L->ev_fill, fs));
    MOE_CUDA(L, cudaStreamWaitEvent(st, L->ev_fill, 0));
    waves = (max_miss + g.S - 1) / g.S;
  } else if (fused) {
    any_miss = false;   // computed (and filled) by the launch above
    a.host_pool = nullptr;
  } else if (!resident) {
    int prc = poll_record(L, seq);
    if (prc) return prc;
    const StepRecord* r = L->rec_host;
    U = r->U;
    n_hit = r->n_hit;
    n_miss = r->n_miss;
    waves = (U + g.S - 1) / g.S;
    const int* ae = rec_expert(const_cast<StepRecord*>(r));
    const int* as = rec_slot(const_cast<StepRecord*>(r), g.E);
    const int* ab = rec_buf(const_cast<StepRecord*>(r), g.E);
    if (U < 0 || U > g.E || n_hit < 0 || n_hit > U || U - g.S > g.X)
      return fail(L, MOE_ERR_STATE, "step record is inconsistent (U=%d, hits=%d)", U, n_hit);
    for (int i = 0; i < U; ++i)
      if (ae[i] < 0 || ae[i] >= g.E || as[i] < 0 || as[i] >= g.S || !buf_ok(g, ab[i]))
        return fail(L, MOE_ERR_STATE, "step record entry %d is out of range", i);
    any_miss = n_hit < U;
    if (any_miss) {
      // the misses' expert FFN runs in chunks, each once its own fills have
      // landed, while later fills still run; a chunk pays one expert-FFN
      // launch ramp, so only long miss lists are cut
      n_chunks = miss_chunks(U - n_hit);
    }
    if (any_miss && sm_fill) {
      fill_bytes = (size_t)(U - n_hit) * g.ebytes;   // the copy kernels were queued behind the routing
    } else if (any_miss) {
      // one copy engine queue in access order (more queues add no bandwidth
      // on this link): consecutive experts bound for consecutive slots go as
      // one copy, and each chunk records when its copies have landed
      cudaStream_t fs = L->fill;
      MOE_CUDA(L, cudaStreamWaitEvent(fs, L->ev_route, 0));
      cudaEvent_t* pf = prof_begin(L, MOE_PROF_FILL, fs);
      const int nm = U - n_hit;
      for (int c = 0; c < n_chunks; ++c) {
        int lo, hi;
        miss_chunk(nm, c, n_chunks, &lo, &hi);
        const int c0 = n_hit + lo, c1 = n_hit + hi;
        for (int i = c0; i < c1;) {
          int j = i + 1;
          while (j < c1 && ae[j] == ae[j - 1] + 1 && ab[j] == ab[j - 1] + 1) ++j;
          cudaError_t ce = cudaSuccess;
          if (L->inject_fill) {
            L->inject_fill = false;
            ce = cudaErrorInvalidValue;
          } else {
            ce = cudaMemcpyAsync(L->slots + (size_t)ab[i] * g.ebytes, L->host_pool + (size_t)ae[i] * g.ebytes,
                                 (size_t)(j - i) * g.ebytes, cudaMemcpyHostToDevice, fs);
          }
          if (ce != cudaSuccess) {
            // the step's misses leave the cache (their slots become free, so a
            // later step fills them again); the fills already issued and the
            // hits' expert FFN finish on their own; y is not written
            cudaGetLastError();
            mirror_apply(L, r);
            mirror_drop_misses(L, r);
            MOE_CUDA(L, launch_lru_drop_misses(g, L->rec, L->slot_of, L->expert_of, st));
            return fail(L, MOE_ERR_FILL, "fill of expert %d could not be issued (%s); the step's %d misses were "
                        "dropped from the cache and y was not written", ae[i], cudaGetErrorString(ce), U - n_hit);
          }
          fill_bytes += (size_t)(j - i) * g.ebytes;
          i = j;
        }
        MOE_CUDA(L, cudaEventRecord(L->ev_chunk[c], fs));
      }
      prof_end(pf, fs);
    }
    mirror_apply(L, r);
  }
  if (sm_fill) {
    grc = gemv(cap + (g.has_shared ? 1 : 0), 2);
    if (grc) return grc;
  }
  if (!resident && any_miss) {
    a.mode = kRangeMisses;
    a.with_shared = 0;
    if (n_chunks > 1 && !prefill) {
      // chunk c of the misses runs once its own copies landed
      const int nm = U - n_hit;
      a.n_chunks = n_chunks;
      for (int c = 0; c < n_chunks; ++c) {
        MOE_CUDA(L, cudaStreamWaitEvent(st, L->ev_chunk[c], 0));
        a.chunk = c;
        int lo, hi;
        miss_chunk(nm, c, n_chunks, &lo, &hi);
        const int c0 = n_hit + lo, c1 = n_hit + hi;
        grc = gemv(c1 - c0, 3);
        if (grc) return grc;
      }
    } else {
      // one launch over every miss once the last copy (one queue, in order) has landed
      if (n_chunks > 0) MOE_CUDA(L, cudaStreamWaitEvent(st, L->ev_chunk[n_chunks - 1], 0));
      grc = gemv(max_miss, 3);
      if (grc) return grc;
    }
  }
  if (sm_fill) MOE_CUDA(L, cudaStreamWaitEvent(st, L->ev_fill, 0));
  pe = prof_begin(L, MOE_PROF_COMBINE, st);
  MOE_CUDA(L, launch_combine(g, L->O, prefill, L->gates, L->row_of, N, yd, st));
  prof_end(pe, st);
  L->launches += 1;
  if (!y_dev) {
    if (!y_direct) MOE_CUDA(L, cudaMemcpyAsync(y, yd, xbytes, cudaMemcpyDeviceToHost, st));
    MOE_CUDA(L, cudaStreamSynchronize(st));
  }
  L->last_N = N;
  L->last_prefill = prefill;
  if (info) {
    info->regime = prefill ? MOE_REGIME_PREFILL : MOE_REGIME_DECODE;
    info->n_distinct = U;
    info->n_hits = n_hit;
    info->n_misses = n_miss;
    info->n_waves = resident ? 1 : waves;
    info->fill_bytes = fill_bytes;
    info->host_synced = (resident || dev_fill || fused) ? 0 : 1;
    info->n_launches = L->launches;
  }
  return MOE_OK;
}

int moe_set_fill_mode(moe_layer_t L, int mode) {
  if (!L) return MOE_ERR_ARG;
  if (mode != MOE_FILL_MEMCPY && mode != MOE_FILL_DEVICE && mode != MOE_FILL_KERNEL && mode != MOE_FILL_FUSED &&
      mode != MOE_FILL_AUTO)
    return fail(L, MOE_ERR_ARG, "unknown fill mode %d", mode);
  if (mode != MOE_FILL_MEMCPY && !L->pool_dev)
    return fail(L, MOE_ERR_STATE, "copy-kernel fills need a registered pinned host pool the device can address");
  L->fill_mode = mode;
  L->fill_mode_chosen = true;
  return MOE_OK;
}

int moe_set_decode_path(moe_layer_t L, int path) {
  if (!L) return MOE_ERR_ARG;
  if (path != MOE_DECODE_AUTO && path != MOE_DECODE_CHAIN && path != MOE_DECODE_STEP)
    return fail(L, MOE_ERR_ARG, "unknown decode path %d", path);
  L->decode_path = path;
  return MOE_OK;
}

int moe_stats(moe_layer_t L, uint64_t* out4) {
  if (!L || !out4) return MOE_ERR_ARG;
  MOE_CUDA(L, cudaDeviceSynchronize());
  MOE_CUDA(L, cudaMemcpy(out4, L->stats, 4 * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

int moe_profile(moe_layer_t L, int enable) {
  if (!L) return MOE_ERR_ARG;
  MOE_CUDA(L, cudaDeviceSynchronize());
  if (enable && L->prof_pool.empty()) {
    L->prof_pool.resize(2 * kProfPairs);
    for (auto& e : L->prof_pool) MOE_CUDA(L, cudaEventCreate(&e));
  }
  L->prof_on = enable != 0;
  L->prof_used = 0;
  L->prof_kind.clear();
  return MOE_OK;
}

int moe_profile_read(moe_layer_t L, double* ms, int* launches) {
  if (!L) return MOE_ERR_ARG;
  MOE_CUDA(L, cudaDeviceSynchronize());
  double acc[MOE_PROF_KINDS] = {0};
  int cnt[MOE_PROF_KINDS] = {0};
  for (size_t i = 0; i < L->prof_kind.size(); ++i) {
    float t = 0.f;
    MOE_CUDA(L, cudaEventElapsedTime(&t, L->prof_pool[2 * i], L->prof_pool[2 * i + 1]));
    acc[L->prof_kind[i]] += t;
    cnt[L->prof_kind[i]] += 1;
  }
  for (int k = 0; k < MOE_PROF_KINDS; ++k) {
    if (ms) ms[k] = acc[k];
    if (launches) launches[k] = cnt[k];
  }
  return MOE_OK;
}

int moe_debug_router(moe_layer_t L, const void* x, int N, int* idx, float* gates, float* logits,
                     void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (N < 0 || N > L->desc.max_tokens) return fail(L, MOE_ERR_ARG, "N out of range");
  if (N == 0) return MOE_OK;
  if (!x || !idx || !gates) return fail(L, MOE_ERR_ARG, "NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(L, launch_router(L->g, static_cast<const __nv_bfloat16*>(x), N, L->Wr, L->Wr_hl,
                            L->g.has_bias ? L->bias : nullptr, logits ? logits : L->logits, idx,
                            gates, L->xexp, L->rcounter, L->err_dev, L->logits2, st));
  return MOE_OK;
}

int moe_debug_permute(moe_layer_t L, const int* idx, int N, int* counts, int* offsets, int* row_of,
                      int* tok_of, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (N < 0 || N > L->desc.max_tokens) return fail(L, MOE_ERR_ARG, "N out of range");
  if (N == 0) return MOE_OK;
  if (!idx || !counts || !offsets || !row_of || !tok_of) return fail(L, MOE_ERR_ARG, "NULL pointer");
  MOE_CUDA(L, launch_permute(L->g, idx, N, counts, offsets, row_of, tok_of, L->perm_scratch,
                             static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_debug_inject(moe_layer_t L, int what, long long arg) {
  if (!L) return MOE_ERR_ARG;
  switch (what) {
    case MOE_INJECT_NONE:
      L->inject_fill = false;
      L->inject_wait = 0;
      return MOE_OK;
    case MOE_INJECT_FILL:
      L->inject_fill = true;
      return MOE_OK;
    case MOE_INJECT_WAIT_LIMIT:
      if (arg <= 0) return fail(L, MOE_ERR_ARG, "the wait limit must be positive");
      L->inject_wait = arg;
      return MOE_OK;
    default:
      return fail(L, MOE_ERR_ARG, "unknown injection %d", what);
  }
}

int moe_debug_alloc_fault(long long nth, long long* live_out) {
  if (nth < 0) return MOE_ERR_ARG;
  g_alloc_countdown.store(nth);
  if (live_out) {
    live_out[0] = g_live_dev.load();
    live_out[1] = g_live_host.load();
  }
  return MOE_OK;
}

int moe_debug_last_step(moe_layer_t L, int* idx, float* gates, int* counts, int* offsets, int* row_of,
                        int* tok_of, int* n_out, void* stream) {
  if (!L) return MOE_ERR_ARG;
  const int N = L->last_N;
  if (N <= 0) return fail(L, MOE_ERR_STATE, "no moe_forward has run on this layer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Geo& g = L->g;
  const size_t nk = (size_t)N * g.k;
  if (idx) MOE_CUDA(L, cudaMemcpyAsync(idx, L->idx, nk * 4, cudaMemcpyDeviceToDevice, st));
  if (gates) MOE_CUDA(L, cudaMemcpyAsync(gates, L->gates, nk * 4, cudaMemcpyDeviceToDevice, st));
  if (counts) MOE_CUDA(L, cudaMemcpyAsync(counts, L->counts, (size_t)g.E * 4, cudaMemcpyDeviceToDevice, st));
  if (offsets) MOE_CUDA(L, cudaMemcpyAsync(offsets, L->offsets, (size_t)(g.E + 1) * 4, cudaMemcpyDeviceToDevice, st));
  if (row_of) MOE_CUDA(L, cudaMemcpyAsync(row_of, L->row_of, nk * 4, cudaMemcpyDeviceToDevice, st));
  if (tok_of) MOE_CUDA(L, cudaMemcpyAsync(tok_of, L->tok_of, nk * 4, cudaMemcpyDeviceToDevice, st));
  if (n_out) *n_out = N;
  return MOE_OK;
}

int moe_debug_last_hidden(moe_layer_t L, float* h, uint8_t* hq_codes, uint8_t* hq_scales, void* stream) {
  if (!L) return MOE_ERR_ARG;
  const int N = L->last_N;
  if (N <= 0) return fail(L, MOE_ERR_STATE, "no moe_forward has run on this layer");
  if (h && L->last_prefill) return fail(L, MOE_ERR_STATE, "the last call ran the prefill regime (no fp32 h)");
  if ((hq_codes || hq_scales) && !L->last_prefill)
    return fail(L, MOE_ERR_STATE, "the last call ran the decode regime (no quantised h)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Geo& g = L->g;
  const size_t rows = (size_t)N * g.k + (g.has_shared ? N : 0);
  if (h) MOE_CUDA(L, cudaMemcpyAsync(h, L->h, rows * 2 * g.f * 4, cudaMemcpyDeviceToDevice, st));
  if (hq_codes)
    MOE_CUDA(L, cudaMemcpyAsync(hq_codes, L->hq_codes, rows * g.f * fmt_code_bits(g.afmt) / 8,
                                cudaMemcpyDeviceToDevice, st));
  if (hq_scales && fmt_scale_row(g.afmt, g.f))   // stored by padded block: back to rows
    MOE_CUDA(L, launch_untile_hscales(g, L->hq_scales, L->offsets, L->pbase, N, hq_scales, st));
  return MOE_OK;
}

int moe_debug_step_trace(moe_layer_t L, uint64_t* out, int cap, int* n_cta, int* n_marks) {
  if (!L) return MOE_ERR_ARG;
  const int G = L->step_trace_grid;
  if (n_cta) *n_cta = G;
  if (n_marks) *n_marks = kStepMarks;
  if (G == 0) return fail(L, MOE_ERR_STATE, "no fused step ran while kernel timing was on");
  if (!out || cap < G * kStepMarks) return fail(L, MOE_ERR_ARG, "out must hold %d entries", G * kStepMarks);
  MOE_CUDA(L, cudaDeviceSynchronize());
  MOE_CUDA(L, cudaMemcpy(out, L->step_trace, (size_t)G * kStepMarks * 8, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

int moe_debug_dequant(moe_layer_t L, int slot, int m, float* out, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (m < 0 || m > 2 || !out) return fail(L, MOE_ERR_ARG, "bad matrix or NULL out");
  const uint8_t* base;
  if (slot == -1) {
    if (!L->g.has_shared) return fail(L, MOE_ERR_STATE, "no shared expert");
    base = L->shared_w;
  } else if (slot >= 0 && slot < L->g.S) {
    int b = -1;
    int rc = slot_buffer(L, slot, &b);
    if (rc) return rc;
    base = L->slots + (size_t)b * L->g.ebytes;
  } else {
    return fail(L, MOE_ERR_ARG, "slot %d out of range", slot);
  }
  MOE_CUDA(L, launch_dequant(L->g, base, m, out, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_debug_actquant(moe_layer_t L, const float* v, int rows, int K, uint8_t* codes, uint8_t* scales,
                       int which, void* stream) {
  if (!L) return MOE_ERR_ARG;
  if (rows < 0 || K <= 0 || K % 32) return fail(L, MOE_ERR_ARG, "rows >= 0 and K a multiple of 32");
  if (rows == 0) return MOE_OK;
  if (!v || !codes || !scales) return fail(L, MOE_ERR_ARG, "NULL pointer");
  const float gs = which ? L->desc.act_scale_h : L->desc.act_scale_x;
  MOE_CUDA(L, launch_actquant(L->g, v, rows, K, codes, scales, L->g.fmt == MOE_NVFP4 ? gs : 1.0f,
                              static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}


// ---------------------------------------------------------------- stacks

const char* moe_stack_last_error(moe_stack_t K) { return K ? K->err.c_str() : "null stack"; }

static int stack_fail(moe_stack* K, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  K->err = buf;
  return code;
}

static void stack_free(moe_stack* K) {
  cudaDeviceSynchronize();
  for (int l = (int)K->layers.size() - 1; l >= 0; --l) {
    release(K->layers[l]);
    delete K->layers[l];
  }
  K->layers.clear();
  if (K->ev_pf) cudaEventDestroy(K->ev_pf);
  if (K->ev_in) cudaEventDestroy(K->ev_in);
  if (K->ev_route) cudaEventDestroy(K->ev_route);
  delete K;
}

int moe_stack_create(const moe_layer_desc* desc, int n_layers, moe_stack_t* out) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  if (!desc || n_layers < 1 || n_layers > kMaxStackLayers) return MOE_ERR_ARG;
  std::string why;
  const long long keys = (long long)n_layers * desc->E;
  int rc = check_desc(desc, &why, (int)std::min<long long>(keys, kMaxE));
  if (rc) return rc;
  moe_stack* K = new (std::nothrow) moe_stack();
  if (!K) return MOE_ERR_OOM;
  for (int l = 0; l < n_layers && rc == MOE_OK; ++l) {
    moe_layer* L = nullptr;
    rc = create_layer(desc, l ? K->layers[0] : nullptr, l, n_layers, &L);
    if (rc == MOE_OK) {
      L->stack = K;
      K->layers.push_back(L);
    }
  }
  if (rc == MOE_OK) {
    moe_layer* L0 = K->layers[0];
    const Geo& g = L0->g;
    const size_t hb = (size_t)desc->max_tokens * g.d * 2;
    rc = dalloc(L0, &K->hid[0], hb);
    if (rc == MOE_OK) rc = dalloc(L0, &K->hid[1], hb);
    if (rc == MOE_OK) rc = dalloc(L0, &K->ones, (size_t)g.E * 4);
    if (rc == MOE_OK) rc = dalloc(L0, &K->pf_stats, 64);
    if (rc == MOE_OK) {
      std::vector<int> one(g.E, 1);
      if (cudaMemcpy(K->ones, one.data(), (size_t)g.E * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
          cudaMemset(K->pf_stats, 0, 64) != cudaSuccess ||
          cudaEventCreateWithFlags(&K->ev_pf, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&K->ev_in, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&K->ev_route, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        rc = MOE_ERR_CUDA;
      }
    }
  }
  if (rc != MOE_OK) {
    stack_free(K);
    return rc;
  }
  *out = K;
  return MOE_OK;
}

int moe_stack_destroy(moe_stack_t K) {
  if (!K) return MOE_ERR_ARG;
  for (moe_layer* L : K->layers) L->stack = nullptr;
  stack_free(K);
  return MOE_OK;
}

int moe_stack_layer(moe_stack_t K, int l, moe_layer_t* out) {
  if (!K || !out) return MOE_ERR_ARG;
  if (l < 0 || l >= (int)K->layers.size())
    return stack_fail(K, MOE_ERR_ARG, "layer %d outside [0, %d)", l, (int)K->layers.size());
  *out = K->layers[l];
  return MOE_OK;
}

int moe_stack_set_prefetch_copy(moe_stack_t K, int fill) {
  if (!K) return MOE_ERR_ARG;
  if (fill == MOE_FILL_AUTO) fill = MOE_FILL_MEMCPY;
  if (fill != MOE_FILL_KERNEL && fill != MOE_FILL_MEMCPY)
    return stack_fail(K, MOE_ERR_ARG, "prefetch copies are MOE_FILL_KERNEL or MOE_FILL_MEMCPY (got %d)", fill);
  K->prefetch_copy = fill;
  return MOE_OK;
}

int moe_stack_set_prefetch(moe_stack_t K, int mode) {
  if (!K) return MOE_ERR_ARG;
  const Geo& g = K->layers[0]->g;
  if (mode != MOE_PREFETCH_AUTO && mode != MOE_PREFETCH_NONE && mode != MOE_PREFETCH_SERIAL &&
      mode != MOE_PREFETCH_OVERLAP)
    return stack_fail(K, MOE_ERR_ARG, "unknown prefetch mode %d", mode);
  if (mode == MOE_PREFETCH_SERIAL && g.S < g.E)
    return stack_fail(K, MOE_ERR_UNSUPPORTED, "a whole-layer prefetch needs n_slots >= E (%d < %d)", g.S, g.E);
  if (mode == MOE_PREFETCH_OVERLAP && g.S < 2 * g.E)
    return stack_fail(K, MOE_ERR_UNSUPPORTED, "an overlapped prefetch needs n_slots >= 2 E (%d < %d)", g.S, 2 * g.E);
  K->prefetch = mode;
  return MOE_OK;
}

int moe_stack_prefetch_stats(moe_stack_t K, uint64_t* out4) {
  if (!K || !out4) return MOE_ERR_ARG;
  moe_layer* L0 = K->layers[0];
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(out4, K->pf_stats, 32, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return stack_fail(K, MOE_ERR_CUDA, "reading the prefetch counters failed");
  }
  (void)L0;
  return MOE_OK;
}

// The whole of layer m as one step of the shared table (every expert accessed,
// hits first, misses ascending), then its misses copied from the layer's host
// pool, all on stream st: by kFillSms CTAs reading the step record on the
// device, or (copy_engine) by cudaMemcpyAsync once the host has read the
// record the LRU kernel writes into mapped pinned memory (runs of experts
// bound for consecutive buffers as one copy).
static int stack_prefetch(moe_stack* K, int m, cudaStream_t st, bool copy_engine) {
  moe_layer* M = K->layers[m];
  const Geo& g = M->g;
  const unsigned long long seq = copy_engine ? ++M->step_seq : 0ull;
  cudaError_t e = launch_lru_step(g, K->ones, nullptr, M->slot_of, M->expert_of, M->stamp, M->clock, M->buf, M->rec,
                                  K->pf_stats, copy_engine ? M->rec_host_dev : nullptr, seq, st);
  M->launches += 1;
  if (e == cudaSuccess && !copy_engine) {
    for (int c = 0; e == cudaSuccess && c < miss_chunks(g.E); ++c)
      e = launch_fill_sm(g, M->rec, c, M->pool_dev, M->slots, st);
    M->launches += miss_chunks(g.E);
  }
  if (e == cudaSuccess && copy_engine) e = cudaEventRecord(M->ev_route, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return stack_fail(K, MOE_ERR_CUDA, "prefetch of layer %d: %s", m, cudaGetErrorString(e));
  }
  if (!copy_engine) return MOE_OK;
  const int prc = poll_record(M, seq);
  if (prc) return stack_fail(K, prc, "prefetch of layer %d: %s", m, M->err.c_str());
  const StepRecord* r = M->rec_host;
  const int U = r->U, nh = r->n_hit;
  const int* ae = rec_expert(const_cast<StepRecord*>(r));
  const int* as = rec_slot(const_cast<StepRecord*>(r), g.E);
  const int* ab = rec_buf(const_cast<StepRecord*>(r), g.E);
  if (U != g.E || nh < 0 || nh > U)
    return stack_fail(K, MOE_ERR_STATE, "prefetch record of layer %d is inconsistent (U=%d, hits=%d)", m, U, nh);
  for (int i = 0; i < U; ++i)
    if (ae[i] < 0 || ae[i] >= g.E || as[i] < 0 || as[i] >= g.S || !buf_ok(g, ab[i]))
      return stack_fail(K, MOE_ERR_STATE, "prefetch record entry %d of layer %d is out of range", i, m);
  for (int i = nh; i < U;) {
    int j = i + 1;
    while (j < U && ae[j] == ae[j - 1] + 1 && ab[j] == ab[j - 1] + 1) ++j;
    e = cudaMemcpyAsync(M->slots + (size_t)ab[i] * g.ebytes, M->host_pool + (size_t)ae[i] * g.ebytes,
                        (size_t)(j - i) * g.ebytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return stack_fail(K, MOE_ERR_FILL, "prefetch copy of layer %d, expert %d: %s", m, ae[i], cudaGetErrorString(e));
    }
    i = j;
  }
  return MOE_OK;
}

int moe_stack_forward(moe_stack_t K, const void* x, int N, void* y, void* stream, int regime,
                      moe_forward_info* info) {
  if (!K) return MOE_ERR_ARG;
  const int nl = (int)K->layers.size();
  moe_layer* L0 = K->layers[0];
  const Geo& g = L0->g;
  if (info) {
    std::memset(info, 0, sizeof *info);
    info->n_tokens = N;
  }
  if (N < 0 || N > L0->desc.max_tokens)
    return stack_fail(K, MOE_ERR_ARG, "N = %d outside [0, max_tokens = %d]", N, L0->desc.max_tokens);
  if (N == 0) return MOE_OK;
  if (!x || !y) return stack_fail(K, MOE_ERR_ARG, "x or y is NULL");
  if (regime != MOE_REGIME_AUTO && regime != MOE_REGIME_DECODE && regime != MOE_REGIME_PREFILL)
    return stack_fail(K, MOE_ERR_ARG, "unknown regime %d", regime);
  const bool prefill = regime == MOE_REGIME_PREFILL || (regime == MOE_REGIME_AUTO && N > 64 && L0->plan);
  if (prefill && !L0->plan)
    return stack_fail(K, MOE_ERR_UNSUPPORTED, "the prefill regime needs d_model and d_ff multiples of 256");
  int mode = MOE_PREFETCH_NONE;
  if (prefill) {
    mode = K->prefetch;
    if (mode == MOE_PREFETCH_AUTO)
      mode = g.S >= 2 * g.E ? MOE_PREFETCH_OVERLAP : g.S >= g.E ? MOE_PREFETCH_SERIAL : MOE_PREFETCH_NONE;
    if (mode != MOE_PREFETCH_NONE)
      for (moe_layer* M : K->layers)
        if (!M->pool_dev)
          return stack_fail(K, MOE_ERR_NOT_INSTALLED, "layer %d has no device-addressable host pool", M->index);
  }
  const int reg = prefill ? MOE_REGIME_PREFILL : MOE_REGIME_DECODE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t fs = L0->fill;
  int launches = 0, fused = 0;
  auto fwd = [&](int l, const void* in, void* outp) -> int {
    moe_layer* M = K->layers[l];
    moe_forward_info fi{};
    const int rc = moe_forward(M, in, N, outp, stream, reg, &fi);
    if (rc) return stack_fail(K, rc, "layer %d: %s", l, M->err.c_str());
    launches += fi.n_launches;
    fused += fi.fused_step;
    return MOE_OK;
  };
  auto cuda_k = [&](cudaError_t e, const char* what) -> int {
    if (e == cudaSuccess) return MOE_OK;
    cudaGetLastError();
    return stack_fail(K, MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  };
  int rc = MOE_OK;
  const bool ce = K->prefetch_copy == MOE_FILL_MEMCPY;
  if (mode != MOE_PREFETCH_NONE) {
    // layer 0's experts, after the caller's earlier work on st
    L0->launches = 0;
    if ((rc = cuda_k(cudaEventRecord(K->ev_in, st), "cudaEventRecord"))) return rc;
    if ((rc = cuda_k(cudaStreamWaitEvent(fs, K->ev_in, 0), "cudaStreamWaitEvent"))) return rc;
    if ((rc = stack_prefetch(K, 0, fs, ce))) return rc;
    launches += L0->launches;
    if ((rc = cuda_k(cudaEventRecord(K->ev_pf, fs), "cudaEventRecord"))) return rc;
    if ((rc = cuda_k(cudaStreamWaitEvent(st, K->ev_pf, 0), "cudaStreamWaitEvent"))) return rc;
  }
  const void* in = x;
  for (int l = 0; l < nl; ++l) {
    void* outp = l == nl - 1 ? y : static_cast<void*>(K->hid[l & 1]);
    moe_layer* M = K->layers[l];
    const bool ov = mode == MOE_PREFETCH_OVERLAP && l + 1 < nl;
    M->assume_resident = mode != MOE_PREFETCH_NONE;
    M->ev_after_route = ov ? K->ev_route : nullptr;
    // the prefill GEMM leaves the fill kernels' SMs free while the next
    // layer streams in (copy-engine prefetches need no SM)
    M->gemm_sms = ov && !ce ? M->num_sms - kFillSms : 0;
    rc = fwd(l, in, outp);
    M->assume_resident = false;
    M->ev_after_route = nullptr;
    M->gemm_sms = 0;
    if (rc) return rc;
    if (mode != MOE_PREFETCH_NONE && l + 1 < nl) {
      moe_layer* Mn = K->layers[l + 1];
      Mn->launches = 0;
      if (ov) {
        // layer l + 1 streams in while layer l computes: its table step
        // follows layer l's (its experts are the most recent, so with
        // n_slots >= 2 E none of them is evicted), its copies run on the fill
        // SMs, and layer l + 1 starts once they landed
        if ((rc = cuda_k(cudaStreamWaitEvent(fs, K->ev_route, 0), "cudaStreamWaitEvent"))) return rc;
        if ((rc = stack_prefetch(K, l + 1, fs, ce))) return rc;
        if ((rc = cuda_k(cudaEventRecord(K->ev_pf, fs), "cudaEventRecord"))) return rc;
        if ((rc = cuda_k(cudaStreamWaitEvent(st, K->ev_pf, 0), "cudaStreamWaitEvent"))) return rc;
      } else {
        // after layer l on the caller's stream
        if ((rc = stack_prefetch(K, l + 1, st, ce))) return rc;
      }
      launches += Mn->launches;
    }
    in = outp;
  }
  if (info) {
    info->regime = reg;
    info->n_distinct = info->n_hits = info->n_misses = -1;
    info->n_waves = 1;
    info->n_launches = launches;
    info->fused_step = fused;
  }
  return MOE_OK;
}

}  // extern "C"
