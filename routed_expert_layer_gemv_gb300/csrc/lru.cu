// Device-side LRU slot table of the expert cache, updated once per step.
//
// FreeToken keeps the routed experts in a global LRU expert cache in GPU
// memory; hits are served from it and misses are loaded into it from host
// memory ("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二, "Decode" and
// "LRU 为什么赢" paragraphs).  The pages leave the per-step order open; this
// table takes the step's distinct experts U as accesses, hits first (ascending
// id) then misses (ascending id).  A hit becomes most recently used; a miss
// takes the lowest free slot, else evicts the least recently used expert.
//
// Closed form used here (one CTA, no sequential loop over accesses).  Let
// h = #hits and Q = the victim queue: free slots ascending, then the occupied
// slots whose expert is not hit this step, by ascending recency stamp; |Q| =
// S - h.  Access i (in access order) uses
//   slot(i) = slot of the hit           if i < h,
//             Q[i - h]                  if h <= i < S,
//             slot(i - S)               if i >= S,
// because once Q is used up every slot holds an expert accessed this step and
// they leave in access order.  So two accesses share a slot only if they are a
// multiple of S apart: the accesses form waves of S, each wave's slots are
// distinct, and a wave's fills must wait for the previous wave's compute.
// Stamps: access i gets clock + 1 + i; the clock advances by |U|.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kLruThreads = 1024;

MOE_DEV int excl_scan_1024(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = sh[lane];
    int si = s;
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    sh[lane] = si - s;
    if (lane == 31) sh[32] = si;
  }
  __syncthreads();
  int r = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kLruThreads)
lru_step_kernel(const int* __restrict__ counts, int E, int S, int* __restrict__ slot_of,
                int* __restrict__ expert_of, unsigned long long* __restrict__ stamp,
                unsigned long long* __restrict__ clock, StepRecord* __restrict__ rec) {
  __shared__ int sh[33];
  __shared__ int q[kMaxE];        // victim queue (slots)
  __shared__ int q_old[kMaxE];    // expert that held q[i] before the step (-1 free)
  __shared__ int acc_e[kMaxE], acc_s[kMaxE];
  const int tid = threadIdx.x;
  const unsigned long long clk = *clock;

  // hits / misses over experts (E <= 1024: one expert per thread)
  const int e = tid;
  const bool inU = e < E && counts[e] > 0;
  const int cur = e < E ? slot_of[e] : -1;
  const bool hit = inU && cur >= 0, miss = inU && cur < 0;
  int n_hit, n_miss;
  const int hr = excl_scan_1024(hit ? 1 : 0, &n_hit, sh);
  const int mr = excl_scan_1024(miss ? 1 : 0, &n_miss, sh);
  const int U = n_hit + n_miss;

  // victim queue over slots (S <= E <= 1024: one slot per thread)
  const int s = tid;
  int old = -1;
  bool fre = false, stale = false;
  unsigned long long st = 0;
  if (s < S) {
    old = expert_of[s];
    fre = old < 0 || old >= E;
    stale = !fre && counts[old] == 0;
    st = stamp[s];
  }
  int n_free;
  const int fr = excl_scan_1024(fre ? 1 : 0, &n_free, sh);
  if (fre) { q[fr] = s; q_old[fr] = -1; }
  if (stale) {
    int r = 0;
    for (int s2 = 0; s2 < S; ++s2) {
      int o2 = expert_of[s2];
      if (o2 < 0 || o2 >= E || counts[o2] > 0) continue;
      unsigned long long t2 = stamp[s2];
      r += (t2 < st || (t2 == st && s2 < s)) ? 1 : 0;
    }
    if (n_free + r < S) {
      q[n_free + r] = s;
      q_old[n_free + r] = old;
    }
  }
  __syncthreads();

  // accesses 0 .. min(U, S)-1 first, then the later waves reuse slot(i - S)
  if (hit) { acc_e[hr] = e; acc_s[hr] = cur; }
  if (miss) {
    const int i = n_hit + mr;
    acc_e[i] = e;
    if (i < S) acc_s[i] = q[i - n_hit];   // i - n_hit < S - n_hit = |Q|
  }
  __syncthreads();
  for (int i = S + tid; i < U; i += kLruThreads) acc_s[i] = acc_s[i % S];
  __syncthreads();

  int* r_e = rec_expert(rec);
  int* r_s = rec_slot(rec, E);
  int* r_v = rec_evicted(rec, E);
  for (int i = tid; i < U; i += kLruThreads) {
    r_e[i] = acc_e[i];
    r_s[i] = acc_s[i];
    int ev = -1;
    if (i >= S) ev = acc_e[i - S];
    else if (i >= n_hit) ev = q_old[i - n_hit];
    r_v[i] = ev;
  }
  if (tid == 0) {
    rec->U = U;
    rec->n_hit = n_hit;
    rec->n_miss = n_miss;
    rec->S = S;
  }
  // table update: experts pushed out of Q lose their slot
  for (int i = n_hit + tid; i < min(U, S); i += kLruThreads) {
    int ev = q_old[i - n_hit];
    if (ev >= 0 && ev < E) slot_of[ev] = -1;
  }
  __syncthreads();
  for (int i = tid; i < U; i += kLruThreads) {
    const int ex = acc_e[i], sl = acc_s[i];
    if (sl < 0 || sl >= S) continue;   // only a corrupted table gets here
    if (i + S < U) {
      slot_of[ex] = -1;            // evicted later in this same step
    } else {
      slot_of[ex] = sl;
      expert_of[sl] = ex;
      stamp[sl] = clk + 1ull + (unsigned long long)i;
    }
  }
  if (tid == 0) *clock = clk + (unsigned long long)U;
}

__global__ void lru_install_kernel(int expert, int slot, int* slot_of, int* expert_of,
                                   unsigned long long* stamp, unsigned long long* clock) {
  const int prev = slot_of[expert];
  if (prev >= 0 && prev != slot) expert_of[prev] = -1;
  const int old = expert_of[slot];
  if (old >= 0 && old != expert) slot_of[old] = -1;
  expert_of[slot] = expert;
  slot_of[expert] = slot;
  const unsigned long long c = *clock + 1ull;
  *clock = c;
  stamp[slot] = c;
}

__global__ void counts_from_list_kernel(const int* __restrict__ list, int n, int E,
                                        int* __restrict__ counts) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int c = 0;
  for (int i = 0; i < n; ++i) c += list[i] == e ? 1 : 0;
  counts[e] = c;
}

}  // namespace

cudaError_t launch_lru_step(const Geo& g, const int* counts, int* slot_of, int* expert_of,
                            unsigned long long* stamp, unsigned long long* clock,
                            StepRecord* rec, cudaStream_t st) {
  lru_step_kernel<<<1, kLruThreads, 0, st>>>(counts, g.E, g.S, slot_of, expert_of, stamp, clock,
                                             rec);
  return cudaGetLastError();
}

cudaError_t launch_lru_install(const Geo& g, int expert, int slot, int* slot_of, int* expert_of,
                               unsigned long long* stamp, unsigned long long* clock,
                               cudaStream_t st) {
  (void)g;
  lru_install_kernel<<<1, 1, 0, st>>>(expert, slot, slot_of, expert_of, stamp, clock);
  return cudaGetLastError();
}

cudaError_t launch_counts_from_list(const Geo& g, const int* experts, int n, int* counts,
                                    cudaStream_t st) {
  counts_from_list_kernel<<<(g.E + 255) / 256, 256, 0, st>>>(experts, n, g.E, counts);
  return cudaGetLastError();
}

}  // namespace moe
