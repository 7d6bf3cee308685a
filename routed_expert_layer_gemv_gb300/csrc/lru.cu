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
#include "lru_dev.cuh"
#include "permute_dev.cuh"
#include "tiles_dev.cuh"

namespace moe {

namespace {

constexpr int kLruThreads = 1024;
using lru::LruRegs;
using lru::LruSmem;
using lru::lru_load;
using lru::lru_park;

__global__ void __launch_bounds__(kLruThreads)
lru_step_kernel(const int* __restrict__ counts, const int* __restrict__ offsets, int E, int S, int X,
                int key0, int keys, int* __restrict__ slot_of, int* __restrict__ expert_of, unsigned long long* __restrict__ stamp,
                unsigned long long* __restrict__ clock, int* __restrict__ buf, StepRecord* __restrict__ rec,
                unsigned long long* __restrict__ stats, StepRecord* host_rec, unsigned long long seq) {
  __shared__ LruSmem m;
  lru_park(lru_load(E, S, X, key0, slot_of, expert_of, stamp, clock, buf), E, S, X, m);
  __syncthreads();
  lru::lru_body<kLruThreads>(counts, offsets, nullptr, E, S, X, key0, keys, slot_of, expert_of, stamp, clock, buf,
                             rec, stats, host_rec, seq, m);
}

// Middle of the routing tail of large batches (N > 128), one CTA: the scan
// of the permutation's block histograms (counts, offsets), the padded
// 128-row blocks of each expert's rows for the prefill GEMM (pbase, when
// given: expert e's first block, pbase[E] the shared expert's, pbase[E + 1]
// the total), then the LRU step on the counts, then (tiles given) the
// prefill GEMM's tile list of the step's hits and the shared expert.  The
// scatter of the rows follows in its own launch.
__global__ void __launch_bounds__(kLruThreads)
scan_lru_kernel(int* __restrict__ hist, int nblk, int E, int S, int X, int key0, int keys, int* __restrict__ counts,
                int* __restrict__ offsets, int* __restrict__ pbase, int N, int k, int with_shared, int shb,
                int* __restrict__ slot_of, int* __restrict__ expert_of, unsigned long long* __restrict__ stamp,
                unsigned long long* __restrict__ clock, int* __restrict__ buf, StepRecord* __restrict__ rec,
                unsigned long long* __restrict__ stats, StepRecord* host_rec, unsigned long long seq,
                tl::Tile* __restrict__ tiles, int* __restrict__ ents, int* __restrict__ n_tiles) {
  __shared__ LruSmem m;
  __shared__ int carry;
  const LruRegs lr = lru_load(E, S, X, key0, slot_of, expert_of, stamp, clock, buf);
  const int c = perm::scan_hist(hist, nblk, E, counts, offsets, m.sh);
  if (pbase != nullptr) {
    const int e = threadIdx.x;
    int total;
    const int pre = perm::block_excl_scan(e < E ? (c + kPrefillTileRows - 1) / kPrefillTileRows : 0, &total, m.sh);
    if (e < E) pbase[e] = pre;
    if (e == 0) {
      pbase[E] = total;
      pbase[E + 1] = total + (with_shared ? (N + kPrefillTileRows - 1) / kPrefillTileRows : 0);
    }
  }
  lru_park(lr, E, S, X, m);
  __syncthreads();   // counts and offsets (global, this CTA's writes) are visible to every thread
  lru::lru_body<kLruThreads>(counts, offsets, nullptr, E, S, X, key0, keys, slot_of, expert_of, stamp, clock, buf,
                             rec, stats, host_rec, seq, m);
  if (tiles != nullptr && pbase != nullptr) {
    __syncthreads();   // the record (global, this CTA's writes) is visible to every thread
    tl::build_tiles(rec, offsets, pbase, E, S, X, shb, key0, N, k, kRangeHits, with_shared, tiles, ents, n_tiles,
                    m.sh, &carry);
  }
}

// Decode routing tail in one CTA (N <= 128): the permutation of the top-k ids
// (as perm_single in permute.cu), then the LRU step on the counts it found.
__global__ void __launch_bounds__(kLruThreads)
route_tail_kernel(const int* __restrict__ idx, int N, int k, int E, int S, int X, int key0, int keys,
                  int* __restrict__ counts,
                  int* __restrict__ offsets, int* __restrict__ row_of, int* __restrict__ tok_of,
                  int* __restrict__ slot_of, int* __restrict__ expert_of,
                  unsigned long long* __restrict__ stamp, unsigned long long* __restrict__ clock,
                  int* __restrict__ buf, StepRecord* __restrict__ rec, unsigned long long* __restrict__ stats,
                  StepRecord* host_rec, unsigned long long seq) {
  __shared__ LruSmem m;
  extern __shared__ uint32_t dsm[];
  uint32_t* cm = dsm;                                            // [E][4]
  int* cnt = reinterpret_cast<int*>(cm + E * perm::kPermWarps);  // [E]
  int* off = cnt + E;                                            // [E]
  int* rows = off + E;                                           // [128][k]
  uint32_t* tb = reinterpret_cast<uint32_t*>(rows + perm::kTokPerBlock * k);   // [128][ceil(E/32)]
  // the table was last written by the previous step's tail, which finished
  // before the router began: its loads go out before waiting for the router
  pdl_trigger();
  const LruRegs lr = lru_load(E, S, X, key0, slot_of, expert_of, stamp, clock, buf);
  pdl_wait();
  perm::stage_rows(idx, N, k, 0, rows);
  lru_park(lr, E, S, X, m);
  __syncthreads();
  perm::build_ballots_par(rows, k, E, N, tb, cm);
  const int e = threadIdx.x;
  const int c = e < E ? perm::block_count(cm, e) : 0;
  int tot;
  const int ex = perm::block_excl_scan(c, &tot, m.sh);
  if (e < E) {
    counts[e] = c;
    offsets[e] = ex;
    cnt[e] = c;
    off[e] = ex;
  }
  if (e == 0) offsets[E] = tot;
  __syncthreads();
  const int t = threadIdx.x;
  if (t < N) {
    for (int j = 0; j < k; ++j) {
      const int ej = rows[t * k + j];
      const int r = off[ej] + perm::rank_in_block(cm, ej);
      row_of[(size_t)t * k + j] = r;
      tok_of[r] = t;
    }
  }
  __syncthreads();
  lru::lru_body<kLruThreads>(cnt, off, cm, E, S, X, key0, keys, slot_of, expert_of, stamp, clock, buf, rec, stats,
                             host_rec, seq, m);
}

// Key `expert` (a key of the table) into `slot`, most recently used.
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

__global__ void lru_drop_misses_kernel(const StepRecord* __restrict__ rec, int E, int S, int key0, int* slot_of,
                                       int* expert_of) {
  const int U = min(max(rec->U, 0), E), nh = min(max(rec->n_hit, 0), U);
  const int* ae = rec_expert(const_cast<StepRecord*>(rec));
  for (int i = nh + (int)threadIdx.x; i < U; i += blockDim.x) {
    const int e = ae[i];
    if (e < 0 || e >= E) continue;
    const int s = slot_of[key0 + e];
    if (s >= 0 && s < S) {
      expert_of[s] = -1;
      slot_of[key0 + e] = -1;
    }
  }
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

cudaError_t launch_lru_step(const Geo& g, const int* counts, const int* offsets, int* slot_of,
                            int* expert_of, unsigned long long* stamp, unsigned long long* clock,
                            int* buf, StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                            unsigned long long seq, cudaStream_t st) {
  lru_step_kernel<<<1, kLruThreads, 0, st>>>(counts, offsets, g.E, g.S, g.X, g.key0, g.keys, slot_of, expert_of,
                                             stamp, clock, buf, rec, stats, host_rec, seq);
  return cudaGetLastError();
}

cudaError_t launch_scan_lru(const Geo& g, int N, void* perm_scratch, int* counts, int* offsets, int* pbase,
                            int* slot_of, int* expert_of, unsigned long long* stamp, unsigned long long* clock,
                            int* buf, StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                            unsigned long long seq, void* tiles, int* n_tiles, cudaStream_t st) {
  const int nblk = (N + perm::kTokPerBlock - 1) / perm::kTokPerBlock;
  tl::Tile* tp = static_cast<tl::Tile*>(tiles);
  int* ents = tp ? reinterpret_cast<int*>(tp + prefill_max_tiles(g, N)) : nullptr;
  scan_lru_kernel<<<1, kLruThreads, 0, st>>>(static_cast<int*>(perm_scratch), nblk, g.E, g.S, g.X, g.key0, g.keys,
                                             counts, offsets, pbase, N, g.k, g.has_shared, g.shb, slot_of, expert_of,
                                             stamp, clock, buf, rec, stats, host_rec, seq, tp, ents, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_route_tail(const Geo& g, const int* idx, int N, int* counts, int* offsets,
                              int* row_of, int* tok_of, int* slot_of, int* expert_of,
                              unsigned long long* stamp, unsigned long long* clock, int* buf,
                              StepRecord* rec, unsigned long long* stats, StepRecord* host_rec,
                              unsigned long long seq, cudaStream_t st) {
  const size_t smem = (size_t)g.E * perm::kPermWarps * 4 + (size_t)2 * g.E * 4 +
                      (size_t)perm::kTokPerBlock * g.k * 4 + (size_t)perm::kTokPerBlock * ((g.E + 31) / 32) * 4;
  cudaError_t e = ensure_smem_limit((const void*)route_tail_kernel, 64 * 1024);
  if (e != cudaSuccess) return e;
  return launch_pdl(route_tail_kernel, dim3(1), dim3(kLruThreads), smem, st, idx, N, g.k, g.E, g.S, g.X, g.key0,
                    g.keys, counts,
                    offsets, row_of, tok_of, slot_of, expert_of, stamp, clock, buf, rec, stats, host_rec, seq);
}

cudaError_t launch_lru_install(const Geo& g, int expert, int slot, int* slot_of, int* expert_of,
                               unsigned long long* stamp, unsigned long long* clock,
                               cudaStream_t st) {
  lru_install_kernel<<<1, 1, 0, st>>>(g.key0 + expert, slot, slot_of, expert_of, stamp, clock);
  return cudaGetLastError();
}

cudaError_t launch_lru_drop_misses(const Geo& g, const StepRecord* rec, int* slot_of, int* expert_of,
                                   cudaStream_t st) {
  lru_drop_misses_kernel<<<1, 256, 0, st>>>(rec, g.E, g.S, g.key0, slot_of, expert_of);
  return cudaGetLastError();
}

cudaError_t launch_counts_from_list(const Geo& g, const int* experts, int n, int* counts,
                                    cudaStream_t st) {
  counts_from_list_kernel<<<(g.E + 255) / 256, 256, 0, st>>>(experts, n, g.E, counts);
  return cudaGetLastError();
}

}  // namespace moe
