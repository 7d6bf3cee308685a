// Device pieces of the per-step LRU slot table, shared by the LRU kernels
// (one CTA of 1024 threads) and the fused decode step (whose routing CTA has
// fewer threads): the table's state parked in shared memory and one step of it.
//
// FreeToken keeps the routed experts in a global LRU expert cache in GPU
// memory; hits are served from it and misses are loaded into it from host
// memory ("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二, "Decode" and
// "LRU 为什么赢" paragraphs).  The pages leave the per-step order open; this
// table takes the step's distinct experts U as accesses, hits first (ascending
// id) then misses (ascending id).  A hit becomes most recently used; a miss
// takes the lowest free slot, else evicts the least recently used expert.
// The closed form used by lru_body is described at the top of lru.cu.
#pragma once
#include "common.cuh"
#include "permute_dev.cuh"

namespace moe {
namespace lru {


// Exclusive scan of a 64-bit value over the NT threads of the CTA (NT a
// multiple of 32, at most 1024; three counters packed in 21-bit fields scan
// at once); *total gets the sum.
template <int NT>
MOE_DEV unsigned long long excl_scan_u64(unsigned long long v, unsigned long long* total,
                                         unsigned long long* sh) {
  constexpr int kNW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long s = lane < kNW ? sh[lane] : 0ull;
    unsigned long long si = s;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    if (lane < kNW) sh[lane] = si - s;
    if (lane == 31) sh[32] = si;
  }
  __syncthreads();
  const unsigned long long r = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

// Shared-memory scratch of one LRU step.
struct LruSmem {
  int sh[33];
  unsigned long long sh64[33];
  unsigned long long clk;         // clock, staged
  int so[kMaxE];       // slot_of, staged
  int q[kMaxE];        // victim queue (slots)
  int q_old[kMaxE];    // expert that held q[i] before the step (-1 free)
  int acc_e[kMaxE], acc_s[kMaxE];
  int eo[kMaxE];       // expert_of, staged
  int buf[kMaxE];      // slot -> buffer map and spare buffers, staged
  unsigned long long st[kMaxE];   // stamps, staged
  unsigned char stale[kMaxE];     // occupied by an expert not routed this step
};

// The table's state, read once per step: every thread issues its loads
// together (one memory round trip) and parks them in shared memory; callers
// put other independent loads between lru_load and lru_park.  slot_of is
// indexed by key; the layer's experts are keys key0 .. key0 + E - 1.
struct LruRegs {
  int so, eo, buf;
  unsigned long long st, clk;
};
MOE_DEV LruRegs lru_load(int E, int S, int X, int key0, const int* __restrict__ slot_of,
                         const int* __restrict__ expert_of, const unsigned long long* __restrict__ stamp,
                         const unsigned long long* __restrict__ clock, const int* __restrict__ buf) {
  const int t = threadIdx.x;
  LruRegs r;
  r.so = t < E ? slot_of[key0 + t] : -1;
  r.eo = t < S ? expert_of[t] : -1;
  r.buf = t < S + X ? buf[t] : -1;
  r.st = t < S ? stamp[t] : 0ull;
  r.clk = t == 0 ? *clock : 0ull;
  return r;
}
MOE_DEV void lru_park(const LruRegs& r, int E, int S, int X, LruSmem& m) {
  const int t = threadIdx.x;
  if (t < E) m.so[t] = r.so;
  if (t < S) { m.eo[t] = r.eo; m.st[t] = r.st; }
  if (t < S + X) m.buf[t] = r.buf;
  if (t == 0) m.clk = r.clk;
}

// One step of the table (blockDim.x == NT, E <= NT, S + X <= NT) on the
// state parked in m (the caller synchronises after lru_park).  counts may
// live in shared or global memory.  The layer's expert e is key key0 + e of
// a table of `keys` keys (slot_of [keys], expert_of holds keys); the record
// names the layer's experts (e) and, as evicted, keys.
template <int NT>
MOE_DEV void lru_body(const int* counts, const int* offs, const uint32_t* cm, int E, int S, int X,
                      int key0, int keys, int* __restrict__ slot_of,
                      int* __restrict__ expert_of, unsigned long long* __restrict__ stamp,
                      unsigned long long* __restrict__ clock, int* __restrict__ buf, StepRecord* __restrict__ rec,
                      unsigned long long* __restrict__ stats, StepRecord* host_rec, unsigned long long seq,
                      LruSmem& m) {
  const int tid = threadIdx.x;
  const unsigned long long clk = m.clk;

  // hits / misses over experts (E <= NT: one expert per thread) and the
  // free / stale slots (S <= NT: one slot per thread), counted by one scan of
  // three packed 21-bit counters
  const int e = tid;
  const bool inU = e < E && counts[e] > 0;
  const int cur = e < E ? m.so[e] : -1;
  const bool hit = inU && cur >= 0, miss = inU && cur < 0;
  const int s = tid;
  int old = -1;
  bool fre = false, stale = false;
  unsigned long long st = 0;
  if (s < S) {
    old = m.eo[s];
    fre = old < 0 || old >= keys;
    // another layer's key, or this layer's expert routed to no token
    stale = !fre && (old < key0 || old >= key0 + E || counts[old - key0] == 0);
    st = m.st[s];
    m.stale[s] = stale ? 1 : 0;
  }
  constexpr unsigned long long kF = 0x1FFFFFull;
  unsigned long long tot;
  const unsigned long long pre = excl_scan_u64<NT>(
      (hit ? 1ull : 0ull) | (miss ? 1ull << 21 : 0ull) | (fre ? 1ull << 42 : 0ull), &tot, m.sh64);
  const int hr = (int)(pre & kF), mr = (int)((pre >> 21) & kF), fr = (int)((pre >> 42) & kF);
  const int n_hit = (int)(tot & kF), n_miss = (int)((tot >> 21) & kF), n_free = (int)((tot >> 42) & kF);
  const int U = n_hit + n_miss;

  // victim queue Q (its barriers published m.stale): free slots, then stale
  // slots by ascending stamp; hits keep their slots.  The step reads only
  // Q[0 .. min(U, S) - n_hit): a stale slot needs its exact rank only while
  // that rank is below the n_need stale victims, so it stops counting there
  // (a pool of hundreds of slots and a handful of misses scans a few entries
  // per slot, not all of them)
  if (fre) { m.q[fr] = s; m.q_old[fr] = -1; }
  const int n_need = max(0, min(U, S) - n_hit - n_free);
  if (stale && n_need > 0) {
    int r = 0;
    for (int s2 = 0; s2 < S && r < n_need; ++s2) {
      if (!m.stale[s2]) continue;
      const unsigned long long t2 = m.st[s2];
      r += (t2 < st || (t2 == st && s2 < s)) ? 1 : 0;
    }
    if (r < n_need) {
      m.q[n_free + r] = s;
      m.q_old[n_free + r] = old;
    }
  }
  if (hit) { m.acc_e[hr] = e; m.acc_s[hr] = cur; }
  __syncthreads();

  // misses of the first wave take Q in order; later waves reuse slot(i - S)
  if (miss) {
    const int i = n_hit + mr;
    m.acc_e[i] = e;
    if (i < S) m.acc_s[i] = m.q[i - n_hit];   // i - n_hit < S - n_hit = |Q|
  }
  __syncthreads();
  if (U > S) {
    for (int i = S + tid; i < U; i += NT) m.acc_s[i] = m.acc_s[i % S];
    __syncthreads();
  }

  int* r_e = rec_expert(rec);
  int* r_s = rec_slot(rec, E);
  int* r_v = rec_evicted(rec, E);
  int* r_b = rec_buf(rec, E);
  int4* r_n = rec_entry(rec, E);
  for (int i = tid; i < U; i += NT) {
    const int ex = m.acc_e[i], sl = m.acc_s[i];
    r_e[i] = ex;
    r_s[i] = sl;
    int ev = -1;   // a key
    if (i >= S) ev = key0 + m.acc_e[i - S];
    else if (i >= n_hit) ev = m.q_old[i - n_hit];
    r_v[i] = ev;
    // buffer: the LRU slot's, or spare i - S for later waves
    const bool ok = ex >= 0 && ex < E && sl >= 0 && sl < S && i - S < X;
    const int ps = !ok ? -1 : i < S ? m.buf[sl] : m.buf[S + (i - S)];
    r_b[i] = ps;
    const int row0 = offs && ok ? offs[ex] : 0, nrow = offs && ok ? counts[ex] : 0;
    // first token of the access, from the per-warp token ballots of its
    // expert (tokens 32 w + lane); unknown without them
    uint32_t toks = 0xffff0000u;
    if (cm && ok && nrow > 0) {
      int t0 = -1;
      for (int w = 0; w < perm::kPermWarps && t0 < 0; ++w) {
        const uint32_t b = cm[ex * perm::kPermWarps + w];
        if (b) t0 = 32 * w + __ffs(b) - 1;
      }
      toks = (uint32_t)t0 & 0xffffu;
    }
    r_n[i] = make_int4(ps, row0, nrow, (int)toks);
    if (host_rec) {
      rec_expert(host_rec)[i] = ex;
      rec_slot(host_rec, E)[i] = sl;
      rec_evicted(host_rec, E)[i] = ev;
      rec_buf(host_rec, E)[i] = ps;
    }
  }
  if (host_rec) {
    // the host polls seq: every writer's stores reach the system before it
    if (tid == 0) {
      host_rec->U = U;
      host_rec->n_hit = n_hit;
      host_rec->n_miss = n_miss;
      host_rec->S = S;
    }
    // each writer's fence completes before the barrier, so seq is stored
    // after every other field is visible to the host
    if (tid < U || tid == 0) __threadfence_system();
    __syncthreads();
    if (tid == 0) *reinterpret_cast<volatile unsigned long long*>(&host_rec->seq) = seq;
  }
  if (tid == 0) {
    rec->U = U;
    rec->n_hit = n_hit;
    rec->n_miss = n_miss;
    rec->S = S;
  }
  // table update: experts pushed out of Q lose their slot (they are not in
  // U, so these writes never meet the assignments below)
  for (int i = n_hit + tid; i < min(U, S); i += NT) {
    const int ev = m.q_old[i - n_hit];
    if (ev >= 0 && ev < keys) slot_of[ev] = -1;
  }
  for (int i = tid; i < U; i += NT) {
    const int ex = m.acc_e[i], sl = m.acc_s[i];
    if (sl < 0 || sl >= S || ex < 0 || ex >= E) continue;   // only a corrupted table gets here
    if (i + S < U) {
      slot_of[key0 + ex] = -1;     // evicted later in this same step
    } else {
      slot_of[key0 + ex] = sl;
      expert_of[sl] = key0 + ex;
      stamp[sl] = clk + 1ull + (unsigned long long)i;
    }
  }
  // a later-wave miss that keeps its slot takes over the spare buffer it was
  // filled into, and the slot's old buffer becomes that spare (the slots and
  // spares of these accesses are all distinct)
  __syncthreads();   // every read of m.buf above is done
  for (int i = max(S, U - S) + tid; i < U; i += NT) {
    const int sl = m.acc_s[i], j = S + (i - S);
    if (sl < 0 || sl >= S || i - S >= X) continue;
    const int t = m.buf[sl];
    m.buf[sl] = m.buf[j];
    m.buf[j] = t;
  }
  __syncthreads();
  if (U > S && tid < S + X) buf[tid] = m.buf[tid];
  if (tid == 0) {
    *clock = clk + (unsigned long long)U;
    if (stats) {   // fire-and-forget adds: no round trip
      atomicAdd(stats + 0, 1ull);
      atomicAdd(stats + 1, (unsigned long long)U);
      atomicAdd(stats + 2, (unsigned long long)n_hit);
      atomicAdd(stats + 3, (unsigned long long)n_miss);
    }
  }
}

}  // namespace lru
}  // namespace moe
