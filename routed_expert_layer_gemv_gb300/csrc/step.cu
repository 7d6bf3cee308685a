// Fused decode step: one launch for the whole decode step of a small batch --
// router logits, top-k and gates, permutation, LRU step, the expert FFN
// (gate/up, then down) over hits and misses, the shared expert, and the
// combine.
//
// A decode step moves each routed expert's weights once for a handful of
// tokens, so its floor is the bytes it must move (the pages' decode is bound
// by them: "FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二 "Decode"
// paragraph).  At batch 1 of the 35B-A3B-shaped layer that is ~21 MB, about
// 3 us at HBM speed, while a chain of five dependent launches costs that much
// in start-up and tails alone.  So the step runs as one persistent,
// cooperative launch, one CTA per SM, whose phases meet at grid barriers:
//
//   routing   every CTA computes the logits of its experts (8 warps split K,
//             the same arithmetic as the stand-alone router), warps 16..19
//             stage the tokens' activations for phase 1;            barrier 1
//             every CTA then recomputes the top-k, gates, permutation and the
//             hit / miss access table of the whole step from the logits (a
//             few thousand values), so no CTA waits for another to hand them
//             out; hits' buffers come from the slot table as it was before
//             the step.  CTA 0 alone runs the LRU step (state update, step
//             record) and then publishes the misses' buffers; it computes no
//             expert rows itself.
//   phase 1   gate/up units over CTAs 1..G-1 (the stand-alone GEMV's role
//             loops); an epilogue that finished arrives at barrier 2
//             while its producer already streams its phase-2 weights;
//   phase 2   down units, the activations h = SiLU(a) * u staged after
//             barrier 2 (h of every CTA is then written);         barrier 3
//   combine   y = sum_j gate_j O_j (+ shared), ascending expert, fp32 -> bf16,
//             split over every thread of the grid.
//
// Misses (fused fills) stream their weights from the pinned host pool inside
// phases 1 and 2 and are written on to the buffers CTA 0 published; hits
// need nothing from CTA 0.  The routing, the GEMV arithmetic and the combine
// are the chained path's own, so both paths give bit-identical outputs.
//
// Grid barriers: one 64-bit arrival counter per barrier that only grows; the
// host passes the count the launch starts from, each launch adds G to each,
// and every CTA arrives at every barrier exactly once, even after a timeout,
// so the counts stay aligned with the host's.  CTA 0 computes no expert rows,
// so it arrives at barriers 2 and 3 before its LRU step: the table update is
// never on the path of a step whose experts all hit.  Every wait is bounded (~2 s); a
// timeout sets the layer's error word and the CTA skips the rest of its work.
#include "gemv_dev.cuh"
#include "lru_dev.cuh"
#include "permute_dev.cuh"
#include "router_dev.cuh"
#include "step.cuh"

namespace moe {

namespace {

using namespace gv;

constexpr int kBufPending = -2;   // a miss's buffer, decided by CTA 0

// Per-CTA copy of the step's routing, in shared memory after the GEMV layout.
struct Ctl {
  int idx[kStepMaxPairs];        // [N][k] ascending expert id
  float gates[kStepMaxPairs];
  int row_of[kStepMaxPairs];
  int tok_of[kStepMaxPairs];
  int counts[kStepMaxE];
  int offs[kStepMaxE + 1];
  int so[kStepMaxE];             // slot_of before the step
  int bufm[kStepMaxE];           // slot -> buffer map before the step (S + X entries)
  int4 ent[kStepMaxPairs];       // access table: {buffer, first row, rows, first token}
  int aexp[kStepMaxPairs];       // access -> expert
  int xexp[kStepMaxTokens];      // per-token exponents of x (f16 staging)
  int sh[33];
  int n_hit, U;
  int pub_ok;                    // the misses' buffers were published in time
};

// Bounded wait (one thread) for a publication word to reach `seq` (acquire);
// false on a timeout, which sets the CTA's abort flag and the error word.
MOE_DEV bool wait_word(const unsigned long long* w, unsigned long long seq, volatile int* abort_flag, int* err) {
  const long long t0 = clock64();
  while (!*abort_flag) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(w) : "memory");
    if (v == seq) return true;
    if (clock64() - t0 > tc::kWaitCycles) {
      *abort_flag = 1;
      atomicExch(err, 1);
      return false;
    }
    __nanosleep(32);
  }
  return false;
}

// Grid barrier: arrive (one thread per CTA), then wait until all G CTAs of
// this barrier have arrived (count >= target).  Bounded.
MOE_DEV unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

MOE_DEV void gbar_arrive(unsigned long long* cnt) {
  __threadfence();
  atomicAdd(cnt, 1ull);
}
MOE_DEV bool gbar_wait(const unsigned long long* cnt, unsigned long long target, volatile int* abort_flag, int* err) {
  const long long t0 = clock64();
  while (true) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
    if (v >= target) return true;
    if (clock64() - t0 > tc::kWaitCycles) {
      *abort_flag = 1;
      atomicExch(err, 1);
      return false;
    }
    __nanosleep(32);
  }
}

template <int FMT, bool HOST>
__global__ void __launch_bounds__(kThreads, 1)
step_kernel(const __grid_constant__ CUtensorMap mg, const __grid_constant__ CUtensorMap mu,
            const __grid_constant__ CUtensorMap md, const __grid_constant__ CUtensorMap sg,
            const __grid_constant__ CUtensorMap su, const __grid_constant__ CUtensorMap sd, Geo g, GemvArgs a,
            StepArgs s, SG p1, SG p2) {
  extern __shared__ uint8_t smem_raw[];
  Smem S;
  S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  S.full = reinterpret_cast<uint64_t*>(S.base + p1.off_bar);
  S.empty = S.full + p1.D;
  S.rfull = S.empty + p1.D;
  S.rempty = S.rfull + 2;
  S.xfull = S.rempty + 2;
  S.xempty = S.xfull + 2;
  Ctl& C = *reinterpret_cast<Ctl*>(S.base + s.ctl_off);
  __shared__ Small sm;
  __shared__ float part[2][rt::kRouterWarps][kStepMaxTokens];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int N = a.N, E = g.E, k = g.k, d = g.d;
  const long long wl = a.wait_cycles > 0 ? a.wait_cycles : tc::kWaitCycles;
  unsigned long long* mark = s.trace ? s.trace + (size_t)cta * kStepMarks : nullptr;
  if (mark && tid == 0) {
    mark[11] = (unsigned long long)clock64();
    mark[0] = gtimer();
  }
  if (tid == 0) {
    for (int i = 0; i < p1.D; ++i) {
      tc::mbar_init(&S.full[i], 1);
      tc::mbar_init(&S.empty[i], kCW);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&S.rfull[i], kCW);
      tc::mbar_init(&S.rempty[i], kEW);
      tc::mbar_init(&S.xfull[i], kEW);
      tc::mbar_init(&S.xempty[i], kCW);
    }
    sm.abort = 0;
    tc::mbar_init_fence();
  }
  if (warp == kProd && lane == 0) {
    tc::prefetch_tmap(&mg);
    tc::prefetch_tmap(&mu);
    tc::prefetch_tmap(&md);
    if (p1.smode) {
      tc::prefetch_tmap(&sg);
      tc::prefetch_tmap(&su);
    }
    if (p2.smode) tc::prefetch_tmap(&sd);
  }
  // the slot table as it was before the step (the LRU CTA rewrites it only
  // after barrier 1, when every CTA has read it): loaded now, parked in
  // shared memory after the router, so the loads overlap its work
  const int so_r = tid < E ? s.slot_of[g.key0 + tid] : -1;   // E <= kThreads
  const int bm_r = tid < g.S + g.X ? s.buf[tid] : -1;        // S + X <= kThreads
  lru::LruRegs lr{};
  if (cta == 0) lr = lru::lru_load(E, g.S, g.X, g.key0, s.slot_of, s.expert_of, s.stamp, s.clock, s.buf);
  __syncthreads();

  // ---------------------------------------------------------------- routing
  // logits of this CTA's experts: warps 0..7 take expert e, warps 8..15
  // expert e + G (the stand-alone router's K split and summation order)
  const bool ALL = p1.all != 0;
  for (int eb = cta; eb < E; eb += 2 * G) {
    const int grp = warp >> 3;
    const int e = eb + grp * G;
    if (warp < 2 * rt::kRouterWarps && e < E) {
      float sum[kStepMaxTokens];
      rt::router_dot<kStepMaxTokens>(s.x, 0, N, d, s.Wr + (size_t)e * d, warp & 7, sum);
#pragma unroll
      for (int t = 0; t < kStepMaxTokens; ++t)
        if (lane == 0) part[grp][warp & 7][t] = sum[t];
    } else if (warp >= 2 * rt::kRouterWarps && eb == cta) {
      // warps 16..19: the tokens' exponents (f16 staging of x)
      for (int t = warp - 2 * rt::kRouterWarps; t < N; t += 4) {
        const int se = rt::token_exp(s.x + (size_t)t * d, d);
        if (lane == 0) C.xexp[t] = se;
      }
    }
    __syncthreads();
    for (int q = tid; q < 2 * N; q += kThreads) {
      const int grp = q / N, t = q % N;
      const int e2 = eb + grp * G;
      if (e2 < E)
        s.logits[(size_t)t * E + e2] =
            rt::logit_from_parts(&part[grp][0][t], kStepMaxTokens, s.bias ? s.bias[e2] : 0.f);
    }
    __syncthreads();
  }
  if (cta >= E && warp >= 2 * rt::kRouterWarps) {
    // CTAs without an expert still compute the exponents
    for (int t = warp - 2 * rt::kRouterWarps; t < N; t += 4) {
      const int se = rt::token_exp(s.x + (size_t)t * d, d);
      if (lane == 0) C.xexp[t] = se;
    }
  }
  if (tid < E) C.so[tid] = so_r;
  if (tid < g.S + g.X) C.bufm[tid] = bm_r;
  __syncthreads();
  const unsigned long long target = s.gbar_base + (unsigned long long)G;   // of each barrier
  if (tid == 0) {
    if (mark) mark[1] = gtimer();
    gbar_arrive(s.gbar + 0);
    gbar_wait(s.gbar + 0, target, &sm.abort, a.err);
    if (mark) mark[2] = gtimer();
  }
  __syncwarp();   // lane 0 waited alone: the warp runs the top-k below converged
  __syncthreads();
  const bool routed = !sm.abort;

  // every CTA: top-k and gates of every token (warps 0..15, one token each;
  // the logits row is staged in the ring area, which no copy uses yet) while
  // warps 16..19 stage every token (N <= 8) for phase 1
  if (routed) {
    if (warp < 2 * rt::kRouterWarps) {
      float* Ls = reinterpret_cast<float*>(S.base) + (size_t)warp * E;
      for (int t = warp; t < N; t += 2 * rt::kRouterWarps) {
        rt::stage_logits(s.logits, t, E, Ls);
        rt::topk_row(Ls, E, k, g.norm_topk, C.idx + t * k, C.gates + t * k);
        __syncwarp();
      }
    } else if (ALL) {
      stage_all<FMT>(p1, N, s.x, reinterpret_cast<uint2*>(S.base + p1.off_x), &sm.sexp[0][0],
                     tid - 2 * rt::kRouterWarps * 32, 128, 3);
    }
  }
  __syncthreads();
  if (mark && tid == 0) mark[3] = gtimer();
  // permutation: counts, offsets, rows in ascending token order per expert
  int cnt = 0;
  if (routed && tid < E)
    for (int q = 0; q < N * k; ++q) cnt += C.idx[q] == tid ? 1 : 0;
  int total;
  const int off = perm::block_excl_scan(tid < E ? cnt : 0, &total, C.sh);
  if (tid < E) {
    C.counts[tid] = cnt;
    C.offs[tid] = off;
  }
  if (tid == 0) C.offs[E] = total;
  __syncthreads();
  if (routed && tid < N * k) {
    const int t = tid / k, e = C.idx[tid];
    int r = C.offs[e];
    for (int t2 = 0; t2 < t; ++t2)
      for (int j = 0; j < k; ++j)
        if (C.idx[t2 * k + j] == e) {
          ++r;
          break;
        }
    C.row_of[tid] = r;
    C.tok_of[r] = t;
  }
  __syncthreads();
  if (mark && tid == 0) mark[4] = gtimer();
  // access table: hits ascending id, then misses ascending id
  {
    const bool inU = routed && tid < E && cnt > 0;
    const int cur = tid < E ? C.so[tid] : -1;
    const bool hit = inU && cur >= 0 && cur < g.S, miss = inU && !hit;
    int tot2;
    const int pre = perm::block_excl_scan((hit ? 1 : 0) | (miss ? 1 << 16 : 0), &tot2, C.sh);
    const int n_hit = tot2 & 0xffff, U = (tot2 & 0xffff) + (tot2 >> 16);
    if (inU) {
      const int i = hit ? (pre & 0xffff) : n_hit + (pre >> 16);
      C.aexp[i] = tid;
      C.ent[i] = make_int4(hit ? C.bufm[cur] : kBufPending, off, cnt, C.tok_of[off] & 0xffff);
    }
    if (tid == 0) {
      C.n_hit = n_hit;
      C.U = routed ? U : 0;
    }
  }
  __syncthreads();
  if (mark && tid == 0) mark[5] = gtimer();
  const bool lru_cta = cta == 0 && routed;   // arrives at barriers 2 and 3 below, before the LRU step
  if (lru_cta) {
    // the layer's copy of the routing (what moe_debug_last_step returns)
    for (int q = tid; q < N * k; q += kThreads) {
      s.idx[q] = C.idx[q];
      s.gates[q] = C.gates[q];
      s.row_of[q] = C.row_of[q];
      s.tok_of[q] = C.tok_of[q];
    }
    for (int e = tid; e < E; e += kThreads) {
      s.counts[e] = C.counts[e];
      s.offsets[e] = C.offs[e];
    }
    if (tid == 0) {
      s.offsets[E] = C.offs[E];
      // no expert rows here: barriers 2 and 3 need nothing more from this CTA
      gbar_arrive(s.gbar + 1);
      gbar_arrive(s.gbar + 2);
    }
    // the LRU step (its shared state in the ring area, after the top-k rows)
    lru::LruSmem& m = *reinterpret_cast<lru::LruSmem*>(S.base);
    lru::lru_park(lr, E, g.S, g.X, m);
    __syncthreads();
    lru::lru_body<kThreads>(C.counts, C.offs, nullptr, E, g.S, g.X, g.key0, g.keys, s.slot_of, s.expert_of, s.stamp, s.clock,
                            s.buf, s.rec, s.stats, nullptr, 0ull, m);
    __syncthreads();
    if (tid == 0) {
      // the misses' buffers (rec_buf) are final: publish them
      __threadfence();
      asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(s.ready), "l"(s.seq) : "memory");
    }
  }

  // ---------------------------------------------------------------- expert FFN
  EntryTable T{};
  T.ent = C.ent;
  T.expert = C.aexp;
  T.base = 0;
  T.nr = C.U;
  T.n_hit = C.n_hit;
  T.shared = g.has_shared && routed ? 1 : 0;
  GemvArgs ga = a;
  ga.tok_of = C.tok_of;          // this CTA's copies (generic pointers into shared memory)
  ga.offsets = C.offs;
  Range r1{0, 0}, r2{0, 0};
  if (cta > 0) {
    r1 = cta_range(T, p1, cta - 1, G - 1);
    r2 = cta_range(T, p2, cta - 1, G - 1);
  }
  // misses in this CTA's ranges: their buffers once CTA 0 has published them
  // (resolved here, once for the CTA, so every role then reads the same table)
  {
    auto touches = [&](const Range& r, int UE) {
      return r.u1 > r.u0 && (r.u1 - 1) / UE >= T.n_hit && r.u0 / UE < T.nr;
    };
    const bool need = T.n_hit < T.nr && (touches(r1, p1.UE) || touches(r2, p2.UE));
    if (need) {
      if (tid == 0) C.pub_ok = wait_word(s.ready, s.seq, &sm.abort, a.err) ? 1 : 0;
      __syncthreads();
      const int* pub = rec_buf(s.rec, E);
      for (int i = T.n_hit + tid; i < T.nr; i += kThreads) C.ent[i].x = C.pub_ok ? __ldcg(pub + i) : -1;
      __syncthreads();
    }
  }
  bool first_staged = false;
  if (!ALL && warp != kProd) {
    Cursor c0;
    cursor_init(c0, r1);
    if (cursor_next(c0, g, ga, T, p1, r1)) {
      const int t2 = warp < kCW ? tid : tid - 32;
      stage_block<FMT, 1>(g, ga, p1, c0.en, c0.tg, reinterpret_cast<uint2*>(S.base + p1.off_x), sm.sexp[0], sm.stok,
                          s.x, C.xexp, s.h, t2, kThreads - 32, 2);
      asm volatile("bar.sync 2, %0;" :: "n"(kThreads - 32) : "memory");
      if (warp > kCW && lane == 0) mbar_arrive(&S.xfull[0]);
      first_staged = true;
    }
  }
  Ring ring;
  if (warp == kProd) {
    // the producer runs straight on from phase 1's weights into phase 2's
    produce<FMT, 1, HOST>(g, ga, p1, T, r1, S, sm, ring, &mg, &mu, &sg, &su, wl);
    produce<FMT, 2, HOST>(g, ga, p2, T, r2, S, sm, ring, &md, &md, &sd, &sd, wl);
    produce_drain(S, p1.D, ring, a.err);
  } else if (warp < kCW) {
    compute<FMT, 1, HOST>(g, ga, p1, T, r1, S, sm, ring, wl, mark ? mark + 13 : nullptr);
    compute<FMT, 2, HOST>(g, ga, p2, T, r2, S, sm, ring, wl, mark ? mark + 15 : nullptr);
  } else {
    reduce<FMT, 1, HOST>(g, ga, p1, T, r1, S, sm, ring, first_staged, s.x, C.xexp, s.h, s.O, wl);
    // this CTA's h rows are written: barrier 2, then phase 2 stages h of any CTA
    epi_sync();
    if (warp == kCW + 1 && lane == 0) {
      if (mark) mark[6] = gtimer();
      if (!lru_cta) gbar_arrive(s.gbar + 1);
      gbar_wait(s.gbar + 1, target, &sm.abort, a.err);
      if (mark) mark[7] = gtimer();
    }
    __syncwarp();
    epi_sync();
    reduce<FMT, 2, HOST>(g, ga, p2, T, r2, S, sm, ring, false, s.x, C.xexp, s.h, s.O, wl, mark ? mark + 17 : nullptr);
    epi_sync();
    if (warp == kCW + 1 && lane == 0) {
      if (mark) mark[8] = gtimer();
      if (!lru_cta) gbar_arrive(s.gbar + 2);
    }
  }
  __syncthreads();
  if (tid == 0) {
    gbar_wait(s.gbar + 2, target, &sm.abort, a.err);
    if (mark) mark[9] = gtimer();
  }
  __syncwarp();
  __syncthreads();

  // ---------------------------------------------------------------- combine
  // the chained path's combine: per output 4 columns, ascending j, fp32
  if (!sm.abort) {
    const int q = d / 4;
    const int rows = N * k;
    for (int v = cta * kThreads + tid; v < N * q; v += G * kThreads) {
      const int t = v / q, cv = v % q;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; ++j) {
        const float gj = C.gates[t * k + j];
        const int r = C.row_of[t * k + j];
        if (r < 0 || r >= rows) continue;
        const float4 o = __ldcg(reinterpret_cast<const float4*>(s.O + (size_t)r * d) + cv);
        acc[0] = fmaf(gj, o.x, acc[0]);
        acc[1] = fmaf(gj, o.y, acc[1]);
        acc[2] = fmaf(gj, o.z, acc[2]);
        acc[3] = fmaf(gj, o.w, acc[3]);
      }
      if (g.has_shared) {
        const float4 o = __ldcg(reinterpret_cast<const float4*>(s.O + (size_t)(rows + t) * d) + cv);
        acc[0] += o.x;
        acc[1] += o.y;
        acc[2] += o.z;
        acc[3] += o.w;
      }
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
      const __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
      reinterpret_cast<uint2*>(s.y + (size_t)t * d)[cv] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
    }
  }
  if (mark) {
    __syncthreads();
    if (tid == 0) {
      mark[10] = gtimer();
      mark[12] = (unsigned long long)clock64();
    }
  }
}

}  // namespace

bool step_plan(const Geo& g, int N, StepPlan* out) {
  StepPlan P{};
  if (N < 1 || N > kStepMaxTokens || g.E > kStepMaxE || (long long)N * g.k > kStepMaxPairs) return false;
  if (g.S + g.X > kThreads) return false;   // the LRU step: one slot per thread of CTA 0
  if (g.d % (rt::kRouterWarps * 16) || g.d > 8192 || g.f > 8192 || g.d % 128 || g.f % 128) return false;
  SG a = make_sg(g, 1, N), b = make_sg(g, 2, N);
  a.all = N <= kTG ? 1 : 0;
  a.XB = a.all ? 1 : 2;
  b.all = 0;
  b.XB = 2;
  a.xbytes = a.K * 2 * kTG;
  b.xbytes = b.K * 2 * kTG;
  const int xregion = std::max(a.XB * a.xbytes, b.XB * b.xbytes);
  const int stage = std::max(a.stage_bytes, b.stage_bytes);
  const int bars = 2 * kMaxD * 8 + 8 * 8;
  const int red = 2 * a.rbytes;
  // dynamic shared memory: 1 KB alignment slack, the GEMV layout, the routing copy
  const int budget = kStepSmemMax - 1024 - (int)sizeof(Ctl) - 16;
  const int D = std::min(kMaxD, (budget - xregion - red - bars) / stage);
  if (D < 2) return false;
  for (SG* q : {&a, &b}) {
    q->stage_bytes = stage;
    q->D = D;
    q->RS = 2;
    q->off_x = D * stage;
    q->off_red = q->off_x + xregion;
    q->off_bar = q->off_red + red;
    q->smem = 1024 + q->off_bar + bars;
  }
  // the routing scratch (a logits row per warp) and the LRU CTA's state live
  // in the ring area before any copy starts
  const size_t ring_bytes = (size_t)D * stage;
  if ((size_t)(2 * rt::kRouterWarps) * g.E * 4 > ring_bytes || sizeof(lru::LruSmem) > ring_bytes) return false;
  P.p1 = a;
  P.p2 = b;
  P.ctl_off = (a.off_bar + bars + 15) & ~15;
  P.smem = 1024 + P.ctl_off + (int)sizeof(Ctl);
  if (P.smem > kStepSmemMax) return false;
  *out = P;
  return true;
}

cudaError_t launch_step(const Geo& g, const GemvPlan* pl, const GemvArgs& a, StepArgs s, const StepPlan& P,
                        int grid, cudaStream_t st) {
  s.ctl_off = P.ctl_off;
  const bool host = a.host_pool != nullptr;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const CUtensorMap, Geo, GemvArgs, StepArgs, SG, SG);
  if (g.fmt == MOE_MXFP4) kern = host ? step_kernel<MOE_MXFP4, true> : step_kernel<MOE_MXFP4, false>;
  else if (g.fmt == MOE_NVFP4) kern = host ? step_kernel<MOE_NVFP4, true> : step_kernel<MOE_NVFP4, false>;
  else if (g.fmt == MOE_MXFP8) kern = host ? step_kernel<MOE_MXFP8, true> : step_kernel<MOE_MXFP8, false>;
  else kern = host ? step_kernel<MOE_BF16, true> : step_kernel<MOE_BF16, false>;
  cudaError_t e = ensure_smem_limit((const void*)kern, P.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident at once: the grid barriers need it
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, pl->w[0], pl->w[1], pl->w[2], pl->s[0], pl->s[1], pl->s[2], g, a, s, P.p1,
                            P.p2);
}

}  // namespace moe
