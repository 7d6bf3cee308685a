// Decode expert FFN: a persistent, warp-specialised grouped GEMV over the
// experts of one work range, weights read through the slot table and
// dequantised in registers.
//
// Decode moves each routed expert's weights once per step for a handful of
// tokens, so the kernel is bound by HBM bandwidth (the pages' decode is bound
// by the bytes each step must move: "FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).  Design:
//  * work unit = one expert entry x one matrix x a 64-row block (all of K);
//    one CTA per SM, persistent, each taking an equal contiguous range of
//    the launch's units, so every SM streams from the first cycle;
//  * three roles that only meet at mbarriers, so loads, math and reductions
//    overlap and no warp waits for a CTA-wide barrier:
//    - a producer warp streams the unit's codes as TMA boxes of 64 rows x
//      256 K (128 bytes per row, 128-byte swizzle), four boxes per stage,
//      plus their scale bytes (one more TMA box, or one bulk copy), into a
//      ring of shared-memory stages; tall boxes and a handful of copy
//      instructions per 32 KB keep the copy engine near the HBM rate;
//    - 16 compute warps: warp (b, q) takes the 16-row quarter q of box b of
//      every stage, so a unit's K splits four ways and each warp accumulates
//      its share across the unit's stages;
//    - 3 epilogue warps stage the next token group's activations and add the
//      four partial sums of each output in a fixed order (deterministic);
//  * the token dimension goes through tensor-core MMAs (mma.sync m16n8k16,
//    f16 x f16 -> f32): a lane's 32-bit word of codes becomes four f16x2 A
//    registers with cvt.rn.f16x2.e2m1x2 (exact); the activations are staged
//    once per token group as f16 (power-of-two scaled per token so nothing
//    overflows) in B-fragment order, so each B load is one contiguous 256-byte
//    warp access; each MMA stays inside one scale block, whose scale is
//    applied to the MMA sum in fp32; the swizzle makes the A loads
//    conflict-free.
// Phase 1: a = W_g x and u = W_u x (separate units), fp32 [rows, 2 d_ff].
// Phase 2: O = W_d h with h = SiLU(a) * u formed while staging, fp32 [rows, d_model].
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace moe {

struct GemvPlan {
  CUtensorMap w[3];   // gate, up, down codes of all slots (+ the shared expert)
  CUtensorMap s[3];   // their scale bytes (used when a scale row is a 16-byte multiple)
  bool ready;
};

namespace {

constexpr int kCW = 16;                      // compute warps
constexpr int kEW = 3;                       // epilogue warps
constexpr int kProd = kCW;                   // producer warp index
constexpr int kThreads = (kCW + 1 + kEW) * 32;
constexpr int kET = kEW * 32;                // epilogue threads
constexpr int kTG = 8;                       // tokens per group (one MMA N)
constexpr int kBoxRows = 64;
constexpr int kBoxK = 256;                   // codes per box row (128 bytes)
constexpr int kBoxBytes = kBoxRows * kBoxK / 2;
constexpr int kBoxes = 4;                    // boxes per stage
constexpr int kMaxD = 8;                     // ring stages at most
constexpr int kSmemBudget = 220 * 1024;

// Geometry of one phase (host-computed, passed by value).
struct SG {
  int K, R;           // reduction length, output rows per matrix
  int KB;             // 256-K boxes per row (the last one may be half valid)
  int NS;             // stages per unit
  int RB;             // 64-row blocks per matrix
  int UE;             // units per entry (RB per matrix, gate and up separately in phase 1)
  int SBB;            // scale bytes per box row (8 MXFP4, 16 NVFP4)
  int smode;          // 1: a TMA box of the stage's scales; 0: the unit's whole scale rows
  int srow;           // staged scale bytes per row (4 * SBB, or scale_row)
  int codes_bytes;    // kBoxes code boxes
  int stage_bytes, D;
  int XB, xbytes;     // activation buffers and bytes of one
  int RS, rbytes;     // partial-sum slots and bytes of one
  int off_x, off_red, off_bar, smem;
  int scale_row;      // scale bytes per weight row
  int all;            // phase 1, N <= 8: every token staged once, entries pick theirs
};

MOE_DEV float pow2i(int s) { return __int_as_float((127 + s) << 23); }  // |s| <= 126

MOE_DEV uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Contiguous global -> shared copy by the bulk-copy engine (16-byte aligned
// addresses, size a multiple of 16), completing on `bar`.
MOE_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(tc::su32(dst)), "l"(src), "r"(bytes), "r"(tc::su32(bar)) : "memory");
}
MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::su32(bar)) : "memory");
}
// Barrier of the epilogue warps only.
MOE_DEV void epi_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kET) : "memory"); }

// Four E2M1 pairs (one word, low nibble = even K) -> four f16x2, exact.
MOE_DEV void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// E8M0 byte (J & 3) of a scale word -> 2^(x-127) (x = 0 gives 2^-127 as the
// format defines; x = 255 gives +inf).
template <int J>
MOE_DEV float e8m0_byte(uint32_t w) {
  constexpr int b = J & 3;
  const uint32_t v = b < 3 ? (w << (23 - 8 * b)) & 0x7F800000u : (w >> 1) & 0x7F800000u;
  return __uint_as_float(max(v, 0x00400000u));
}

MOE_DEV void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y), "f"(0.0f));
}

MOE_DEV void mma16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

struct Entry {
  int slot, row0, nrows, shared;
  int tok0;        // token of the first row (-1: read tok_of)
  int ex;          // a miss read from the host pool (and written on to `slot`): its expert; else -1
};

// Entries of this launch: the access-order range the mode selects (+ the
// shared expert).  *base = first access index, *nr = routed entries.
MOE_DEV int count_entries(const Geo& g, const GemvArgs& a, int* base, int* nr) {
  const StepRecord* rec = a.rec;
  const int U = min(max(rec->U, 0), g.E), nh = min(max(rec->n_hit, 0), U), S = g.S;
  (void)S;
  int b = 0, e = nh;
  if (a.mode == kRangeAll) {
    e = U;
  } else if (a.mode != kRangeHits) {
    // misses [nh, U), or chunk `chunk` of n_chunks of them
    const int C = max(a.n_chunks, 1), c = min(max(a.chunk, 0), C - 1);
    int lo, hi;
    miss_chunk(U - nh, c, C, &lo, &hi);
    b = nh + lo;
    e = nh + hi;
  }
  *base = b;
  *nr = max(0, e - b);
  return *nr + (a.with_shared ? 1 : 0);
}

MOE_DEV bool get_entry(const Geo& g, const GemvArgs& a, int base, int nr, int ent, Entry& out) {
  if (ent < nr) {
    // one 16-byte load: physical slot, first row, rows (the LRU step wrote it)
    const int4 v = rec_entry(const_cast<StepRecord*>(a.rec), g.E)[base + ent];
    const bool slot_ok = (v.x >= 0 && v.x < g.S) || (v.x > g.S && v.x <= g.S + g.X);
    out.slot = v.x;
    out.row0 = v.y;
    out.nrows = v.z;
    out.shared = 0;
    const uint32_t tk = (uint32_t)v.w;
    out.tok0 = (tk >> 16) == 0xffffu ? -1 : (int)(tk & 0xffffu);
    out.ex = -1;
    if (a.host_pool && base + ent >= min(max(a.rec->n_hit, 0), g.E)) {
      out.ex = rec_expert(const_cast<StepRecord*>(a.rec))[base + ent];
      if (out.ex < 0 || out.ex >= g.E) return false;
    }
    return slot_ok && out.nrows > 0 && out.row0 >= 0 && out.row0 + out.nrows <= a.N * g.k;
  }
  if (a.with_shared && ent == nr) {
    out.slot = g.S;
    out.row0 = a.N * g.k;
    out.nrows = a.N;
    out.shared = 1;
    out.tok0 = 0;
    out.ex = -1;
    return a.N > 0;
  }
  return false;
}

// This CTA's unit range [u0, u1) of the launch's n_ent * UE units.  (A launch
// that streams misses from the host pool keeps them in a contiguous run of
// CTAs: spreading them over every CTA measured slower on the host link.)
struct Range {
  int base, nr, u0, u1;
};

MOE_DEV Range cta_range(const Geo& g, const GemvArgs& a, const SG& p) {
  Range r;
  const int n_ent = count_entries(g, a, &r.base, &r.nr);
  const long long T = (long long)n_ent * p.UE;
  r.u0 = (int)(T * blockIdx.x / gridDim.x);
  r.u1 = (int)(T * (blockIdx.x + 1) / gridDim.x);
  return r;
}

// Walks the CTA's blocks (entry segment x token group of 8) in the order
// every role uses: for each entry segment of the range, for each token
// group; the block's units are ue0 .. ue1 - 1.
struct Cursor {
  int t, ue0, ue1, tg, ntg;
  Entry en;
};

MOE_DEV void cursor_init(Cursor& c, const Range& rr) {
  c.t = rr.u0;
  c.tg = 0;
  c.ntg = 0;
}

MOE_DEV bool cursor_next(Cursor& c, const Geo& g, const GemvArgs& a, const SG& p, const Range& rr) {
  if (c.tg + 1 < c.ntg) {
    ++c.tg;
    return true;
  }
  while (c.t < rr.u1) {
    const int ent = c.t / p.UE;
    c.ue0 = c.t % p.UE;
    c.ue1 = min(p.UE, c.ue0 + (rr.u1 - c.t));
    c.t += c.ue1 - c.ue0;
    if (get_entry(g, a, rr.base, rr.nr, ent, c.en)) {
      c.tg = 0;
      c.ntg = p.all ? 1 : (c.en.nrows + kTG - 1) / kTG;
      return true;
    }
  }
  c.ntg = 0;
  return false;
}

// Staged activation slot (in 8-byte units) of token t, K = 4 k4 .. 4 k4 + 3:
// B-fragment order [32-K block][MMA step][lane = 4 t + q].  MXFP4 steps take
// K 32J + 8q + 4s .. + 3, NVFP4 steps (one 16-block each) 32J + 16s + 4q ...
MOE_DEV int xslot(int fmt, int t, int k4) {
  const int J = k4 >> 3, i = k4 & 7;
  const int s = fmt == MOE_MXFP4 ? (i & 1) : (i >> 2);
  const int q = fmt == MOE_MXFP4 ? (i >> 1) : (i & 3);
  return (J * 2 + s) * 32 + 4 * t + q;
}

// One warp's 16 x 256 MXFP4 tile: acc += W x.  Codes: 128-byte rows, 16-byte
// chunk j of row r stored at chunk j ^ (r & 7) (128-byte swizzle).  Lane
// (g = lane / 4, q = lane % 4) takes word q of chunk j (codes 8q..8q+7 of
// block j) of rows g and g + 8; MMA step s uses codes 8q + 4s .. + 3.
// Blocks j >= nvb lie past K and are skipped.
MOE_DEV void tile_mx(const uint8_t* cs, const uint8_t* s0p, const uint8_t* s1p, const uint2* xb, int nvb,
                     int lane, float (&acc)[4]) {
  const int g = lane >> 2, q = lane & 3;
  // scale rows are only 4-byte aligned when a whole unit's rows are staged
  const uint2 sc0 = make_uint2(lds32(s0p), lds32(s0p + 4)), sc1 = make_uint2(lds32(s1p), lds32(s1p + 4));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nvb) {
      const uint2 b0 = xb[(2 * j) * 32 + lane], b1 = xb[(2 * j + 1) * 32 + lane];
      const int co = ((j ^ g) << 4) + 4 * q;
      uint32_t f0[4], f1[4];
      e2m1x8_to_f16x8(lds32(cs + 128 * g + co), f0);
      e2m1x8_to_f16x8(lds32(cs + 128 * (g + 8) + co), f1);
      const uint32_t w0 = j < 4 ? sc0.x : sc0.y, w1 = j < 4 ? sc1.x : sc1.y;
      float sg, sg8;
      if ((j & 3) == 0) { sg = e8m0_byte<0>(w0); sg8 = e8m0_byte<0>(w1); }
      else if ((j & 3) == 1) { sg = e8m0_byte<1>(w0); sg8 = e8m0_byte<1>(w1); }
      else if ((j & 3) == 2) { sg = e8m0_byte<2>(w0); sg8 = e8m0_byte<2>(w1); }
      else { sg = e8m0_byte<3>(w0); sg8 = e8m0_byte<3>(w1); }
      float d[4];
      mma16816(d, f0[0], f1[0], f0[1], f1[1], b0);
      mma16816_acc(d, f0[2], f1[2], f0[3], f1[3], b1);
      acc[0] = fmaf(d[0], sg, acc[0]);
      acc[1] = fmaf(d[1], sg, acc[1]);
      acc[2] = fmaf(d[2], sg8, acc[2]);
      acc[3] = fmaf(d[3], sg8, acc[3]);
    }
  }
}

// NVFP4 tile: 16-code blocks, so each MMA must stay inside one.  Lane q takes
// codes 4q..4q+3 of both blocks of chunk j (half q & 1 of words q / 2 and
// 2 + q / 2); MMA step s covers block 2j + s.
MOE_DEV void tile_nv(const uint8_t* cs, const uint8_t* s0p, const uint8_t* s1p, const uint2* xb, int nvb,
                     int lane, float (&acc)[4]) {
  const int g = lane >> 2, q = lane & 3;
  const uint32_t sel = (q & 1) ? 0x7632u : 0x5410u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nvb) {
      const uint2 b0 = xb[(2 * j) * 32 + lane], b1 = xb[(2 * j + 1) * 32 + lane];
      const int co = ((j ^ g) << 4) + 4 * (q >> 1);
      const uint8_t* r0 = cs + 128 * g + co;
      const uint8_t* r1 = cs + 128 * (g + 8) + co;
      uint32_t f0[4], f1[4];
      e2m1x8_to_f16x8(__byte_perm(lds32(r0), lds32(r0 + 8), sel), f0);
      e2m1x8_to_f16x8(__byte_perm(lds32(r1), lds32(r1 + 8), sel), f1);
      const uint32_t e0 = *reinterpret_cast<const uint16_t*>(s0p + 2 * j);
      const uint32_t e1 = *reinterpret_cast<const uint16_t*>(s1p + 2 * j);
      const float sa0 = e4m3_to_f32(e0 & 0xffu), sb0 = e4m3_to_f32(e0 >> 8);
      const float sa1 = e4m3_to_f32(e1 & 0xffu), sb1 = e4m3_to_f32(e1 >> 8);
      float d[4], e[4];
      mma16816(d, f0[0], f1[0], f0[1], f1[1], b0);
      mma16816(e, f0[2], f1[2], f0[3], f1[3], b1);
      acc[0] = fmaf(d[0], sa0, fmaf(e[0], sb0, acc[0]));
      acc[1] = fmaf(d[1], sa0, fmaf(e[1], sb0, acc[1]));
      acc[2] = fmaf(d[2], sa1, fmaf(e[2], sb1, acc[2]));
      acc[3] = fmaf(d[3], sa1, fmaf(e[3], sb1, acc[3]));
    }
  }
}

// The part of a stage that compute warp w = 4b + q reads -- rows 16q .. 16q + 15
// of code box b and those rows' scale bytes of the box -- for a miss whose
// weights stream from the host pool: loaded from the pool into the stage in
// the layout the TMA boxes give (16-byte chunk c of a 128-byte code row r at
// chunk c ^ (r & 7)) and stored on to the miss's slot.  Bytes past K are
// neither read nor written.
MOE_DEV void host_part(const Geo& g, const SG& p, const GemvArgs& a, const Entry& en, int mm, int rb, int st,
                       uint8_t* stg, int warp, int lane) {
  const int bslot = warp >> 2, quarter = warp & 3;
  const int kb = st * kBoxes + bslot, rowb = p.K / 2;
  if (kb < p.KB) {
    const uint8_t* hw = a.host_pool + (size_t)en.ex * g.ebytes;
    uint8_t* ew = const_cast<uint8_t*>(a.slots) + (size_t)en.slot * g.ebytes;
    const size_t co = g.off_codes[mm] + (size_t)rb * kBoxRows * rowb + (size_t)kb * 128;
    const int vb = min(128, rowb - kb * 128);
    uint8_t* box = stg + (size_t)bslot * kBoxBytes;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = lane + 32 * j, r = 16 * quarter + (i >> 3), c = i & 7;
      if (c * 16 < vb) v[j] = *reinterpret_cast<const uint4*>(hw + co + (size_t)r * rowb + c * 16);
    }
    uint32_t sw[4];
    const int r_s = 16 * quarter + (lane & 15);
    const size_t so = g.off_scales[mm] + (size_t)(rb * kBoxRows + r_s) * p.scale_row + (size_t)kb * p.SBB;
    const int vsw = min(p.SBB, p.scale_row - kb * p.SBB) / 4;   // 1, 2 or 4 words
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (lane < 16 && w < vsw) sw[w] = *reinterpret_cast<const uint32_t*>(hw + so + 4 * w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = lane + 32 * j, r = 16 * quarter + (i >> 3), c = i & 7;
      if (c * 16 < vb) {
        *reinterpret_cast<uint4*>(box + r * 128 + ((c ^ (r & 7)) << 4)) = v[j];
        *reinterpret_cast<uint4*>(ew + co + (size_t)r * rowb + c * 16) = v[j];
      }
    }
    uint8_t* sd = stg + p.codes_bytes + r_s * p.srow + (p.smode ? bslot : kb) * p.SBB;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      if (lane < 16 && w < vsw) {
        *reinterpret_cast<uint32_t*>(sd + 4 * w) = sw[w];
        *reinterpret_cast<uint32_t*>(ew + so + 4 * w) = sw[w];
      }
  }
  __syncwarp();
}

// Shared state of one CTA.
struct Smem {
  uint8_t* base;            // 1024-aligned dynamic block
  uint64_t *full, *empty;   // weight ring
  uint64_t *rfull, *rempty; // partial-sum slots
  uint64_t *xfull, *xempty; // activation buffers
};

// Bounded wait that gives up at once after an earlier timeout anywhere in
// the CTA; a timeout sets the CTA abort flag and the launch error word.
MOE_DEV bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                           long long limit) {
  if (*abort_flag) return false;
  if (tc::mbar_wait(bar, parity, limit)) return true;
  *abort_flag = 1;
  atomicExch(err, 1);
  return false;
}

MOE_DEV float silu_mul(float a, float u) { return a / (1.0f + __expf(-a)) * u; }

// Stage all N <= 8 tokens of the step (phase 1, `all` geometry) into the group
// buffer at xs, as stage_block does for one entry's group, with the per-token
// exponent computed here from x (the same rule as the router's: amax 2^-s in
// [2^14, 2^15)); columns past N are zero.  x is final before the router
// starts, so this runs before the programmatic wait.  By `nthr` threads
// (index tid) meeting on named barrier `bar`.
template <int FMT>
MOE_DEV void stage_all(const SG& p, int N, const __nv_bfloat16* __restrict__ x, uint2* xs, int* sexp, int tid,
                       int nthr, int bar) {
  const int w = tid >> 5, l = tid & 31, nw = nthr >> 5;
  for (int t = w; t < N; t += nw) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * p.K);
    float m = 0.f;
    for (int i = l; i < p.K / 8; i += 32) {
      const uint4 v = xr[i];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[e] << 16)), fabsf(__uint_as_float(wv[e] & 0xffff0000u))));
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (l == 0) {
      int s = 0;
      if (m > 0.f) {
        int ex;
        frexpf(m, &ex);
        s = max(-100, min(100, ex - 15));
      }
      sexp[t] = s;
    }
  }
  asm volatile("bar.sync %0, %1;" :: "r"(bar), "r"(nthr) : "memory");
  const int k8n = p.K / 8;
  for (int it = tid; it < kTG * k8n; it += nthr) {
    const int t = it / k8n, k8 = it % k8n;
    uint32_t o[4] = {0u, 0u, 0u, 0u};
    if (t < N) {
      const uint4 v = reinterpret_cast<const uint4*>(x + (size_t)t * p.K)[k8];
      const float sc = pow2i(-sexp[t]);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                             __uint_as_float(wv[e] & 0xffff0000u) * sc);
        o[e] = *reinterpret_cast<const uint32_t*>(&hh);
      }
    }
    xs[xslot(FMT, t, 2 * k8)] = make_uint2(o[0], o[1]);
    xs[xslot(FMT, t, 2 * k8 + 1)] = make_uint2(o[2], o[3]);
  }
  asm volatile("bar.sync %0, %1;" :: "r"(bar), "r"(nthr) : "memory");
}

// Stage one token group's activations into buffer xs as f16 in B-fragment
// order, by `nthr` threads (index tid) that meet on named barrier `bar`.
// Phase 1: x (bf16) scaled by the router's per-token 2^-xexp.  Phase 2:
// h = SiLU(a) * u, scaled by 2^-s with s from the bound |h| <= max|a| max|u|
// (phase 1 recorded both maxima per row and 64-column block), so one pass
// suffices and nothing overflows f16.
template <int FMT, int PH>
MOE_DEV void stage_block(const Geo& g, const GemvArgs& a, const SG& p, const Entry& en, int tg, uint2* xs,
                         int* sexp_b, int* stok, const __nv_bfloat16* __restrict__ x,
                         const int* __restrict__ xexp, const float* __restrict__ h, int tid, int nthr,
                         int bar) {
  const int nt = min(kTG, en.nrows - tg * kTG);
  const int rowt = en.row0 + tg * kTG;
  if (PH == 1) {
    if (tid < nt) {
      const int row = rowt + tid;
      const int tok = en.shared ? row - en.row0 : a.tok_of[row];
      stok[tid] = tok;
      sexp_b[tid] = xexp[tok];
    }
    asm volatile("bar.sync %0, %1;" :: "r"(bar), "r"(nthr) : "memory");
    const int k8n = p.K / 8;
#pragma unroll 4
    for (int it = tid; it < nt * k8n; it += nthr) {
      const int t = it / k8n, k8 = it % k8n;
      const uint4 v = reinterpret_cast<const uint4*>(x + (size_t)stok[t] * p.K)[k8];
      const float sc = pow2i(-sexp_b[t]);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                             __uint_as_float(wv[e] & 0xffff0000u) * sc);
        o[e] = *reinterpret_cast<const uint32_t*>(&hh);
      }
      xs[xslot(FMT, t, 2 * k8)] = make_uint2(o[0], o[1]);
      xs[xslot(FMT, t, 2 * k8 + 1)] = make_uint2(o[2], o[3]);
    }
  } else {
    const int nrb = p.K / kBoxRows;   // phase-1 column blocks per matrix
    if (tid < nt) {
      const float* hm = a.hmax + (size_t)(rowt + tid) * 2 * nrb;
      float ma = 0.f, mu = 0.f;
      for (int i = 0; i < nrb; ++i) {
        ma = fmaxf(ma, hm[i]);
        mu = fmaxf(mu, hm[nrb + i]);
      }
      const float bound = ma * mu;
      int s = 0;
      if (bound > 0.f && bound < 3.0e38f) {
        int ex;
        frexpf(bound, &ex);
        s = max(-100, min(100, ex - 15));
      }
      sexp_b[tid] = s;
    }
    asm volatile("bar.sync %0, %1;" :: "r"(bar), "r"(nthr) : "memory");
    const int k4n = p.K / 4;
#pragma unroll 4
    for (int it = tid; it < nt * k4n; it += nthr) {
      const int t = it / k4n, k4 = it % k4n;
      const float4* ar = reinterpret_cast<const float4*>(h + (size_t)(rowt + t) * 2 * p.K);
      const float4 av = ar[k4], uv = ar[k4 + p.K / 4];
      const float sc = pow2i(-sexp_b[t]);
      const __half2 lo = __floats2half2_rn(silu_mul(av.x, uv.x) * sc, silu_mul(av.y, uv.y) * sc);
      const __half2 hi = __floats2half2_rn(silu_mul(av.z, uv.z) * sc, silu_mul(av.w, uv.w) * sc);
      xs[xslot(FMT, t, k4)] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
}

// HOST: the launch may stream misses from the host pool (GemvArgs::host_pool);
// launches over resident weights only use the variant without that path.
template <int FMT, int PH, bool HOST>
__global__ void __launch_bounds__(kThreads, 1)
gemv_stream_kernel(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
                   const __grid_constant__ CUtensorMap smap0, const __grid_constant__ CUtensorMap smap1,
                   Geo g, GemvArgs a, SG p, const __nv_bfloat16* __restrict__ x,
                   const int* __restrict__ xexp, float* __restrict__ h, float* __restrict__ O) {
  extern __shared__ uint8_t smem_raw[];
  Smem S;
  S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  S.full = reinterpret_cast<uint64_t*>(S.base + p.off_bar);
  S.empty = S.full + p.D;
  S.rfull = S.empty + p.D;
  S.rempty = S.rfull + 2;
  S.xfull = S.rempty + 2;
  S.xempty = S.xfull + 2;
  __shared__ int sexp[2][kTG];
  __shared__ int stok[2 * kTG];
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // operational waits give up after wl cycles; the final wait for the
  // producer's own copies in flight keeps the default limit
  const long long wl = a.wait_cycles > 0 ? a.wait_cycles : tc::kWaitCycles;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.D; ++i) {
      tc::mbar_init(&S.full[i], 1);
      tc::mbar_init(&S.empty[i], kCW);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&S.rfull[i], kCW);
      tc::mbar_init(&S.rempty[i], kEW);
      tc::mbar_init(&S.xfull[i], kEW);
      tc::mbar_init(&S.xempty[i], kCW);
    }
    s_abort = 0;
    tc::mbar_init_fence();
  }
  __syncthreads();
  // launched as a dependent of the previous kernel: phase 2's producer only
  // reads the step record and weights, both final before phase 1 got past its
  // own wait, so it starts streaming at once; everything else waits for the
  // predecessor.  The successor is released only after this wait, so what
  // the successor's producer reads without waiting is final by then.
  if (warp == kProd && lane == 0) {
    // descriptor fetches overlap the wait for the predecessor
    tc::prefetch_tmap(&map0);
    tc::prefetch_tmap(&map1);
    if (p.smode) {
      tc::prefetch_tmap(&smap0);
      tc::prefetch_tmap(&smap1);
    }
  }
  const bool ALL = PH == 1 && p.all;
  if (ALL && warp != kProd) {
    // every token of the step, before the wait: x is final before the router starts
    const int tid = warp < kCW ? threadIdx.x : threadIdx.x - 32;
    stage_all<FMT>(p, a.N, x, reinterpret_cast<uint2*>(S.base + p.off_x), &sexp[0][0], tid, kThreads - 32, 2);
  }
  if (PH == 1 || warp != kProd) pdl_wait();
  pdl_trigger();
  const Range rr = cta_range(g, a, p);
  // the first token group is staged by every warp but the producer (its
  // latency is on the critical path); the epilogue stages later ones ahead
  if (!ALL && warp != kProd) {
    Cursor c0;
    cursor_init(c0, rr);
    if (cursor_next(c0, g, a, p, rr)) {
      const int tid = warp < kCW ? threadIdx.x : threadIdx.x - 32;
      stage_block<FMT, PH>(g, a, p, c0.en, c0.tg, reinterpret_cast<uint2*>(S.base + p.off_x), sexp[0], stok, x,
                           xexp, h, tid, kThreads - 32, 2);
      asm volatile("bar.sync 2, %0;" :: "n"(kThreads - 32) : "memory");
      if (warp > kCW && lane == 0) mbar_arrive(&S.xfull[0]);
    }
  }

  if (warp == kProd) {
    // ------------------------------------------------------------ producer
    uint32_t n = 0;
    Cursor cu;
    cursor_init(cu, rr);
    bool stop = false;
    while (!stop && cursor_next(cu, g, a, p, rr)) {
      const uint8_t* ew = a.slots + (size_t)cu.en.slot * g.ebytes;
      const bool hw = HOST && cu.en.ex >= 0;
      for (int u = cu.ue0; u < cu.ue1 && !stop; ++u) {
        const int m = PH == 1 ? u / p.RB : 0;          // 0: gate / down, 1: up
        const int rb = PH == 1 ? u % p.RB : u;
        const CUtensorMap* map = m == 0 ? &map0 : &map1;
        const CUtensorMap* smap = m == 0 ? &smap0 : &smap1;
        const uint8_t* sgl = ew + g.off_scales[PH == 1 ? m : 2] + (size_t)rb * kBoxRows * p.scale_row;
        for (int st = 0; st < p.NS; ++st) {
          const int slot = n % p.D;
          const uint32_t k = n / p.D;
          if (k > 0 && !wait_or_abort(&S.empty[slot], (k - 1) & 1, &s_abort, a.err, wl)) {
            stop = true;
            break;
          }
          uint8_t* stg = S.base + (size_t)slot * p.stage_bytes;
          const int nbx = min(kBoxes, p.KB - st * kBoxes);
          const uint32_t sbytes = kBoxRows * p.srow;
          if (hw) {
            // a miss streamed from the host pool: the compute warps load their
            // own parts of the stage (one warp keeps far too few loads in
            // flight over the host link), so the stage is theirs once it is free
            if (lane == 0) mbar_arrive(&S.full[slot]);
            ++n;
            continue;
          }
          if (lane == 0) tc::mbar_expect_tx(&S.full[slot], (uint32_t)(nbx * kBoxBytes) + sbytes);
          __syncwarp();
          if (lane < nbx)
            tc::tma_load_3d(stg + (size_t)lane * kBoxBytes, map, &S.full[slot], (st * kBoxes + lane) * (kBoxK / 2),
                            rb * kBoxRows, cu.en.slot);
          else if (lane == kBoxes) {
            // the scales of the stage's boxes: 64 rows x (4 boxes' bytes), or the unit's whole rows
            if (p.smode)
              tc::tma_load_3d(stg + p.codes_bytes, smap, &S.full[slot], st * kBoxes * p.SBB, rb * kBoxRows,
                              cu.en.slot);
            else
              bulk_load(stg + p.codes_bytes, sgl, sbytes, &S.full[slot]);
          }
          ++n;
        }
      }
    }
    // copies still in flight land before the CTA exits (bounded wait)
    if (lane == 0) {
      const uint32_t first = n > (uint32_t)p.D ? n - p.D : 0;
      for (uint32_t i = first; i < n; ++i)
        if (!tc::mbar_wait(&S.full[i % p.D], (i / p.D) & 1)) {
          atomicExch(a.err, 1);
          break;
        }
    }
  } else if (warp < kCW) {
    // ------------------------------------------------------------ compute
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float* red = reinterpret_cast<float*>(S.base + p.off_red);
    const int bslot = warp >> 2, quarter = warp & 3, gq = lane >> 2;
    uint32_t n = 0, us = 0, bs = 0;
    Cursor cu;
    cursor_init(cu, rr);
    while (cursor_next(cu, g, a, p, rr)) {
      const int xb = bs % p.XB;
      if (!ALL) wait_or_abort(&S.xfull[xb], (bs / p.XB) & 1, &s_abort, a.err, wl);
      const uint2* xs = reinterpret_cast<const uint2*>(S.base + p.off_x + (size_t)xb * p.xbytes);
      for (int u = cu.ue0; u < cu.ue1; ++u) {
        for (int st = 0; st < p.NS; ++st, ++n) {
          const int slot = n % p.D;
          const bool ok = wait_or_abort(&S.full[slot], (n / p.D) & 1, &s_abort, a.err, wl);
          const int kb = st * kBoxes + bslot;
          if (HOST && ok && cu.en.ex >= 0)
            host_part(g, p, a, cu.en, PH == 1 ? u / p.RB : 2, PH == 1 ? u % p.RB : u, st,
                      S.base + (size_t)slot * p.stage_bytes, warp, lane);
          if (ok && kb < p.KB) {
            const uint8_t* stg = S.base + (size_t)slot * p.stage_bytes;
            const uint8_t* cs = stg + (size_t)bslot * kBoxBytes + quarter * (16 * kBoxK / 2);
            const uint8_t* sc = stg + p.codes_bytes + (16 * quarter + gq) * p.srow + (p.smode ? bslot : kb) * p.SBB;
            const int nvb = min(8, (p.K - kb * kBoxK) / 32);
            const uint2* xk = xs + (size_t)kb * 512;   // 8 blocks x 2 steps x 32 lanes
            if (FMT == MOE_MXFP4) tile_mx(cs, sc, sc + 8 * p.srow, xk, nvb, lane, acc);
            else tile_nv(cs, sc, sc + 8 * p.srow, xk, nvb, lane, acc);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.empty[slot]);
        }
        // unit done: hand the partial sums to the epilogue
        const int r = us % p.RS;
        if (us >= (uint32_t)p.RS) wait_or_abort(&S.rempty[r], (us / p.RS - 1) & 1, &s_abort, a.err, wl);
        reinterpret_cast<float4*>(red + (size_t)r * (p.rbytes / 4))[warp * 32 + lane] =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.rfull[r]);
        ++us;
      }
      if (!ALL) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.xempty[xb]);
      }
      ++bs;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int te = threadIdx.x - (kCW + 1) * 32;   // 0 .. kET - 1
    const int ew_ = warp - (kCW + 1);              // epilogue warp 0 .. kEW - 1
    const float* red = reinterpret_cast<const float*>(S.base + p.off_red);
    // stage block number bs_st into its buffer (waits for the buffer to be free)
    // stage block number bs_st into its buffer once that buffer is free
    auto stage = [&](const Cursor& c, uint32_t bs_st) {
      const int xb = bs_st % p.XB;
      epi_sync();   // the previous staging's token list and exponents are no longer read
      if (bs_st >= (uint32_t)p.XB) wait_or_abort(&S.xempty[xb], (bs_st / p.XB - 1) & 1, &s_abort, a.err, wl);
      stage_block<FMT, PH>(g, a, p, c.en, c.tg, reinterpret_cast<uint2*>(S.base + p.off_x + (size_t)xb * p.xbytes),
                           sexp[xb], stok, x, xexp, h, te, kET, 1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.xfull[xb]);
    };
    Cursor cs, cr;   // staging runs XB blocks ahead of the reduction
    cursor_init(cs, rr);
    cursor_init(cr, rr);
    uint32_t bs_st = 1, bs_rd = 0, us = 0;   // block 0 was staged by all warps
    if (!ALL) {
      cursor_next(cs, g, a, p, rr);
      for (int i = 1; i < p.XB; ++i)
        if (cursor_next(cs, g, a, p, rr)) stage(cs, bs_st++);
    }
    while (cursor_next(cr, g, a, p, rr)) {
      const int xb = bs_rd % p.XB;
      const int nt = ALL ? cr.en.nrows : min(kTG, cr.en.nrows - cr.tg * kTG);
      const int rowt = cr.en.row0 + cr.tg * kTG;
      if (ALL) {
        // the entry's tokens (all N tokens are staged; entries pick theirs)
        epi_sync();
        if (te < nt)
          stok[te] = cr.en.shared ? te : (te == 0 && cr.en.tok0 >= 0) ? cr.en.tok0 : a.tok_of[rowt + te];
        epi_sync();
      }
      const float* tsp = reinterpret_cast<const float*>(
          (HOST && cr.en.ex >= 0 ? a.host_pool + (size_t)cr.en.ex * g.ebytes : a.slots + (size_t)cr.en.slot * g.ebytes) +
          g.off_tscale);
      if (HOST && PH == 1 && cr.en.ex >= 0 && te == 0)   // a miss's tensor scales go on to its slot too
        *reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.slots) + (size_t)cr.en.slot * g.ebytes + g.off_tscale) =
            *reinterpret_cast<const uint4*>(tsp);
      for (int u = cr.ue0; u < cr.ue1; ++u) {
        const int m = PH == 1 ? u / p.RB : 0;
        const int rb = PH == 1 ? u % p.RB : u;
        const float ts = tsp[PH == 1 ? m : 2];
        const int r = us % p.RS;
        const bool ok = wait_or_abort(&S.rfull[r], (us / p.RS) & 1, &s_abort, a.err, wl);
        const float4* rs = reinterpret_cast<const float4*>(red + (size_t)r * (p.rbytes / 4));
        // warp w takes tokens w, w + kEW, ...; lane c takes columns c, c + 32 of the block
        for (int tk = ew_; ok && tk < nt; tk += kEW) {
          // column of this row's token among the staged ones
          const int cc = ALL ? stok[tk] : tk;
          const float sc = pow2i(ALL ? sexp[0][cc] : sexp[xb][tk]) * ts;
          float mx = 0.f;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int col = lane + 32 * c2;
            const int qr = col >> 4, rr_ = col & 15;
            const int lo = 4 * (rr_ & 7) + (cc >> 1), jj = 2 * (rr_ >> 3) + (cc & 1);
            float s = 0.f;
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) {
              const float4 v = rs[(b * 4 + qr) * 32 + lo];
              s += jj == 0 ? v.x : jj == 1 ? v.y : jj == 2 ? v.z : v.w;
            }
            const float val = s * sc;
            mx = fmaxf(mx, fabsf(val));
            if (PH == 1) h[(size_t)(rowt + tk) * 2 * p.R + m * p.R + rb * kBoxRows + col] = val;
            else O[(size_t)(rowt + tk) * p.R + rb * kBoxRows + col] = val;
          }
          if (PH == 1) {
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) a.hmax[(size_t)(rowt + tk) * 2 * p.RB + m * p.RB + rb] = mx;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.rempty[r]);
        ++us;
      }
      ++bs_rd;
      if (!ALL) {
        // every epilogue warp is done with this block's exponents before they are restaged
        epi_sync();
        if (cursor_next(cs, g, a, p, rr)) stage(cs, bs_st++);
      }
    }
  }
  __syncthreads();
}

// N: tokens of the launch (phase 1 with N <= 8 stages every token once, one
// MMA group, when a ring of at least 3 stages still fits; 0 = the per-group
// geometry).  With more tokens an entry's own group is staged per block:
// staging two groups per launch cost more than it saved.
SG make_sg(const Geo& g, int ph, int N) {
  SG p{};
  p.K = ph == 1 ? g.d : g.f;
  p.R = ph == 1 ? g.f : g.d;
  p.KB = (p.K + kBoxK - 1) / kBoxK;
  p.NS = (p.KB + kBoxes - 1) / kBoxes;
  p.RB = p.R / kBoxRows;
  p.UE = p.RB * (ph == 1 ? 2 : 1);
  p.SBB = g.fmt == MOE_MXFP4 ? 8 : 16;
  p.scale_row = p.K / g.blk;
  // scale rows that are 16-byte multiples can be cut into TMA boxes; others
  // are bulk-copied whole (a stage then carries the unit's full scale rows)
  p.smode = p.scale_row % 16 == 0 ? 1 : 0;
  p.srow = p.smode ? kBoxes * p.SBB : p.scale_row;
  p.codes_bytes = kBoxes * kBoxBytes;
  p.stage_bytes = (p.codes_bytes + kBoxRows * p.srow + 1023) & ~1023;
  p.xbytes = p.K * 2 * kTG;                   // f16, 8 tokens
  p.rbytes = kCW * 32 * 16;                   // one float4 per compute lane
  const int bars = 2 * kMaxD * 8 + 8 * 8;
  // two activation buffers and two partial-sum slots when a 3-stage ring still fits
  p.XB = 2;
  p.RS = 2;
  if (2 * p.xbytes + 2 * p.rbytes + 3 * p.stage_bytes + bars > kSmemBudget) p.XB = 1;
  const int fixed = p.XB * p.xbytes + p.RS * p.rbytes + bars;
  p.D = std::min(kMaxD, (kSmemBudget - fixed) / p.stage_bytes);
  p.all = 0;
  if (ph == 1 && N > 0 && N <= kTG) {
    SG q = p;
    q.all = 1;
    q.XB = 1;
    const int fq = q.xbytes + q.RS * q.rbytes + bars;
    q.D = std::min(kMaxD, (kSmemBudget - fq) / q.stage_bytes);
    if (q.D >= 3) p = q;
  }
  p.off_x = p.D * p.stage_bytes;
  p.off_red = p.off_x + p.XB * p.xbytes;
  p.off_bar = p.off_red + p.RS * p.rbytes;
  p.smem = 1024 + p.off_bar + bars;
  return p;
}

template <int FMT, int PH, bool HOST>
cudaError_t launch_phase(const Geo& g, const GemvPlan* pl, const GemvArgs& a, const SG& p,
                         const __nv_bfloat16* x, const int* xexp, float* h, float* O, int n_ent_max,
                         int num_sms, cudaStream_t st) {
  cudaError_t e = ensure_smem_limit((const void*)gemv_stream_kernel<FMT, PH, HOST>, kSmemBudget + 1024);
  if (e != cudaSuccess) return e;
  const long long units = (long long)n_ent_max * p.UE;
  // phase 1 is launched while the one-CTA routing tail still holds an SM, and
  // a CTA of this size cannot share it: leave that SM out rather than have
  // one CTA start after the tail and finish last
  const int grid = (int)std::min<long long>(PH == 1 ? std::max(1, num_sms - 1) : num_sms, units);
  if (grid <= 0) return cudaSuccess;
  const CUtensorMap& m0 = PH == 1 ? pl->w[0] : pl->w[2];
  const CUtensorMap& m1 = PH == 1 ? pl->w[1] : pl->w[2];
  const CUtensorMap& s0 = PH == 1 ? pl->s[0] : pl->s[2];
  const CUtensorMap& s1 = PH == 1 ? pl->s[1] : pl->s[2];
  return launch_pdl(gemv_stream_kernel<FMT, PH, HOST>, dim3(grid), dim3(kThreads), (size_t)p.smem, st, m0, m1, s0,
                    s1, g, a, p, x, xexp, h, O);
}

template <int FMT>
cudaError_t launch_fmt(const Geo& g, const GemvPlan* pl, const GemvArgs& a, const __nv_bfloat16* x,
                       const int* xexp, float* h, float* O, int n_ent_max, int num_sms,
                       cudaStream_t st, const cudaEvent_t* ev, int phases) {
  cudaError_t e = cudaSuccess;
  if (phases & 1) {
    const SG p1 = make_sg(g, 1, a.N);
    if (ev) cudaEventRecord(ev[0], st);
    e = a.host_pool ? launch_phase<FMT, 1, true>(g, pl, a, p1, x, xexp, h, O, n_ent_max, num_sms, st)
                    : launch_phase<FMT, 1, false>(g, pl, a, p1, x, xexp, h, O, n_ent_max, num_sms, st);
    if (ev) cudaEventRecord(ev[1], st);
    if (e != cudaSuccess) return e;
  }
  if (phases & 2) {
    const SG p2 = make_sg(g, 2, a.N);
    if (ev) cudaEventRecord(ev[2], st);
    e = a.host_pool ? launch_phase<FMT, 2, true>(g, pl, a, p2, x, xexp, h, O, n_ent_max, num_sms, st)
                    : launch_phase<FMT, 2, false>(g, pl, a, p2, x, xexp, h, O, n_ent_max, num_sms, st);
    if (ev) cudaEventRecord(ev[3], st);
  }
  return e;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// Codes of one matrix in every slot: [slot][row][K/2 bytes], boxes of
// 64 rows x 128 bytes, 128-byte swizzle; a box past the row end reads zeros.
bool make_box_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                  uint64_t slot_stride) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {kBoxK / 2, kBoxRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale bytes of one matrix in every slot: [slot][row][scale_row], boxes of
// 64 rows x (4 code boxes' scale bytes), no swizzle.
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                    uint64_t slot_stride, uint32_t box_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {box_bytes, kBoxRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Shapes the decode kernels accept: d_model and d_ff multiples of 128 (so
// the 64-row blocks tile both) up to 8192, and a ring of at least two stages
// next to the staged activations.
bool gemv_shape_ok(const Geo& g) {
  if (g.d > 8192 || g.f > 8192 || g.d % 128 || g.f % 128) return false;
  return make_sg(g, 1, 0).D >= 2 && make_sg(g, 2, 0).D >= 2;
}

GemvPlan* gemv_plan_create(const Geo& g, const uint8_t* slots) {
  GemvPlan* pl = new GemvPlan();
  const int ns = g.S + 1 + g.X;   // LRU slots' buffers, the shared expert's, the spares
  pl->ready = make_box_map(&pl->w[0], slots + g.off_codes[0], g.d / 2, g.f, ns, g.ebytes) &&
              make_box_map(&pl->w[1], slots + g.off_codes[1], g.d / 2, g.f, ns, g.ebytes) &&
              make_box_map(&pl->w[2], slots + g.off_codes[2], g.f / 2, g.d, ns, g.ebytes);
  // scale maps only where a scale row is a 16-byte multiple (the phase uses them then)
  const SG p1 = make_sg(g, 1, 0), p2 = make_sg(g, 2, 0);
  const uint32_t sb = kBoxes * (g.fmt == MOE_MXFP4 ? 8 : 16);
  if (pl->ready && p1.smode)
    pl->ready = make_scale_map(&pl->s[0], slots + g.off_scales[0], p1.scale_row, g.f, ns, g.ebytes, sb) &&
                make_scale_map(&pl->s[1], slots + g.off_scales[1], p1.scale_row, g.f, ns, g.ebytes, sb);
  if (pl->ready && p2.smode)
    pl->ready = make_scale_map(&pl->s[2], slots + g.off_scales[2], p2.scale_row, g.d, ns, g.ebytes, sb);
  return pl;
}

void gemv_plan_destroy(GemvPlan* pl) { delete pl; }
bool gemv_plan_ready(const GemvPlan* pl) { return pl && pl->ready; }

cudaError_t launch_gemv_decode(const Geo& g, const GemvPlan* pl, const GemvArgs& a,
                               const __nv_bfloat16* x, const int* xexp, float* h, float* O,
                               int n_ent_max, int num_sms, cudaStream_t st, const cudaEvent_t* ev,
                               int phases) {
  if (g.fmt == MOE_MXFP4)
    return launch_fmt<MOE_MXFP4>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
  return launch_fmt<MOE_NVFP4>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
}

}  // namespace moe
