// Device pieces of the decode expert FFN (a persistent, warp-specialised
// grouped GEMV over FP4 weights), shared by the stand-alone GEMV launches
// (gemv.cu) and the fused decode step (step.cu).
//
// Decode moves each routed expert's weights once per step for a handful of
// tokens, so the expert FFN is bound by HBM bandwidth (the pages' decode is
// bound by the bytes each step must move: "FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).  The design is described in gemv.cu;
// this header holds its pieces:
//  * the phase geometry (SG) and the tensor maps of the slot pool (GemvPlan);
//  * the FP4 tile math (cvt.rn.f16x2.e2m1x2 + mma.sync m16n8k16) and the
//    activation staging in B-fragment order;
//  * the work list (EntryTable: the launch's accesses in access order, plus
//    the shared expert) and each CTA's contiguous range of work units;
//  * the three role loops -- produce (TMA weight ring), compute (MMAs),
//    reduce (fixed-order partial sums, outputs, activation staging) -- which
//    meet only at mbarriers.  Each keeps its ring counters in a Ring, so a
//    kernel can run phase 1 and then phase 2 through one ring (the fused step).
#pragma once
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "router_dev.cuh"
#include "tc.cuh"

namespace moe {

struct GemvPlan {
  CUtensorMap w[3];   // gate, up, down codes of all slots (+ the shared expert)
  CUtensorMap s[3];   // their scale bytes (used when a scale row is a 16-byte multiple)
  bool ready;
};


namespace gv {


constexpr int kCW = 16;                      // compute warps
constexpr int kEW = 3;                       // epilogue warps
constexpr int kProd = kCW;                   // producer warp index
constexpr int kThreads = (kCW + 1 + kEW) * 32;
constexpr int kET = kEW * 32;                // epilogue threads
constexpr int kTG = 8;                       // tokens per group (one MMA N)
constexpr int kBoxRows = 64;
constexpr int kBoxRowBytes = 128;           // bytes per box row (256 FP4, 128 FP8, 64 bf16 elements)
constexpr int kBoxBytes = kBoxRows * kBoxRowBytes;
constexpr int kBoxes = 4;                    // boxes per stage
constexpr int kMaxD = 8;                     // ring stages at most
constexpr int kSmemBudget = 220 * 1024;

// Geometry of one phase (host-computed, passed by value).
struct SG {
  int K, R;           // reduction length, output rows per matrix
  int bk;             // K elements per 128-byte box row: 256 (FP4), 128 (MXFP8), 64 (BF16)
  int KB;             // boxes per row (an FP4 row's last one may be half valid)
  int NS;             // stages per unit
  int RB;             // 64-row blocks per matrix
  int UE;             // units per entry (RB per matrix, gate and up separately in phase 1)
  int SBB;            // scale bytes per box row (8 MXFP4, 16 NVFP4, 4 MXFP8, 0 BF16)
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


// The work of one launch: accesses [base, base + nr) of an access-ordered
// table (hits ascending id, then misses ascending id), plus the shared expert
// when `shared`.  Every role of a CTA walks this table with the same result
// (get_entry never waits), so the roles' named barriers stay matched.
struct EntryTable {
  const int4* ent;      // per access {buffer, first permuted row, rows, first token}
  const int* expert;    // per access: expert id
  int base, nr;
  int n_hit;            // accesses before this index are hits
  int shared;
};

MOE_DEV bool get_entry(const Geo& g, const GemvArgs& a, const EntryTable& T, int ent, Entry& out) {
  if (ent < T.nr) {
    const int i = T.base + ent;
    // one 16-byte load: physical slot, first row, rows, first token
    const int4 v = T.ent[i];
    const bool slot_ok = (v.x >= 0 && v.x < g.S) || (v.x > g.S && v.x <= g.S + g.X);
    out.slot = v.x;
    out.row0 = v.y;
    out.nrows = v.z;
    out.shared = 0;
    const uint32_t tk = (uint32_t)v.w;
    out.tok0 = (tk >> 16) == 0xffffu ? -1 : (int)(tk & 0xffffu);
    out.ex = -1;
    if (a.host_pool && i >= T.n_hit) {
      out.ex = T.expert[i];
      if (out.ex < 0 || out.ex >= g.E) return false;
    }
    return slot_ok && out.nrows > 0 && out.row0 >= 0 && out.row0 + out.nrows <= a.N * g.k;
  }
  if (T.shared && ent == T.nr) {
    out.slot = g.shb;
    out.row0 = a.N * g.k;
    out.nrows = a.N;
    out.shared = 1;
    out.tok0 = 0;
    out.ex = -1;
    return a.N > 0;
  }
  return false;
}

// This CTA's unit range [u0, u1) of the launch's (nr + shared) * UE units:
// CTA `cta` of `ncta` takes an equal contiguous share.  (A launch that streams
// misses from the host pool keeps them in a contiguous run of CTAs: spreading
// them over every CTA measured slower on the host link.)
struct Range {
  int u0, u1;
};

MOE_DEV Range cta_range(const EntryTable& T, const SG& p, int cta, int ncta) {
  Range r;
  const long long n = (long long)(T.nr + T.shared) * p.UE;
  r.u0 = (int)(n * cta / ncta);
  r.u1 = (int)(n * (cta + 1) / ncta);
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

MOE_DEV bool cursor_next(Cursor& c, const Geo& g, const GemvArgs& a, const EntryTable& T, const SG& p,
                         const Range& rr) {
  if (c.tg + 1 < c.ntg) {
    ++c.tg;
    return true;
  }
  while (c.t < rr.u1) {
    const int ent = c.t / p.UE;
    c.ue0 = c.t % p.UE;
    c.ue1 = min(p.UE, c.ue0 + (rr.u1 - c.t));
    c.t += c.ue1 - c.ue0;
    if (get_entry(g, a, T, ent, c.en)) {
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
  // MXFP8 and BF16: one MMA step per 16 K, lane q holding K 4q .. 4q + 3
  if (fmt == MOE_MXFP8 || fmt == MOE_BF16) return (k4 >> 2) * 32 + 4 * t + (k4 & 3);
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

// Four E4M3 codes (one word, low byte = lowest K) -> two f16x2, exact (every
// E4M3 value is an f16 value).
MOE_DEV void e4m3x4_to_f16x4(uint32_t w, uint32_t (&o)[2]) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(o[0]), "=r"(o[1]) : "r"(w));
}

// One warp's 16 x 128 MXFP8 tile: acc += W x.  Codes: 128-byte rows of E4M3
// bytes, 16-byte chunk j of row r at chunk j ^ (r & 7).  Lane (g, q) takes
// word q of chunk j (codes 16 j + 4q .. + 3) of rows g and g + 8; as f16
// pairs they are the MMA's K slots 2q, 2q + 1 and 2q + 8, 2q + 9, so chunk j
// is one m16n8k16 step (the activations are staged in that order, xslot).
// Chunks 2p and 2p + 1 share E8M0 scale byte p of the box.
MOE_DEV void tile_mx8(const uint8_t* cs, const uint8_t* s0p, const uint8_t* s1p, const uint2* xb, int lane,
                      float (&acc)[4]) {
  const int g = lane >> 2, q = lane & 3;
  const uint32_t w0 = lds32(s0p), w1 = lds32(s1p);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float d[4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int j = 2 * p + hh;
      const int co = ((j ^ g) << 4) + 4 * q;
      uint32_t f0[2], f1[2];
      e4m3x4_to_f16x4(lds32(cs + 128 * g + co), f0);
      e4m3x4_to_f16x4(lds32(cs + 128 * (g + 8) + co), f1);
      const uint2 b = xb[j * 32 + lane];
      if (hh == 0) mma16816(d, f0[0], f1[0], f0[1], f1[1], b);
      else mma16816_acc(d, f0[0], f1[0], f0[1], f1[1], b);
    }
    float sg, sg8;
    if (p == 0) { sg = e8m0_byte<0>(w0); sg8 = e8m0_byte<0>(w1); }
    else if (p == 1) { sg = e8m0_byte<1>(w0); sg8 = e8m0_byte<1>(w1); }
    else if (p == 2) { sg = e8m0_byte<2>(w0); sg8 = e8m0_byte<2>(w1); }
    else { sg = e8m0_byte<3>(w0); sg8 = e8m0_byte<3>(w1); }
    acc[0] = fmaf(d[0], sg, acc[0]);
    acc[1] = fmaf(d[1], sg, acc[1]);
    acc[2] = fmaf(d[2], sg8, acc[2]);
    acc[3] = fmaf(d[3], sg8, acc[3]);
  }
}

MOE_DEV void mma16816_bf16_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// One warp's 16 x 64 bf16 tile: acc += W x (bf16 MMA, fp32 sums).  Rows of
// 128 bytes (64 elements, 16-byte chunks swizzled as above); for each 16-K
// group G lane (g, q) takes 8 bytes -- elements 16 G + 4q .. + 3 -- of rows g
// and g + 8: the MMA's K slots 2q, 2q + 1 and 2q + 8, 2q + 9.
MOE_DEV void tile_bf16(const uint8_t* cs, const uint2* xb, int lane, float (&acc)[4]) {
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    const int c = 2 * G + (q >> 1);
    const int co = ((c ^ g) << 4) + 8 * (q & 1);
    const uint2 r0 = *reinterpret_cast<const uint2*>(cs + 128 * g + co);
    const uint2 r1 = *reinterpret_cast<const uint2*>(cs + 128 * (g + 8) + co);
    mma16816_bf16_acc(acc, r0.x, r1.x, r0.y, r1.y, xb[G * 32 + lane]);
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
  const int kb = st * kBoxes + bslot, rowb = p.K * fmt_code_bits(g.fmt) / 8;
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
// the CTA; a timeout sets the CTA abort flag and the launch error word.  Called
// by whole warps; the result is the same in every lane (a lane that gave up
// makes the warp give up), so a warp never splits around the mma.sync and
// __syncwarp that follow.
MOE_DEV bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                           long long limit) {
  bool ok = false;
  if (!*abort_flag) {
    ok = tc::mbar_wait(bar, parity, limit);
    if (!ok) {
      *abort_flag = 1;
      atomicExch(err, 1);
    }
  }
  return __all_sync(0xffffffffu, ok);
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
    const int s = FMT == MOE_BF16 ? 0 : rt::token_exp(x + (size_t)t * p.K, p.K);   // bf16 MMA: x as it is
    if (l == 0) sexp[t] = s;
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
        if (FMT == MOE_BF16) {
          o[e] = wv[e];
        } else {
          const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                               __uint_as_float(wv[e] & 0xffff0000u) * sc);
          o[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
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
      sexp_b[tid] = FMT == MOE_BF16 ? 0 : xexp[tok];
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
        if (FMT == MOE_BF16) {
          o[e] = wv[e];
        } else {
          const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * sc,
                                               __uint_as_float(wv[e] & 0xffff0000u) * sc);
          o[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
      }
      xs[xslot(FMT, t, 2 * k8)] = make_uint2(o[0], o[1]);
      xs[xslot(FMT, t, 2 * k8 + 1)] = make_uint2(o[2], o[3]);
    }
  } else {
    const int nrb = p.K / kBoxRows;   // phase-1 column blocks per matrix
    // a warp per row (tid is warp-aligned): its lanes load the row's 2 nrb
    // block maxima together -- one round trip, not one per block -- and
    // combine them by a warp max (the same maximum in any order)
    const int lane = tid & 31;
    for (int t = tid >> 5; t < nt; t += nthr >> 5) {
      const float* hm = a.hmax + (size_t)(rowt + t) * 2 * nrb;
      float ma = 0.f, mu = 0.f;
#pragma unroll 4
      for (int i = lane; i < nrb; i += 32) {
        ma = fmaxf(ma, __ldcg(hm + i));
        mu = fmaxf(mu, __ldcg(hm + nrb + i));
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, o));
        mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
      }
      const float bound = ma * mu;
      int s = 0;
      if (FMT != MOE_BF16 && bound > 0.f && bound < 3.0e38f) {   // bf16 h needs no scaling
        int ex;
        frexpf(bound, &ex);
        s = max(-100, min(100, ex - 15));
      }
      if (lane == 0) sexp_b[t] = s;
    }
    asm volatile("bar.sync %0, %1;" :: "r"(bar), "r"(nthr) : "memory");
    const int k4n = p.K / 4;
#pragma unroll 4
    for (int it = tid; it < nt * k4n; it += nthr) {
      const int t = it / k4n, k4 = it % k4n;
      const float4* ar = reinterpret_cast<const float4*>(h + (size_t)(rowt + t) * 2 * p.K);
      const float4 av = __ldcg(ar + k4), uv = __ldcg(ar + k4 + p.K / 4);
      const float sc = pow2i(-sexp_b[t]);
      if (FMT == MOE_BF16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(silu_mul(av.x, uv.x), silu_mul(av.y, uv.y));
        const __nv_bfloat162 hi = __floats2bfloat162_rn(silu_mul(av.z, uv.z), silu_mul(av.w, uv.w));
        xs[xslot(FMT, t, k4)] =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      } else {
        const __half2 lo = __floats2half2_rn(silu_mul(av.x, uv.x) * sc, silu_mul(av.y, uv.y) * sc);
        const __half2 hi = __floats2half2_rn(silu_mul(av.z, uv.z) * sc, silu_mul(av.w, uv.w) * sc);
        xs[xslot(FMT, t, k4)] =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      }
    }
  }
}

// HOST: the launch may stream misses from the host pool (GemvArgs::host_pool);
// launches over resident weights only use the variant without that path.

inline SG make_sg(const Geo& g, int ph, int N) {
  SG p{};
  p.K = ph == 1 ? g.d : g.f;
  p.R = ph == 1 ? g.f : g.d;
  p.bk = 1024 / fmt_code_bits(g.fmt);          // elements in 128 bytes
  p.KB = (p.K + p.bk - 1) / p.bk;
  p.NS = (p.KB + kBoxes - 1) / kBoxes;
  p.RB = p.R / kBoxRows;
  p.UE = p.RB * (ph == 1 ? 2 : 1);
  p.SBB = g.blk ? p.bk / g.blk : 0;
  p.scale_row = fmt_scale_row(g.fmt, p.K);
  // scale rows that are 16-byte multiples can be cut into TMA boxes; others
  // are bulk-copied whole (a stage then carries the unit's full scale rows)
  p.smode = p.SBB > 0 && p.scale_row % 16 == 0 ? 1 : 0;   // (no scales at all: 0, with 0 bytes)
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


// Shared scalars of the role loops (static shared memory of the kernel).
struct Small {
  int sexp[2][kTG];      // per-token exponents of the staged groups (ALL: sexp[0][t], t < 8)
  int stok[2 * kTG];     // tokens of the staged / reduced block
  volatile int abort;    // a bounded wait of this CTA gave up
};

// Ring counters of one role, carried from one phase to the next.
struct Ring {
  uint32_t n = 0;    // weight-ring stages (producer: filled, compute: consumed)
  uint32_t us = 0;   // partial-sum slots (compute: filled, epilogue: drained)
  uint32_t bs = 0;   // activation buffers (compute: consumed, epilogue: staged)
  uint32_t br = 0;   // epilogue: blocks reduced
};

// ---------------------------------------------------------------- producer
// Streams the range's weights into the ring (one warp; lane 0 arms the
// stage's barrier, lanes 0..3 issue the code boxes, lane 4 the scales).
// Misses read from the host pool are loaded by the compute warps instead:
// their stages are handed over as soon as they are free.
template <int FMT, int PH, bool HOST>
MOE_DEV void produce(const Geo& g, const GemvArgs& a, const SG& p, const EntryTable& T, const Range& rr,
                     const Smem& S, Small& sm, Ring& ring, const CUtensorMap* map0, const CUtensorMap* map1,
                     const CUtensorMap* smap0, const CUtensorMap* smap1, long long wl) {
  const int lane = threadIdx.x & 31;
  uint32_t n = ring.n;
  Cursor cu;
  cursor_init(cu, rr);
  bool stop = false;
  while (!stop && cursor_next(cu, g, a, T, p, rr)) {
    const uint8_t* ew = a.slots + (size_t)cu.en.slot * g.ebytes;
    const bool hw = HOST && cu.en.ex >= 0;
    for (int u = cu.ue0; u < cu.ue1 && !stop; ++u) {
      const int m = PH == 1 ? u / p.RB : 0;          // 0: gate / down, 1: up
      const int rb = PH == 1 ? u % p.RB : u;
      const CUtensorMap* map = m == 0 ? map0 : map1;
      const CUtensorMap* smap = m == 0 ? smap0 : smap1;
      const uint8_t* sgl = ew + g.off_scales[PH == 1 ? m : 2] + (size_t)rb * kBoxRows * p.scale_row;
      for (int st = 0; st < p.NS; ++st) {
        const int slot = n % p.D;
        const uint32_t k = n / p.D;
        if (k > 0 && !wait_or_abort(&S.empty[slot], (k - 1) & 1, &sm.abort, a.err, wl)) {
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
          tc::tma_load_3d(stg + (size_t)lane * kBoxBytes, map, &S.full[slot], (st * kBoxes + lane) * 128,
                          rb * kBoxRows, cu.en.slot);
        else if (lane == kBoxes && p.SBB > 0) {
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
  ring.n = n;
}

// The producer's copies still in flight land before the CTA exits (waits
// with the default limit, whatever limit the operational waits had).
MOE_DEV void produce_drain(const Smem& S, int D, const Ring& ring, int* err) {
  if ((threadIdx.x & 31) == 0) {
    const uint32_t n = ring.n;
    const uint32_t first = n > (uint32_t)D ? n - D : 0;
    for (uint32_t i = first; i < n; ++i)
      if (!tc::mbar_wait(&S.full[i % D], (i / D) & 1)) {
        atomicExch(err, 1);
        break;
      }
  }
}

// ---------------------------------------------------------------- compute
// Warp (b, q) of the 16 compute warps takes rows 16q .. 16q + 15 of code box
// b of every stage; a unit's partial sums go to the epilogue through one of
// RS slots.  ALL: every token is staged once (phase 1, N <= 8), so no
// activation-buffer waits.
// mk (may be null): warp 0 stamps the global timer when its first stage has
// landed (mk[0]) and when it has consumed its last (mk[1]).
template <int FMT, int PH, bool HOST>
MOE_DEV void compute(const Geo& g, const GemvArgs& a, const SG& p, const EntryTable& T, const Range& rr,
                     const Smem& S, Small& sm, Ring& ring, long long wl, unsigned long long* mk = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool ALL = PH == 1 && p.all;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float* red = reinterpret_cast<float*>(S.base + p.off_red);
  const int bslot = warp >> 2, quarter = warp & 3, gq = lane >> 2;
  uint32_t n = ring.n, us = ring.us, bs = ring.bs;
  Cursor cu;
  cursor_init(cu, rr);
  while (cursor_next(cu, g, a, T, p, rr)) {
    const int xb = bs % p.XB;
    if (!ALL) wait_or_abort(&S.xfull[xb], (bs / p.XB) & 1, &sm.abort, a.err, wl);
    const uint2* xs = reinterpret_cast<const uint2*>(S.base + p.off_x + (size_t)xb * p.xbytes);
    for (int u = cu.ue0; u < cu.ue1; ++u) {
      for (int st = 0; st < p.NS; ++st, ++n) {
        const int slot = n % p.D;
        const bool ok = wait_or_abort(&S.full[slot], (n / p.D) & 1, &sm.abort, a.err, wl);
        if (mk && warp == 0 && lane == 0 && n == ring.n) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(mk[0]));
        const int kb = st * kBoxes + bslot;
        if (HOST && ok && cu.en.ex >= 0)
          host_part(g, p, a, cu.en, PH == 1 ? u / p.RB : 2, PH == 1 ? u % p.RB : u, st,
                    S.base + (size_t)slot * p.stage_bytes, warp, lane);
        if (ok && kb < p.KB) {
          const uint8_t* stg = S.base + (size_t)slot * p.stage_bytes;
          const uint8_t* cs = stg + (size_t)bslot * kBoxBytes + quarter * (16 * kBoxRowBytes);
          const uint8_t* sc = stg + p.codes_bytes + (16 * quarter + gq) * p.srow + (p.smode ? bslot : kb) * p.SBB;
          const int nvb = min(8, (p.K - kb * p.bk) / 32);
          const uint2* xk = xs + (size_t)kb * 2 * p.bk;   // bk / 16 MMA steps x 32 lanes
          if (FMT == MOE_MXFP4) tile_mx(cs, sc, sc + 8 * p.srow, xk, nvb, lane, acc);
          else if (FMT == MOE_NVFP4) tile_nv(cs, sc, sc + 8 * p.srow, xk, nvb, lane, acc);
          else if (FMT == MOE_MXFP8) tile_mx8(cs, sc, sc + 8 * p.srow, xk, lane, acc);
          else tile_bf16(cs, xk, lane, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
      }
      // unit done: hand the partial sums to the epilogue
      const int r = us % p.RS;
      if (us >= (uint32_t)p.RS) wait_or_abort(&S.rempty[r], (us / p.RS - 1) & 1, &sm.abort, a.err, wl);
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
      ++bs;   // (ALL blocks use no activation buffer of the ring)
    }
  }
  if (mk && warp == 0 && lane == 0 && n != ring.n) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(mk[1]));
  ring.n = n;
  ring.us = us;
  ring.bs = bs;
}

// ---------------------------------------------------------------- epilogue
// The 3 epilogue warps (threads te = 0 .. kET - 1) add the four partial sums
// of each output in a fixed order (deterministic), apply the token and tensor
// scales and write a, u (phase 1, with per-row maxima) or O (phase 2), and
// stage the activations of the blocks ahead (XB buffers).  first_staged: the
// range's first block was staged by the caller into buffer ring.bs % XB.
template <int FMT, int PH, bool HOST>
MOE_DEV void reduce(const Geo& g, const GemvArgs& a, const SG& p, const EntryTable& T, const Range& rr,
                    const Smem& S, Small& sm, Ring& ring, bool first_staged, const __nv_bfloat16* __restrict__ x,
                    const int* __restrict__ xexp, float* __restrict__ h, float* __restrict__ O, long long wl,
                    unsigned long long* mk = nullptr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool ALL = PH == 1 && p.all;
  const int te = threadIdx.x - (kCW + 1) * 32;   // 0 .. kET - 1
  const int ew_ = warp - (kCW + 1);              // epilogue warp 0 .. kEW - 1
  const float* red = reinterpret_cast<const float*>(S.base + p.off_red);
  // stage block number bs_st into its buffer once that buffer is free
  auto stage = [&](const Cursor& c, uint32_t bs_st) {
    const int xb = bs_st % p.XB;
    epi_sync();   // the previous staging's token list and exponents are no longer read
    if (bs_st >= (uint32_t)p.XB) wait_or_abort(&S.xempty[xb], (bs_st / p.XB - 1) & 1, &sm.abort, a.err, wl);
    stage_block<FMT, PH>(g, a, p, c.en, c.tg, reinterpret_cast<uint2*>(S.base + p.off_x + (size_t)xb * p.xbytes),
                         sm.sexp[xb], sm.stok, x, xexp, h, te, kET, 1);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.xfull[xb]);
  };
  Cursor cs, cr;   // staging runs XB blocks ahead of the reduction
  cursor_init(cs, rr);
  cursor_init(cr, rr);
  uint32_t bs_st = ring.bs, bs_rd = ring.br, us = ring.us;
  if (!ALL) {
    int i = 0;
    if (first_staged) {
      cursor_next(cs, g, a, T, p, rr);
      ++bs_st;
      i = 1;
    }
    for (; i < p.XB; ++i) {
      if (cursor_next(cs, g, a, T, p, rr)) stage(cs, bs_st++);
      // mk (may be null): the first block staged, stamped by thread 0
      if (mk && i == 0 && te == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(mk[0]));
    }
  }
  while (cursor_next(cr, g, a, T, p, rr)) {
    const int xb = bs_rd % p.XB;
    const int nt = ALL ? cr.en.nrows : min(kTG, cr.en.nrows - cr.tg * kTG);
    const int rowt = cr.en.row0 + cr.tg * kTG;
    if (ALL) {
      // the entry's tokens (all N tokens are staged; entries pick theirs)
      epi_sync();
      if (te < nt)
        sm.stok[te] = cr.en.shared ? te : (te == 0 && cr.en.tok0 >= 0) ? cr.en.tok0 : a.tok_of[rowt + te];
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
      const bool ok = wait_or_abort(&S.rfull[r], (us / p.RS) & 1, &sm.abort, a.err, wl);
      const float4* rs = reinterpret_cast<const float4*>(red + (size_t)r * (p.rbytes / 4));
      // warp w takes tokens w, w + kEW, ...; lane c takes columns c, c + 32 of the block
      for (int tk = ew_; ok && tk < nt; tk += kEW) {
        // column of this row's token among the staged ones
        const int cc = ALL ? sm.stok[tk] : tk;
        const float sc = pow2i(ALL ? sm.sexp[0][cc] : sm.sexp[xb][tk]) * ts;
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
      if (cursor_next(cs, g, a, T, p, rr)) stage(cs, bs_st++);
    }
  }
  ring.bs = ALL ? ring.bs : bs_st;
  ring.br = ALL ? ring.br : bs_rd;
  ring.us = us;
}

}  // namespace gv
}  // namespace moe
