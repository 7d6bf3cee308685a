// Decode expert FFN: split-K grouped GEMV over the experts of one work range,
// read through the slot table, FP4 weights dequantised in registers.
//
// Decode moves each routed expert's weights once per step for a handful of
// tokens, so the kernel is bound by HBM bandwidth (the pages' decode is bound
// by the bytes each step must move: "FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).  Design:
//  * CTA = (expert entry, 16 output rows); its KS warps split K, each warp
//    owning kTPW tiles of 128 K, so a CTA has all of its weight loads in flight
//    before it touches the activations; partial sums are reduced across the
//    warps in shared memory in a fixed order (deterministic);
//  * the token dimension goes through tensor-core MMAs (mma.sync m16n8k16,
//    f16 x f16 -> f32): the 4 lanes of a row each load one 32-bit word of every
//    16-byte chunk (32 E2M1 codes = one MXFP4 block), convert it with
//    cvt.rn.f16x2.e2m1x2 (exact) straight into the A fragment, and the
//    activations are staged in shared memory in the matching permuted K order,
//    so no lane exchanges are needed and every MMA stays inside one scale
//    block.  Instructions per byte of weight are flat up to 8 tokens per MMA;
//  * the block scale is applied to each block's MMA sum in fp32; NVFP4 blocks
//    (16 codes) split each MMA into two lane-masked halves;
//  * activations are converted to f16 with a per-token power-of-two scale
//    (amax in [2^14, 2^15)), undone after the reduction, so nothing overflows.
// Phase 1: a = W_g x, u = W_u x, h = SiLU(a) * u  (fp32, [rows, d_ff]).
// Phase 2: O = W_d h                           (fp32, [rows, d_model]).
#include "common.cuh"

namespace moe {

namespace {

constexpr int kMaxWarps = 16;

MOE_DEV uint32_t ldg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

MOE_DEV uint2 ldg64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

MOE_DEV float pow2i(int s) { return __int_as_float((127 + s) << 23); }  // |s| <= 126

MOE_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint2 b, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

struct Entry {
  const uint8_t* w;
  int row0, nrows, shared;
};

// Resolve work entry `ent` of the launch; false if past the end.
MOE_DEV bool get_entry(const Geo& g, const GemvArgs& a, int ent, Entry& out) {
  const StepRecord* rec = a.rec;
  const int U = rec->U, nh = rec->n_hit, S = rec->S;
  int b = 0, e = 0;
  if (a.mode == kRangeHits) { b = 0; e = nh; }
  else if (a.mode == kRangeWaveMisses) { b = max(nh, a.wave * S); e = min((a.wave + 1) * S, U); }
  else { b = a.wave * S; e = min((a.wave + 1) * S, U); }
  const int nr = max(0, e - b);
  if (ent < nr) {
    const int acc = b + ent;
    const int ex = rec_expert(const_cast<StepRecord*>(rec))[acc];
    const int sl = rec_slot(const_cast<StepRecord*>(rec), g.E)[acc];
    if (ex < 0 || ex >= g.E || sl < 0 || sl >= g.S) return false;
    out.w = a.slots + (size_t)sl * g.ebytes;
    out.row0 = a.offsets[ex];
    out.nrows = a.offsets[ex + 1] - out.row0;
    out.shared = 0;
    return out.nrows > 0;
  }
  if (a.with_shared && ent == nr) {
    out.w = a.shared_w;
    out.row0 = a.N * g.k;
    out.nrows = a.N;
    out.shared = 1;
    return true;
  }
  return false;
}

MOE_DEV int row_token(const GemvArgs& a, const Entry& en, int row) {
  return en.shared ? row - en.row0 : a.tok_of[row];
}

// One warp's slice of a matrix: rows (g, g+8) of a 16-row group, TPW tiles of
// 128 K.  w[t][h][c] = the lane's word q of 16-byte chunk c (codes 8q..8q+7 of
// that 32-code block); s[t][h] = the tile's scale bytes of that row.
template <int FMT, int TPW>
struct Slice {
  uint32_t w[TPW][2][4];
  uint32_t s[TPW][2][FMT == MOE_MXFP4 ? 1 : 2];
};

template <int FMT, int TPW>
MOE_DEV void load_slice(Slice<FMT, TPW>& sl, const uint8_t* codes, const uint8_t* scales, int K,
                        int row, int kt0, int nkt, int q) {
#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    if (t < nkt) {
      const int kt = kt0 + t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint8_t* cb = codes + (size_t)(row + 8 * h) * (K / 2) + (size_t)kt * 64 + 4 * q;
#pragma unroll
        for (int c = 0; c < 4; ++c) sl.w[t][h][c] = ldg32(cb + 16 * c);
        if (FMT == MOE_MXFP4) {
          sl.s[t][h][0] = ldg32(scales + (size_t)(row + 8 * h) * (K / 32) + 4 * kt);
        } else {
          const uint2 v = ldg64(scales + (size_t)(row + 8 * h) * (K / 16) + 8 * kt);
          sl.s[t][h][0] = v.x;
          sl.s[t][h][FMT == MOE_MXFP4 ? 0 : 1] = v.y;
        }
      }
    }
  }
}

MOE_DEV float scale_of(int fmt, uint32_t sw, int byte) {
  const uint32_t b = (sw >> (8 * byte)) & 0xffu;
  return fmt == MOE_MXFP4 ? e8m0_to_f32(b) : e4m3_to_f32(b);
}

// A fragments of MMA step st (0, 1) of chunk c: rows g and g+8, codes
// 8q + 4 st .. + 3 of the chunk's block.
template <int FMT, int TPW>
MOE_DEV void afrag(const Slice<FMT, TPW>& sl, int t, int c, int st, uint32_t (&a)[4]) {
  const uint32_t w0 = sl.w[t][0][c] >> (16 * st), w1 = sl.w[t][1][c] >> (16 * st);
  a[0] = e2m1x2_to_f16x2(w0 & 0xffu);
  a[1] = e2m1x2_to_f16x2(w1 & 0xffu);
  a[2] = e2m1x2_to_f16x2((w0 >> 8) & 0xffu);
  a[3] = e2m1x2_to_f16x2((w1 >> 8) & 0xffu);
}

// acc[ng] += W(16 rows, this warp's K) x B(ng) for NG token groups of 8.
template <int FMT, int TPW, int NG>
MOE_DEV void slice_mma(const Slice<FMT, TPW>& sl, int kt0, int nkt, const uint2* xs, int ksteps,
                       int lane, float (&acc)[NG][4]) {
  const int q = lane & 3;
  const uint32_t mlo = q < 2 ? 0xffffffffu : 0u, mhi = ~mlo;
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    if (t < nkt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cg = (kt0 + t) * 4 + c;        // global 32-code block
        uint32_t a0[4], a1[4];
        afrag(sl, t, c, 0, a0);
        afrag(sl, t, c, 1, a1);
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const uint2 b0 = xs[((size_t)ng * ksteps + 2 * cg) * 32 + lane];
          const uint2 b1 = xs[((size_t)ng * ksteps + 2 * cg + 1) * 32 + lane];
          if (FMT == MOE_MXFP4) {
            float d[4];
            mma16816(d, a0, b0, z);
            mma16816(d, a1, b1, d);
            const float s0 = scale_of(FMT, sl.s[t][0][0], c), s1 = scale_of(FMT, sl.s[t][1][0], c);
            acc[ng][0] = fmaf(d[0], s0, acc[ng][0]);
            acc[ng][1] = fmaf(d[1], s0, acc[ng][1]);
            acc[ng][2] = fmaf(d[2], s1, acc[ng][2]);
            acc[ng][3] = fmaf(d[3], s1, acc[ng][3]);
          } else {
            // lanes q < 2 hold codes of 16-block 2c, lanes q >= 2 of block 2c+1
            uint32_t l0[4], l1[4], h0[4], h1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              l0[i] = a0[i] & mlo; l1[i] = a1[i] & mlo;
              h0[i] = a0[i] & mhi; h1[i] = a1[i] & mhi;
            }
            float dl[4], dh[4];
            mma16816(dl, l0, b0, z);
            mma16816(dl, l1, b1, dl);
            mma16816(dh, h0, b0, z);
            mma16816(dh, h1, b1, dh);
            const int wb = c >> 1, by = 2 * (c & 1);   // sub-blocks 2c, 2c+1 of the tile
            const float sl0 = scale_of(FMT, sl.s[t][0][wb], by), sh0 = scale_of(FMT, sl.s[t][0][wb], by + 1);
            const float sl1 = scale_of(FMT, sl.s[t][1][wb], by), sh1 = scale_of(FMT, sl.s[t][1][wb], by + 1);
            acc[ng][0] = fmaf(dl[0], sl0, fmaf(dh[0], sh0, acc[ng][0]));
            acc[ng][1] = fmaf(dl[1], sl0, fmaf(dh[1], sh0, acc[ng][1]));
            acc[ng][2] = fmaf(dl[2], sl1, fmaf(dh[2], sh1, acc[ng][2]));
            acc[ng][3] = fmaf(dl[3], sl1, fmaf(dh[3], sh1, acc[ng][3]));
          }
        }
      }
    }
  }
}

// Shared-memory slot of 4 consecutive activation values (real K k0, token tl)
// in B-fragment order: [group][k-step][lane] x 8 bytes, k-step = 2 * block +
// step, lane = 4 * token + q with k0 = 32 block + 8 q + 4 step.
MOE_DEV int frag_slot(int tl, int k0, int ksteps) {
  const int c = k0 >> 5, r = k0 & 31;
  const int q = r >> 3, st = (r >> 2) & 1;
  return ((tl >> 3) * ksteps + 2 * c + st) * 32 + 4 * (tl & 7) + q;
}

MOE_DEV uint2 to_f16x4(float a, float b, float c, float d) {
  const __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&lo);
  o.y = *reinterpret_cast<const uint32_t*>(&hi);
  return o;
}

// ---------------------------------------------------------------- phase 1
template <int FMT, int TPW, int NG>
__global__ void __launch_bounds__(kMaxWarps * 32)
gemv_gateup_kernel(Geo g, GemvArgs a, const __nv_bfloat16* __restrict__ x,
                   const int* __restrict__ xexp, float* __restrict__ h) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int sexp[8 * NG];
  const int K = g.d, ksteps = K / 16, nkt_all = K / 128;
  const int KS = blockDim.x >> 5;
  const int rgs = g.f / 16;
  const int ent = blockIdx.x / rgs, rg = blockIdx.x % rgs;
  Entry en;
  if (!get_entry(g, a, ent, en)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = lane & 3;
  const int kt0 = warp * TPW, nkt = min(TPW, nkt_all - kt0);
  const int row = rg * 16 + (lane >> 2);
  Slice<FMT, TPW> sg, su;
  load_slice(sg, en.w + g.off_codes[0], en.w + g.off_scales[0], K, row, kt0, nkt, q);
  load_slice(su, en.w + g.off_codes[1], en.w + g.off_scales[1], K, row, kt0, nkt, q);
  const float* ts = reinterpret_cast<const float*>(en.w + g.off_tscale);
  const float tsg = ts[0], tsu = ts[1];
  uint2* xs = reinterpret_cast<uint2*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)NG * ksteps * 256);
  const int rstride = NG * 8 + 1;
  for (int t0 = 0; t0 < en.nrows; t0 += 8 * NG) {
    const int n = min(8 * NG, en.nrows - t0);
    if (t0 > 0) {
      __syncthreads();
      load_slice(sg, en.w + g.off_codes[0], en.w + g.off_scales[0], K, row, kt0, nkt, q);
      load_slice(su, en.w + g.off_codes[1], en.w + g.off_scales[1], K, row, kt0, nkt, q);
    }
    // stage x (bf16 -> f16 scaled by 2^-xexp) in B-fragment order
    for (int v = threadIdx.x; v < n * (K / 4); v += blockDim.x) {
      const int tl = v / (K / 4), k0 = (v % (K / 4)) * 4;
      const int tok = row_token(a, en, en.row0 + t0 + tl);
      const int s = xexp[tok];
      if (k0 == 0) sexp[tl] = s;
      const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)tok * K + k0);
      const float sc = pow2i(-s);
      xs[frag_slot(tl, k0, ksteps)] =
          to_f16x4(__uint_as_float(raw.x << 16) * sc, __uint_as_float(raw.x & 0xffff0000u) * sc,
                   __uint_as_float(raw.y << 16) * sc, __uint_as_float(raw.y & 0xffff0000u) * sc);
    }
    __syncthreads();
    float ag[NG][4], au[NG][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 4; ++j) { ag[ng][j] = 0.f; au[ng][j] = 0.f; }
    slice_mma<FMT, TPW, NG>(sg, kt0, nkt, xs, ksteps, lane, ag);
    slice_mma<FMT, TPW, NG>(su, kt0, nkt, xs, ksteps, lane, au);
    float* my = red + (size_t)(warp * 32 + lane) * rstride;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 4; ++j) { my[ng * 8 + j] = ag[ng][j]; my[ng * 8 + 4 + j] = au[ng][j]; }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tk = 8 * ng + 2 * q + (j & 1);
          const int r = row + 8 * (j >> 1);
          float sa = 0.f, su_ = 0.f;
          for (int w = 0; w < KS; ++w) {
            sa += red[(size_t)(w * 32 + lane) * rstride + ng * 8 + j];
            su_ += red[(size_t)(w * 32 + lane) * rstride + ng * 8 + 4 + j];
          }
          if (tk < n) {
            const float sc = pow2i(sexp[tk]);
            const float av = sa * sc * tsg, uv = su_ * sc * tsu;
            h[(size_t)(en.row0 + t0 + tk) * g.f + r] = av / (1.0f + expf(-av)) * uv;
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- phase 2
template <int FMT, int TPW, int NG>
__global__ void __launch_bounds__(kMaxWarps * 32)
gemv_down_kernel(Geo g, GemvArgs a, const float* __restrict__ h, float* __restrict__ O) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int sexp[8 * NG];
  const int K = g.f, ksteps = K / 16, nkt_all = K / 128;
  const int KS = blockDim.x >> 5;
  const int rgs = g.d / 16;
  const int ent = blockIdx.x / rgs, rg = blockIdx.x % rgs;
  Entry en;
  if (!get_entry(g, a, ent, en)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = lane & 3;
  const int kt0 = warp * TPW, nkt = min(TPW, nkt_all - kt0);
  const int row = rg * 16 + (lane >> 2);
  Slice<FMT, TPW> sd;
  load_slice(sd, en.w + g.off_codes[2], en.w + g.off_scales[2], K, row, kt0, nkt, q);
  const float tsd = reinterpret_cast<const float*>(en.w + g.off_tscale)[2];
  uint2* xs = reinterpret_cast<uint2*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)NG * ksteps * 256);
  const int rstride = NG * 4 + 1;
  for (int t0 = 0; t0 < en.nrows; t0 += 8 * NG) {
    const int n = min(8 * NG, en.nrows - t0);
    if (t0 > 0) {
      __syncthreads();
      load_slice(sd, en.w + g.off_codes[2], en.w + g.off_scales[2], K, row, kt0, nkt, q);
    }
    // per-row power-of-two exponent of h, then h -> f16 in B-fragment order
    for (int tl = warp; tl < n; tl += KS) {
      const float* hr = h + (size_t)(en.row0 + t0 + tl) * K;
      float m = 0.f;
      for (int i = lane; i < K; i += 32) m = fmaxf(m, fabsf(hr[i]));
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      int s = 0;
      if (m > 0.f) {
        int ex;
        frexpf(m, &ex);
        s = max(-100, min(100, ex - 15));
      }
      if (lane == 0) sexp[tl] = s;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < n * (K / 4); v += blockDim.x) {
      const int tl = v / (K / 4), k0 = (v % (K / 4)) * 4;
      const float4 hv = *reinterpret_cast<const float4*>(h + (size_t)(en.row0 + t0 + tl) * K + k0);
      const float sc = pow2i(-sexp[tl]);
      xs[frag_slot(tl, k0, ksteps)] = to_f16x4(hv.x * sc, hv.y * sc, hv.z * sc, hv.w * sc);
    }
    __syncthreads();
    float acc[NG][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[ng][j] = 0.f;
    slice_mma<FMT, TPW, NG>(sd, kt0, nkt, xs, ksteps, lane, acc);
    float* my = red + (size_t)(warp * 32 + lane) * rstride;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 4; ++j) my[ng * 4 + j] = acc[ng][j];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tk = 8 * ng + 2 * q + (j & 1);
          const int r = row + 8 * (j >> 1);
          float sum = 0.f;
          for (int w = 0; w < KS; ++w) sum += red[(size_t)(w * 32 + lane) * rstride + ng * 4 + j];
          if (tk < n) O[(size_t)(en.row0 + t0 + tk) * g.d + r] = sum * pow2i(sexp[tk]) * tsd;
        }
      }
    }
  }
}

// Warps per CTA and tiles per warp for a K: the fewest tiles per warp (2 or
// 4) that keep the CTA at <= kMaxWarps warps.
void split_k(int K, int* ks, int* tpw) {
  const int nkt = K / 128;
  *tpw = (nkt + 1) / 2 <= kMaxWarps ? 2 : 4;
  *ks = (nkt + *tpw - 1) / *tpw;
}

size_t smem_bytes(int K, int ks, int ng, int per_token_vals) {
  return (size_t)ng * (K / 16) * 256 + (size_t)ks * 32 * (ng * per_token_vals + 1) * 4;
}

template <int FMT, int TPW, int NG>
cudaError_t launch_fmt(const Geo& g, const GemvArgs& a, const __nv_bfloat16* x, const int* xexp,
                       float* h, float* O, int n_ent_max, cudaStream_t st, const cudaEvent_t* ev,
                       int phase_mask) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e1 = cudaFuncSetAttribute(gemv_gateup_kernel<FMT, TPW, NG>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    cudaError_t e2 = cudaFuncSetAttribute(gemv_down_kernel<FMT, TPW, NG>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e1 != cudaSuccess) return e1;
    if (e2 != cudaSuccess) return e2;
    attr_set = true;
  }
  cudaError_t err = cudaSuccess;
  if (phase_mask & 1) {
    int ks, tpw;
    split_k(g.d, &ks, &tpw);
    const int grid = n_ent_max * (g.f / 16);
    if (ev) cudaEventRecord(ev[0], st);
    if (grid > 0)
      gemv_gateup_kernel<FMT, TPW, NG><<<grid, ks * 32, smem_bytes(g.d, ks, NG, 8), st>>>(g, a, x, xexp, h);
    err = cudaGetLastError();
    if (ev) cudaEventRecord(ev[1], st);
    if (err != cudaSuccess) return err;
  }
  if (phase_mask & 2) {
    int ks, tpw;
    split_k(g.f, &ks, &tpw);
    const int grid = n_ent_max * (g.d / 16);
    if (ev) cudaEventRecord(ev[2], st);
    if (grid > 0)
      gemv_down_kernel<FMT, TPW, NG><<<grid, ks * 32, smem_bytes(g.f, ks, NG, 4), st>>>(g, a, h, O);
    err = cudaGetLastError();
    if (ev) cudaEventRecord(ev[3], st);
  }
  return err;
}

template <int FMT, int NG>
cudaError_t launch_ng(const Geo& g, const GemvArgs& a, const __nv_bfloat16* x, const int* xexp,
                      float* h, float* O, int n_ent_max, cudaStream_t st, const cudaEvent_t* ev) {
  // the two phases may need different tiles per warp (K = d_model, then d_ff)
  int ks1, tpw1, ks2, tpw2;
  split_k(g.d, &ks1, &tpw1);
  split_k(g.f, &ks2, &tpw2);
  cudaError_t err = tpw1 == 2 ? launch_fmt<FMT, 2, NG>(g, a, x, xexp, h, O, n_ent_max, st, ev, 1)
                              : launch_fmt<FMT, 4, NG>(g, a, x, xexp, h, O, n_ent_max, st, ev, 1);
  if (err != cudaSuccess) return err;
  return tpw2 == 2 ? launch_fmt<FMT, 2, NG>(g, a, x, xexp, h, O, n_ent_max, st, ev, 2)
                   : launch_fmt<FMT, 4, NG>(g, a, x, xexp, h, O, n_ent_max, st, ev, 2);
}

int pick_ng(const Geo& g, int N) {
  if (N <= 8) return 1;
  int ks, tpw;
  split_k(g.d, &ks, &tpw);
  return smem_bytes(g.d, ks, 2, 8) <= 200 * 1024 ? 2 : 1;
}

}  // namespace

// Shapes the decode kernels accept: K = d_model and d_ff up to 8192 (16 warps
// x 4 tiles of 128) and the staged activations of one token group in shared
// memory.
bool gemv_shape_ok(const Geo& g) {
  if (g.d > 8192 || g.f > 8192) return false;
  int ks, tpw;
  split_k(g.d, &ks, &tpw);
  if (smem_bytes(g.d, ks, 1, 8) > 220 * 1024) return false;
  split_k(g.f, &ks, &tpw);
  return smem_bytes(g.f, ks, 1, 4) <= 220 * 1024;
}

cudaError_t launch_gemv_decode(const Geo& g, const GemvArgs& a, const __nv_bfloat16* x,
                               const int* xexp, float* h, float* O, int n_ent_max,
                               cudaStream_t st, const cudaEvent_t* ev) {
  const int ng = pick_ng(g, a.N);
  if (g.fmt == MOE_MXFP4)
    return ng == 1 ? launch_ng<MOE_MXFP4, 1>(g, a, x, xexp, h, O, n_ent_max, st, ev)
                   : launch_ng<MOE_MXFP4, 2>(g, a, x, xexp, h, O, n_ent_max, st, ev);
  return ng == 1 ? launch_ng<MOE_NVFP4, 1>(g, a, x, xexp, h, O, n_ent_max, st, ev)
                 : launch_ng<MOE_NVFP4, 2>(g, a, x, xexp, h, O, n_ent_max, st, ev);
}

}  // namespace moe
