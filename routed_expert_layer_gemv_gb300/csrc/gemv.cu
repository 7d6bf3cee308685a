// Decode expert FFN: grouped GEMV over the experts of one work range, read
// through the slot table, FP4 weights dequantised in registers.
//
// Decode moves each routed expert's weights once per step for a handful of
// tokens, so the kernel is bound by HBM bandwidth (the pages' decode is bound
// by the bytes each step must move: "FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).  Design:
//  * work unit = (expert entry, block of output rows); one CTA per unit, grid
//    sized for the most entries a range can hold, extra CTAs exit at once, so
//    a launch needs no host knowledge of the routing (the range is resolved
//    from the step record on the device);
//  * each lane owns fixed 16-byte chunks (32 E2M1 codes = one MXFP4 block, or
//    two NVFP4 blocks) of a row and issues all its 128-bit loads before the
//    activations are staged, so the weight stream is in flight meanwhile;
//  * codes -> f16x2 with cvt.rn.f16x2.e2m1x2 (exact), products with the
//    sm_100+ mixed fma.rn.f32.f16 into fp32, block scale applied per chunk;
//  * activations live in shared memory as f16, scaled per token by a power of
//    two (amax in [2^14, 2^15)) so no value overflows; the 16-byte pieces are
//    XOR-swizzled so the 8 lanes of a shared-memory phase hit distinct banks;
//  * row sums are reduced across the G lanes of a row with shuffles, in a
//    fixed order (deterministic).
// Phase 1: a = W_g x, u = W_u x, h = SiLU(a) * u  (fp32, [rows, d_ff]).
// Phase 2: O = W_d h                           (fp32, [rows, d_model]).
#include "common.cuh"

namespace moe {

namespace {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;

MOE_DEV uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// two mixed-precision FMAs from packed f16 pairs
MOE_DEV void fma2(float& acc, uint32_t w2, uint32_t x2) {
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
      : "+f"(acc) : "r"(w2), "r"(x2));
}

// physical 16-byte slot of logical piece q (0..3) of chunk c in a token row
MOE_DEV int swz(int c, int q) { return 4 * c + (q ^ ((c >> 1) & 3)); }

MOE_DEV float pow2i(int s) { return __int_as_float((127 + s) << 23); }  // |s| <= 126

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

// Dot products of one 16-byte weight chunk with T token pieces in shared
// memory; adds (scaled) into acc[t].
template <int T>
MOE_DEV void chunk_fma(const uint4& w, const uint4* xs, int xstride, int c, int n,
                       int fmt, uint32_t sc, float* acc) {
  uint32_t wh[16];
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int b = 0; b < 4; ++b) wh[4 * q + b] = e2m1x2_to_f16x2((ww[q] >> (8 * b)) & 0xffu);
  float s0, s1;
  if (fmt == MOE_MXFP4) { s0 = e8m0_to_f32(sc & 0xffu); s1 = s0; }
  else { s0 = e4m3_to_f32(sc & 0xffu); s1 = e4m3_to_f32((sc >> 8) & 0xffu); }
#pragma unroll
  for (int t = 0; t < T; ++t) {
    if (t < n) {
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 xv = xs[(size_t)t * xstride + swz(c, q)];
        float& p = q < 2 ? p0 : p1;
        fma2(p, wh[4 * q + 0], xv.x);
        fma2(p, wh[4 * q + 1], xv.y);
        fma2(p, wh[4 * q + 2], xv.z);
        fma2(p, wh[4 * q + 3], xv.w);
      }
      acc[t] = fmaf(p0, s0, fmaf(p1, s1, acc[t]));
    }
  }
}

MOE_DEV float group_sum(float v, int G) {
  for (int o = G >> 1; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MOE_DEV uint32_t load_scale(const uint8_t* sp, int fmt) {
  if (fmt == MOE_MXFP4) return *sp;
  return *reinterpret_cast<const uint16_t*>(sp);
}

// ---------------------------------------------------------------- phase 1
// Unit = (entry, 8 warps x (32/G) rows of d_ff).  A lane keeps up to kCPLM
// chunks of its gate row and of its up row in registers; longer rows loop.
constexpr int kCPLM = 4;

template <int T>
MOE_DEV void stage_x(const GemvArgs& a, const Entry& en, const __nv_bfloat16* __restrict__ x,
                     const int* __restrict__ xexp, int K, int t0, int n, uint4* xs, int* sexp_s) {
  const int xstride = K / 8;
  for (int v = threadIdx.x; v < n * xstride; v += kGemvThreads) {
    const int t = v / xstride, L = v % xstride;
    const int tok = row_token(a, en, en.row0 + t0 + t);
    const uint4 raw = reinterpret_cast<const uint4*>(x + (size_t)tok * K)[L];
    const int s = xexp[tok];
    if (L == 0) sexp_s[t] = s;
    const float sc = pow2i(-s);
    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(rw[i] << 16) * sc;
      const float hi = __uint_as_float(rw[i] & 0xffff0000u) * sc;
      const __half2 hh = __floats2half2_rn(lo, hi);
      o[i] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    xs[(size_t)t * xstride + swz(L >> 2, L & 3)] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int T>
__global__ void __launch_bounds__(kGemvThreads)
gemv_gateup_kernel(Geo g, GemvArgs a, const __nv_bfloat16* __restrict__ x,
                   const int* __restrict__ xexp, float* __restrict__ h) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  __shared__ int sexp_s[T];
  const int K = g.d;
  const int chunks = K / 32;
  const int G = min(32, chunks & -chunks);      // lanes per row (power of 2)
  const int cpl = chunks / G;                   // chunks per lane
  const int rpw = 32 / G;                       // rows per warp
  const int rpc = kGemvWarps * rpw;             // rows per CTA
  const int upe = g.f / rpc;                    // units per entry
  const int ent = blockIdx.x / upe, rb = blockIdx.x % upe;
  Entry en;
  if (!get_entry(g, a, ent, en)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = rb * rpc + warp * rpw + lane / G;   // row of d_ff
  const int sbpc = g.fmt == MOE_MXFP4 ? 1 : 2;      // scale bytes per chunk
  const uint8_t* gc = en.w + g.off_codes[0] + (size_t)r * (K / 2);
  const uint8_t* uc = en.w + g.off_codes[1] + (size_t)r * (K / 2);
  const uint8_t* gs = en.w + g.off_scales[0] + (size_t)r * (K / g.blk);
  const uint8_t* us = en.w + g.off_scales[1] + (size_t)r * (K / g.blk);
  uint4 wg[kCPLM], wu[kCPLM];
  uint32_t sg[kCPLM], su[kCPLM];
  auto load = [&](int j0) {
#pragma unroll
    for (int j = 0; j < kCPLM; ++j) {
      if (j0 + j < cpl) {
        const int c = (lane % G) + G * (j0 + j);
        wg[j] = ldg_stream(gc + (size_t)c * 16);
        wu[j] = ldg_stream(uc + (size_t)c * 16);
        sg[j] = load_scale(gs + (size_t)c * sbpc, g.fmt);
        su[j] = load_scale(us + (size_t)c * sbpc, g.fmt);
      }
    }
  };
  load(0);   // the weight stream is in flight while x is staged
  const float* ts = reinterpret_cast<const float*>(en.w + g.off_tscale);
  const float tg = ts[0], tu = ts[1];
  const int xstride = K / 8;
  for (int t0 = 0; t0 < en.nrows; t0 += T) {
    const int n = min(T, en.nrows - t0);
    __syncthreads();
    stage_x<T>(a, en, x, xexp, K, t0, n, xs, sexp_s);
    __syncthreads();
    float ag[T], au[T];
#pragma unroll
    for (int t = 0; t < T; ++t) { ag[t] = 0.f; au[t] = 0.f; }
    for (int j0 = 0; j0 < cpl; j0 += kCPLM) {
      if (t0 > 0 || j0 > 0) load(j0);
#pragma unroll
      for (int j = 0; j < kCPLM; ++j) {
        if (j0 + j < cpl) {
          const int c = (lane % G) + G * (j0 + j);
          chunk_fma<T>(wg[j], xs, xstride, c, n, g.fmt, sg[j], ag);
          chunk_fma<T>(wu[j], xs, xstride, c, n, g.fmt, su[j], au);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      if (t < n) {
        const float s = pow2i(sexp_s[t]);
        const float av = group_sum(ag[t], G) * s * tg;
        const float uv = group_sum(au[t], G) * s * tu;
        if ((lane % G) == 0) {
          const float silu = av / (1.0f + expf(-av));
          h[(size_t)(en.row0 + t0 + t) * g.f + r] = silu * uv;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- phase 2
// Unit = (entry, 8 warps x (32/G) x kP2 rows of d_model).  h rows staged as
// f16 with a per-row power-of-two scale (computed here from the row's amax).
constexpr int kP2 = 2;

template <int T>
__global__ void __launch_bounds__(kGemvThreads)
gemv_down_kernel(Geo g, GemvArgs a, const float* __restrict__ h, float* __restrict__ O) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint4* xs = reinterpret_cast<uint4*>(smem_raw);
  __shared__ int sexp_s[T];
  const int K = g.f;
  const int chunks = K / 32;
  const int G = min(32, chunks & -chunks);
  const int cpl = chunks / G;
  const int rpw = 32 / G;
  const int rpc = kGemvWarps * rpw * kP2;
  const int upe = g.d / rpc;
  const int ent = blockIdx.x / upe, rb = blockIdx.x % upe;
  Entry en;
  if (!get_entry(g, a, ent, en)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sbpc = g.fmt == MOE_MXFP4 ? 1 : 2;
  const uint8_t* dc[kP2];
  const uint8_t* ds[kP2];
  int rows[kP2];
#pragma unroll
  for (int p = 0; p < kP2; ++p) {
    rows[p] = rb * rpc + (p * kGemvWarps + warp) * rpw + lane / G;
    dc[p] = en.w + g.off_codes[2] + (size_t)rows[p] * (K / 2);
    ds[p] = en.w + g.off_scales[2] + (size_t)rows[p] * (K / g.blk);
  }
  uint4 wd[kP2][kCPLM];
  uint32_t sd[kP2][kCPLM];
  auto load = [&](int j0) {
#pragma unroll
    for (int p = 0; p < kP2; ++p)
#pragma unroll
      for (int j = 0; j < kCPLM; ++j)
        if (j0 + j < cpl) {
          const int c = (lane % G) + G * (j0 + j);
          wd[p][j] = ldg_stream(dc[p] + (size_t)c * 16);
          sd[p][j] = load_scale(ds[p] + (size_t)c * sbpc, g.fmt);
        }
  };
  load(0);
  const float td = reinterpret_cast<const float*>(en.w + g.off_tscale)[2];
  const int xstride = K / 8;
  for (int t0 = 0; t0 < en.nrows; t0 += T) {
    const int n = min(T, en.nrows - t0);
    __syncthreads();
    // one warp per token: amax, exponent, f16 conversion into shared memory
    for (int t = warp; t < n; t += kGemvWarps) {
      const float* hr = h + (size_t)(en.row0 + t0 + t) * K;
      float m = 0.f;
      for (int i = lane; i < K; i += 32) m = fmaxf(m, fabsf(hr[i]));
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      int s = 0;
      if (m > 0.f) {
        int ex;
        frexpf(m, &ex);
        s = max(-100, min(100, ex - 15));
      }
      if (lane == 0) sexp_s[t] = s;
      const float sc = pow2i(-s);
      for (int L = lane; L < xstride; L += 32) {
        const float4 v0 = reinterpret_cast<const float4*>(hr)[2 * L];
        const float4 v1 = reinterpret_cast<const float4*>(hr)[2 * L + 1];
        const __half2 a0 = __floats2half2_rn(v0.x * sc, v0.y * sc);
        const __half2 a1 = __floats2half2_rn(v0.z * sc, v0.w * sc);
        const __half2 a2 = __floats2half2_rn(v1.x * sc, v1.y * sc);
        const __half2 a3 = __floats2half2_rn(v1.z * sc, v1.w * sc);
        xs[(size_t)t * xstride + swz(L >> 2, L & 3)] =
            make_uint4(*reinterpret_cast<const uint32_t*>(&a0), *reinterpret_cast<const uint32_t*>(&a1),
                       *reinterpret_cast<const uint32_t*>(&a2), *reinterpret_cast<const uint32_t*>(&a3));
      }
    }
    __syncthreads();
    float acc[kP2][T];
#pragma unroll
    for (int p = 0; p < kP2; ++p)
#pragma unroll
      for (int t = 0; t < T; ++t) acc[p][t] = 0.f;
    for (int j0 = 0; j0 < cpl; j0 += kCPLM) {
      if (t0 > 0 || j0 > 0) load(j0);
#pragma unroll
      for (int p = 0; p < kP2; ++p)
#pragma unroll
        for (int j = 0; j < kCPLM; ++j)
          if (j0 + j < cpl) {
            const int c = (lane % G) + G * (j0 + j);
            chunk_fma<T>(wd[p][j], xs, xstride, c, n, g.fmt, sd[p][j], acc[p]);
          }
    }
#pragma unroll
    for (int p = 0; p < kP2; ++p)
#pragma unroll
      for (int t = 0; t < T; ++t)
        if (t < n) {
          const float v = group_sum(acc[p][t], G) * pow2i(sexp_s[t]) * td;
          if ((lane % G) == 0) O[(size_t)(en.row0 + t0 + t) * g.d + rows[p]] = v;
        }
  }
}

int tok_bucket(int N) { return N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : 8; }

template <int T>
cudaError_t launch_t(const Geo& g, const GemvArgs& a, const __nv_bfloat16* x, const int* xexp,
                     float* h, float* O, int n_ent_max, cudaStream_t st, const cudaEvent_t* ev) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(gemv_gateup_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    cudaFuncSetAttribute(gemv_down_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  const int c1 = g.d / 32, G1 = min(32, c1 & -c1);
  const int grid1 = n_ent_max * (g.f / (kGemvWarps * (32 / G1)));
  if (ev) cudaEventRecord(ev[0], st);
  if (grid1 > 0)
    gemv_gateup_kernel<T><<<grid1, kGemvThreads, (size_t)T * g.d * 2, st>>>(g, a, x, xexp, h);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (ev) cudaEventRecord(ev[1], st);
  const int c2 = g.f / 32, G2 = min(32, c2 & -c2);
  const int grid2 = n_ent_max * (g.d / (kGemvWarps * (32 / G2) * kP2));
  if (ev) cudaEventRecord(ev[2], st);
  if (grid2 > 0) gemv_down_kernel<T><<<grid2, kGemvThreads, (size_t)T * g.f * 2, st>>>(g, a, h, O);
  if (ev) cudaEventRecord(ev[3], st);
  return cudaGetLastError();
}

}  // namespace

// Shapes the decode kernels accept: the CTA row blocks must tile d_ff (phase
// 1) and d_model (phase 2) exactly, and 8 staged token rows must fit in
// shared memory.
bool gemv_shape_ok(const Geo& g) {
  const int c1 = g.d / 32, c2 = g.f / 32;
  const int G1 = min(32, c1 & -c1), G2 = min(32, c2 & -c2);
  if (g.f % (kGemvWarps * (32 / G1)) != 0) return false;
  if (g.d % (kGemvWarps * (32 / G2) * kP2) != 0) return false;
  return (size_t)8 * (size_t)(g.d > g.f ? g.d : g.f) * 2 <= 200 * 1024;
}

cudaError_t launch_gemv_decode(const Geo& g, const GemvArgs& a, const __nv_bfloat16* x,
                               const int* xexp, float* h, float* O, int n_ent_max,
                               cudaStream_t st, const cudaEvent_t* ev) {
  switch (tok_bucket(a.N)) {
    case 1: return launch_t<1>(g, a, x, xexp, h, O, n_ent_max, st, ev);
    case 2: return launch_t<2>(g, a, x, xexp, h, O, n_ent_max, st, ev);
    case 4: return launch_t<4>(g, a, x, xexp, h, O, n_ent_max, st, ev);
    default: return launch_t<8>(g, a, x, xexp, h, O, n_ent_max, st, ev);
  }
}

}  // namespace moe
