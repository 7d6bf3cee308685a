// Router: logits = x W_r^T (+ b) in fp32, then per token the k largest
// logits (ties -> lower expert id), gates = softmax restricted to them (or
// the full-softmax probabilities), emitted in ascending expert order.
//
// The FreeToken pages do not define the router; they only say routing picks
// a few experts per token and varies per layer and token ("FreeToken：把 284B
// MoE 塞进游戏 PC", zhichai.net, §二 "Decode" paragraph; ananclaw.com
// explainer, §核心方法 1).  This is the standard softmax top-k router.
//
// logits kernel: one warp per expert, a tile of TN tokens per CTA held in
// shared memory as bf16; W_r rows stream through with 128-bit loads.  The
// warp reduces TN dot products with shuffles.  CTA (0, tile) also writes each
// token's power-of-two exponent used by the expert GEMV to convert x to f16
// without overflow.
// topk: one warp per token on its logits row staged in shared memory; k rounds
// of a warp-wide argmax.  For decode-sized batches (router_dec_kernel: one
// CTA per expert, K split over its warps) the last CTA runs it, so routing is
// one launch.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;

MOE_DEV bool better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

// One warp: the k largest of the logits row L (shared memory, E <= 1024
// entries; ties to the lower expert id), gates, written in ascending id order.
MOE_DEV void topk_row(const float* L, int E, int k, int norm_topk, int* idx, float* gates) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit i: entry lane + 32 i already selected
  int my_e = -1;
  float my_v = 0.f, top = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      const float v = L[e];
      if (better(v, e, bv, be)) { bv = v; be = e; }
    }
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (j == 0) top = bv;
    if (lane == j) { my_e = be; my_v = bv; }
  }
  // gates (fp32): softmax over the selected logits, or the full softmax
  const float num = lane < k ? expf(my_v - top) : 0.f;
  float den = 0.f;
  if (norm_topk) {
    den = num;
  } else {
    for (int e = lane; e < E; e += 32) den += expf(L[e] - top);
  }
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  // ascending expert order: rank of my_e among the k selected
  int rank = 0;
  for (int i = 0; i < k; ++i) {
    const int oe = __shfl_sync(0xffffffffu, my_e, i);
    rank += (lane < k && oe < my_e) ? 1 : 0;
  }
  if (lane < k) {
    idx[rank] = my_e;
    gates[rank] = num / den;
  }
}

// Stage row t of the logits into this warp's shared row, bypassing L1 (the
// row may have been written by other CTAs of the same launch).
MOE_DEV void stage_logits(const float* logits, int t, int E, float* Ls) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) Ls[e] = __ldcg(logits + (size_t)t * E + e);
  __syncwarp();
}

// logits = x W_r^T (+ b): one warp per expert, TN tokens per CTA held in
// shared memory.  CTA (0, tile) also writes each token's f16 exponent.  With
// FUSE, the last CTA to finish (a device counter, reset by that CTA) runs the
// top-k of every token, so decode-sized batches route in one launch.
template <int TN, bool FUSE>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(const __nv_bfloat16* __restrict__ x, int N, int d, int E,
                     const float* __restrict__ Wr, const float* __restrict__ bias,
                     float* __restrict__ logits, int* __restrict__ xexp, int k, int norm_topk,
                     int* __restrict__ idx, float* __restrict__ gates,
                     unsigned int* __restrict__ counter) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [TN][d]
  __shared__ bool last;
  const int t0 = blockIdx.y * TN;
  const int nt = min(TN, N - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // stage the token tile (16-byte vectors; d is a multiple of 128)
  const int vec_per_row = d / 8;
  for (int v = threadIdx.x; v < TN * vec_per_row; v += blockDim.x) {
    const int t = v / vec_per_row, c = v % vec_per_row;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (t < nt) val = reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * d)[c];
    reinterpret_cast<uint4*>(xs + (size_t)t * d)[c] = val;
  }
  __syncthreads();

  if (blockIdx.x == 0 && xexp != nullptr) {
    // per-token exponent s with amax(|x|) * 2^-s in [2^14, 2^15)
    for (int t = warp; t < nt; t += kRouterWarps) {
      float m = 0.f;
      for (int i = lane; i < d; i += 32) m = fmaxf(m, fabsf(__bfloat162float(xs[(size_t)t * d + i])));
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) {
        int s = 0;
        if (m > 0.f) {
          int ex;
          frexpf(m, &ex);
          s = max(-100, min(100, ex - 15));
        }
        xexp[t0 + t] = s;
      }
    }
  }

  const int e = blockIdx.x * kRouterWarps + warp;
  if (e < E) {
    float acc[TN];
#pragma unroll
    for (int t = 0; t < TN; ++t) acc[t] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(Wr + (size_t)e * d);
    for (int i4 = lane; i4 < d / 4; i4 += 32) {
      const float4 w = __ldg(w4 + i4);
#pragma unroll
      for (int t = 0; t < TN; ++t) {
        const uint2 xv = reinterpret_cast<const uint2*>(xs + (size_t)t * d)[i4];
        const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
        const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
        acc[t] = fmaf(w.x, x0, acc[t]);
        acc[t] = fmaf(w.y, x1, acc[t]);
        acc[t] = fmaf(w.z, x2, acc[t]);
        acc[t] = fmaf(w.w, x3, acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < TN; ++t) {
      float v = acc[t];
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[t] = v;
    }
    if (lane == 0) {
      const float b = bias ? bias[e] : 0.f;
#pragma unroll
      for (int t = 0; t < TN; ++t)
        if (t < nt) logits[(size_t)(t0 + t) * E + e] = acc[t] + b;
    }
  }
  if (FUSE) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned int n = atomicAdd(counter, 1u);
      last = n == gridDim.x * gridDim.y - 1;
    }
    __syncthreads();
    if (last) {
      __threadfence();
      float* Ls = reinterpret_cast<float*>(smem_raw + (size_t)TN * d * 2) + (size_t)warp * E;
      for (int t = warp; t < N; t += kRouterWarps) {
        stage_logits(logits, t, E, Ls);
        topk_row(Ls, E, k, norm_topk, idx + (size_t)t * k, gates + (size_t)t * k);
        __syncwarp();
      }
      if (threadIdx.x == 0) *counter = 0u;
    }
  }
}

// Decode-sized batches (N <= 64): one CTA per expert and token tile, its 8
// warps splitting K, so each lane issues all of its W_r loads at once (2
// float4 per lane for d = 2048) and the expert's dot products finish after
// about one memory round trip; x comes straight from L2.  The 8 partial sums
// of each logit are added in a fixed order.  The last CTA to finish runs the
// top-k of every token (one launch for the whole routing).
template <int TN>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_dec_kernel(const __nv_bfloat16* __restrict__ x, int N, int d, int E,
                  const float* __restrict__ Wr, const float* __restrict__ bias,
                  float* __restrict__ logits, int* __restrict__ xexp, int k, int norm_topk,
                  int* __restrict__ idx, float* __restrict__ gates, unsigned int* __restrict__ counter) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ float part[kRouterWarps][TN];
  __shared__ bool last;
  pdl_trigger();   // the routing tail may start: it waits for these results before reading them
  const int e = blockIdx.x, t0 = blockIdx.y * TN;
  const int nt = min(TN, N - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ks = d / kRouterWarps;          // this warp's K slice (a multiple of 16)
  const int k0 = warp * ks;
  // W_r: 4 floats per load, every load of the slice issued before any use
  const float4* w4 = reinterpret_cast<const float4*>(Wr + (size_t)e * d + k0);
  const int nv = ks / 4;                     // float4 per warp slice
  float acc[TN];
#pragma unroll
  for (int t = 0; t < TN; ++t) acc[t] = 0.f;
  for (int base = 0; base < nv; base += 4 * 32) {
    float4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * 32 + lane;
      w[u] = i < nv ? __ldg(w4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < TN; ++t) {
      if (t < nt) {
        const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * d + k0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = base + u * 32 + lane;
          if (i < nv) {
            const uint2 xv = xr[i];
            acc[t] = fmaf(w[u].x, __uint_as_float(xv.x << 16), acc[t]);
            acc[t] = fmaf(w[u].y, __uint_as_float(xv.x & 0xffff0000u), acc[t]);
            acc[t] = fmaf(w[u].z, __uint_as_float(xv.y << 16), acc[t]);
            acc[t] = fmaf(w[u].w, __uint_as_float(xv.y & 0xffff0000u), acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TN; ++t) {
    float v = acc[t];
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[warp][t] = v;
  }
  if (e == 0 && xexp != nullptr) {
    // per-token exponent s with amax(|x|) * 2^-s in [2^14, 2^15): warp t takes token t
    for (int t = warp; t < nt; t += kRouterWarps) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * d);
      float m = 0.f;
      for (int i = lane; i < d / 8; i += 32) {
        const uint4 v = xr[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xffff0000u))));
      }
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) {
        int s = 0;
        if (m > 0.f) {
          int ex;
          frexpf(m, &ex);
          s = max(-100, min(100, ex - 15));
        }
        xexp[t0 + t] = s;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float v = bias ? bias[e] : 0.f;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) sum += part[w][threadIdx.x];
    logits[(size_t)(t0 + threadIdx.x) * E + e] = sum + v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int n = atomicAdd(counter, 1u);
    last = n == gridDim.x * gridDim.y - 1;
  }
  __syncthreads();
  if (last) {
    __threadfence();
    float* Ls = reinterpret_cast<float*>(smem_raw) + (size_t)warp * E;
    for (int t = warp; t < N; t += kRouterWarps) {
      stage_logits(logits, t, E, Ls);
      topk_row(Ls, E, k, norm_topk, idx + (size_t)t * k, gates + (size_t)t * k);
      __syncwarp();
    }
    if (threadIdx.x == 0) *counter = 0u;
  }
}

__global__ void __launch_bounds__(256)
router_topk_kernel(const float* __restrict__ logits, int N, int E, int k, int norm_topk,
                   int* __restrict__ idx, float* __restrict__ gates) {
  extern __shared__ float Lsm[];
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= N) return;
  float* Ls = Lsm + (size_t)(threadIdx.x >> 5) * E;
  stage_logits(logits, t, E, Ls);
  topk_row(Ls, E, k, norm_topk, idx + (size_t)t * k, gates + (size_t)t * k);
}

}  // namespace

cudaError_t launch_router(const Geo& g, const __nv_bfloat16* x, int N, const float* Wr,
                          const float* bias, float* logits, int* idx, float* gates,
                          int* xexp, unsigned int* counter, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int TN = N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : 8;
  const bool fuse = N <= 64 && counter != nullptr;
  dim3 grid((g.E + kRouterWarps - 1) / kRouterWarps, (N + TN - 1) / TN);
  const size_t smem = (size_t)TN * g.d * sizeof(__nv_bfloat16) +
                      (fuse ? (size_t)kRouterWarps * g.E * sizeof(float) : 0);
  cudaError_t err = cudaSuccess;
#define MOE_ROUTER_CASE(V, F)                                                                \
  {                                                                                          \
    static bool attr = false;                                                                \
    if (!attr) {                                                                             \
      err = cudaFuncSetAttribute(router_logits_kernel<V, F>,                                 \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);   \
      if (err != cudaSuccess) return err;                                                    \
      attr = true;                                                                           \
    }                                                                                        \
    router_logits_kernel<V, F><<<grid, kRouterWarps * 32, smem, st>>>(                       \
        x, N, g.d, g.E, Wr, bias, logits, xexp, g.k, g.norm_topk, idx, gates, counter);     \
  }
  if (fuse) {
    // decode sizes: one CTA per expert and token tile (router_dec_kernel)
    const dim3 gd(g.E, (N + TN - 1) / TN);
    const size_t sm = (size_t)kRouterWarps * g.E * sizeof(float);
    switch (TN) {
      case 1: router_dec_kernel<1><<<gd, kRouterWarps * 32, sm, st>>>(x, N, g.d, g.E, Wr, bias, logits, xexp, g.k, g.norm_topk, idx, gates, counter); break;
      case 2: router_dec_kernel<2><<<gd, kRouterWarps * 32, sm, st>>>(x, N, g.d, g.E, Wr, bias, logits, xexp, g.k, g.norm_topk, idx, gates, counter); break;
      case 4: router_dec_kernel<4><<<gd, kRouterWarps * 32, sm, st>>>(x, N, g.d, g.E, Wr, bias, logits, xexp, g.k, g.norm_topk, idx, gates, counter); break;
      default: router_dec_kernel<8><<<gd, kRouterWarps * 32, sm, st>>>(x, N, g.d, g.E, Wr, bias, logits, xexp, g.k, g.norm_topk, idx, gates, counter); break;
    }
    return cudaGetLastError();
  }
  switch (TN) {
    case 1: MOE_ROUTER_CASE(1, false) break;
    case 2: MOE_ROUTER_CASE(2, false) break;
    case 4: MOE_ROUTER_CASE(4, false) break;
    default: MOE_ROUTER_CASE(8, false) break;
  }
#undef MOE_ROUTER_CASE
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  router_topk_kernel<<<(N + 7) / 8, 256, (size_t)8 * g.E * sizeof(float), st>>>(logits, N, g.E, g.k,
                                                                              g.norm_topk, idx, gates);
  return cudaGetLastError();
}

}  // namespace moe
