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
// topk kernel: one warp per token; k rounds of a warp-wide argmax.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;

template <int TN>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(const __nv_bfloat16* __restrict__ x, int N, int d, int E,
                     const float* __restrict__ Wr, const float* __restrict__ bias,
                     float* __restrict__ logits, int* __restrict__ xexp) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem_raw);  // [TN][d]
  const int t0 = blockIdx.y * TN;
  const int nt = min(TN, N - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // stage the token tile (16-byte vectors; d is a multiple of 128)
  const int vec_per_row = d / 8;
  for (int v = threadIdx.x; v < TN * vec_per_row; v += blockDim.x) {
    int t = v / vec_per_row, c = v % vec_per_row;
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
  if (e >= E) return;
  float acc[TN];
#pragma unroll
  for (int t = 0; t < TN; ++t) acc[t] = 0.f;
  const float4* w4 = reinterpret_cast<const float4*>(Wr + (size_t)e * d);
  for (int i4 = lane; i4 < d / 4; i4 += 32) {
    float4 w = __ldg(w4 + i4);
#pragma unroll
    for (int t = 0; t < TN; ++t) {
      uint2 xv = reinterpret_cast<const uint2*>(xs + (size_t)t * d)[i4];
      float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xffff0000u);
      float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xffff0000u);
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
    float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int t = 0; t < TN; ++t)
      if (t < nt) logits[(size_t)(t0 + t) * E + e] = acc[t] + b;
  }
}

MOE_DEV bool better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

__global__ void __launch_bounds__(256)
router_topk_kernel(const float* __restrict__ logits, int N, int E, int k, int norm_topk,
                   int* __restrict__ idx, float* __restrict__ gates) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= N) return;
  const float* L = logits + (size_t)t * E;
  uint32_t taken = 0;  // bit i: entry lane + 32 i already selected (E <= 1024)
  int my_e = -1;
  float my_v = 0.f, top = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      float v = L[e];
      if (better(v, e, bv, be)) { bv = v; be = e; }
    }
    for (int o = 16; o; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (j == 0) top = bv;
    if (lane == j) { my_e = be; my_v = bv; }
  }
  // gates (fp32): softmax over the selected logits, or the full softmax
  float num = lane < k ? expf(my_v - top) : 0.f;
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
    int oe = __shfl_sync(0xffffffffu, my_e, i);
    rank += (lane < k && oe < my_e) ? 1 : 0;
  }
  if (lane < k) {
    idx[(size_t)t * k + rank] = my_e;
    gates[(size_t)t * k + rank] = num / den;
  }
}

}  // namespace

cudaError_t launch_router(const Geo& g, const __nv_bfloat16* x, int N, const float* Wr,
                          const float* bias, float* logits, int* idx, float* gates,
                          int* xexp, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int TN = N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : 8;
  dim3 grid((g.E + kRouterWarps - 1) / kRouterWarps, (N + TN - 1) / TN);
  size_t smem = (size_t)TN * g.d * sizeof(__nv_bfloat16);
  switch (TN) {
#define MOE_ROUTER_CASE(V)                                                                   \
  case V:                                                                                    \
    if (smem > 48 * 1024)                                                                    \
      cudaFuncSetAttribute(router_logits_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                       \
    router_logits_kernel<V><<<grid, kRouterWarps * 32, smem, st>>>(x, N, g.d, g.E, Wr, bias,   \
                                                                  logits, xexp);             \
    break;
    MOE_ROUTER_CASE(1)
    MOE_ROUTER_CASE(2)
    MOE_ROUTER_CASE(4)
    MOE_ROUTER_CASE(8)
#undef MOE_ROUTER_CASE
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  router_topk_kernel<<<(N + 7) / 8, 256, 0, st>>>(logits, N, g.E, g.k, g.norm_topk, idx, gates);
  return cudaGetLastError();
}

}  // namespace moe
