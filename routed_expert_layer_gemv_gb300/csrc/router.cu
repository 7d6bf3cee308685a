// Router: logits = x W_r^T (+ b) in fp32, then per token the k largest
// logits (ties -> lower expert id), gates = softmax restricted to them (or
// the full-softmax probabilities), emitted in ascending expert order.
//
// The FreeToken pages do not define the router; they only say routing picks
// a few experts per token and varies per layer and token ("FreeToken：把 284B
// MoE 塞进游戏 PC", zhichai.net, §二 "Decode" paragraph; ananclaw.com
// explainer, §核心方法 1).  This is the standard softmax top-k router.
//
// Decode-sized batches (router_dec_kernel): one CTA per expert and token
// tile, K split over its warps; its last CTA runs the top-k, so routing is
// one launch.  Larger batches (router_tc_kernel): logits on tensor cores from
// a three-part bf16 split of W_r, then router_topk_kernel.  The CTAs that
// see a token's whole row also write its power-of-two exponent, used by the
// expert GEMV to convert x to f16 without overflow.
// topk: one warp per token on its logits row staged in shared memory; k
// rounds of a warp-wide argmax.
#include "common.cuh"
#include "router_dev.cuh"

namespace moe {

namespace {

using rt::kRouterWarps;
using rt::stage_logits;
using rt::topk_row;

// Decode-sized batches (N <= 64): one CTA per expert and token tile, its 8
// warps splitting K, so each lane issues all of its W_r loads at once (2
// float4 per lane for d = 2048) and the expert's dot products finish after
// about one memory round trip; x comes straight from L2.  The 8 partial sums
// of each logit are added in a fixed order.  The last of a token tile's E
// CTAs to finish runs the top-k of the tile's tokens, one warp per token
// (one launch for the whole routing; counter[y] counts tile y's CTAs).
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
  {
    float sum[TN];
    rt::router_dot<TN>(x, t0, nt, d, Wr + (size_t)e * d, warp, sum);
#pragma unroll
    for (int t = 0; t < TN; ++t)
      if (lane == 0) part[warp][t] = sum[t];
  }
  if (e == 0 && xexp != nullptr) {
    // per-token exponent of x (the decode GEMV's f16 conversion): warp t takes token t
    for (int t = warp; t < nt; t += kRouterWarps) {
      const int s = rt::token_exp(x + (size_t)(t0 + t) * d, d);
      if (lane == 0) xexp[t0 + t] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x < nt)
    logits[(size_t)(t0 + threadIdx.x) * E + e] = rt::logit_from_parts(&part[0][threadIdx.x], TN, bias ? bias[e] : 0.f);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int n = atomicAdd(counter + blockIdx.y, 1u);
    last = n == gridDim.x - 1;
  }
  __syncthreads();
  if (last) {
    __threadfence();
    float* Ls = reinterpret_cast<float*>(smem_raw) + (size_t)warp * E;
    for (int t = t0 + warp; t < t0 + nt; t += kRouterWarps) {
      stage_logits(logits, t, E, Ls);
      topk_row(Ls, E, k, norm_topk, idx + (size_t)t * k, gates + (size_t)t * k);
      __syncwarp();
    }
    if (threadIdx.x == 0) counter[blockIdx.y] = 0u;
  }
}

// Large batches (prefill): logits on tensor cores.  W_r is split once into
// three bf16 parts W = W0 + W1 + W2 + r with W0 = bf16(W), W1 = bf16(W - W0),
// W2 = bf16(W - W0 - W1) (each difference is exact in fp32), so |r| <= 2^-24
// |W|: the split is as close to W as W's own fp32 rounding.  x is exact in
// bf16, so x W^T = sum_p x W_p^T with fp32 accumulation (mma.sync m16n8k16
// bf16) gives fp32-class logits at tensor-core rate.  CTA tile 64 tokens x 64
// experts, K in chunks of 64 through a cp.async double buffer; 8 warps as 2
// (tokens) x 4 (experts), each 32 x 16.  CTAs of expert tile 0 also write the
// per-token f16 exponent of x.
constexpr int kTcM = 64, kTcN = 64, kTcK = 64, kTcParts = 3;
constexpr int kTcRow = kTcK + 8;          // padded smem row (bf16): 144 bytes, conflict-free ldmatrix
constexpr int kTcRows = kTcM + kTcParts * kTcN;
constexpr int kTcStage = kTcRows * kTcRow;   // bf16 elements per stage

__global__ void router_split_kernel(const float* __restrict__ W, size_t n, __nv_bfloat16* __restrict__ parts) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float r = W[i];
#pragma unroll
  for (int p = 0; p < kTcParts; ++p) {
    const __nv_bfloat16 h = __float2bfloat16_rn(r);
    parts[(size_t)p * n + i] = h;
    r -= __bfloat162float(h);
  }
}

MOE_DEV void cp16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

MOE_DEV void ldsm_x4(const void* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

MOE_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
               "{%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256)
router_tc_kernel(const __nv_bfloat16* __restrict__ x, int N, int d, int E, const __nv_bfloat16* __restrict__ Wp,
                 const float* __restrict__ bias, float* __restrict__ logits, int* __restrict__ xexp) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* sm = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  const int t0 = blockIdx.x * kTcM, e0 = blockIdx.y * kTcN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp >> 2, wn = warp & 3;      // 2 x 4 warps: 32 tokens x 16 experts each
  const size_t part = (size_t)E * d;
  const int nk = d / kTcK;
  auto load = [&](int kc, int buf) {
    __nv_bfloat16* st = sm + (size_t)buf * kTcStage;
    // rows: 64 tokens, then 64 experts of each W part; 8 chunks of 16 bytes per row
    for (int v = threadIdx.x; v < kTcRows * 8; v += 256) {
      const int r = v >> 3, c = v & 7;
      const __nv_bfloat16* src;
      bool ok;
      if (r < kTcM) {
        ok = t0 + r < N;
        src = x + (size_t)min(t0 + r, N - 1) * d + kc * kTcK + 8 * c;
      } else {
        const int rr = (r - kTcM) % kTcN, p = (r - kTcM) / kTcN;
        ok = e0 + rr < E;
        src = Wp + p * part + (size_t)min(e0 + rr, E - 1) * d + kc * kTcK + 8 * c;
      }
      cp16_zfill(st + (size_t)r * kTcRow + 8 * c, src, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[2][2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;
  load(0, 0);
  for (int kc = 0; kc < nk; ++kc) {
    if (kc + 1 < nk) {
      load(kc + 1, (kc + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const __nv_bfloat16* xa = sm + (size_t)(kc & 1) * kTcStage;
    const __nv_bfloat16* wb = xa + (size_t)kTcM * kTcRow;
#pragma unroll
    for (int k16 = 0; k16 < kTcK / 16; ++k16) {
      uint32_t a[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = wm * 32 + 16 * i + (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4(xa + (size_t)row * kTcRow + 16 * k16 + 8 * (lane >> 4), a[i]);
      }
      // The tensor core's own accumulation is not round-to-nearest, so a
      // long chain of MMAs on one accumulator drifts: each 16-wide step sums
      // its three parts (smallest first) from zero, and the step's result is
      // added to the running sums with ordinary fp32 adds.
      float tmp[2][2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) tmp[i][j][q] = 0.f;
#pragma unroll
      for (int p = kTcParts - 1; p >= 0; --p) {
        uint32_t b[4];   // b0, b1 of experts n0..n0+7, then of n0+8..n0+15
        const int n = p * kTcN + wn * 16 + (lane & 7) + 8 * (lane >> 4);
        ldsm_x4(wb + (size_t)n * kTcRow + 16 * k16 + 8 * ((lane >> 3) & 1), b);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          mma_bf16(tmp[i][0], a[i], b[0], b[1]);
          mma_bf16(tmp[i][1], a[i], b[2], b[3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[i][j][q] += tmp[i][j][q];
    }
    __syncthreads();
  }
  // fragment (i, j): rows wm*32 + 16i + g (+8), columns wn*16 + 8j + 2q (+1)
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + wm * 32 + 16 * i + g + 8 * hh;
        const int e = e0 + wn * 16 + 8 * j + 2 * q;
        if (t < N) {
          if (e < E) logits[(size_t)t * E + e] = acc[i][j][2 * hh] + (bias ? bias[e] : 0.f);
          if (e + 1 < E) logits[(size_t)t * E + e + 1] = acc[i][j][2 * hh + 1] + (bias ? bias[e + 1] : 0.f);
        }
      }
  if (blockIdx.y == 0 && xexp != nullptr) {
    // per-token exponent of x (the decode GEMV's f16 conversion): warp w takes tokens w, w + 8, ...
    for (int tl = warp; tl < kTcM; tl += 8) {
      const int t = t0 + tl;
      if (t >= N) break;
      const int s = rt::token_exp(x + (size_t)t * d, d);
      if (lane == 0) xexp[t] = s;
    }
  }
}

__global__ void __launch_bounds__(256)
router_topk_kernel(float* __restrict__ logits, const float* __restrict__ part2, const float* __restrict__ bias,
                   int N, int E, int k, int norm_topk, int* __restrict__ idx, float* __restrict__ gates) {
  extern __shared__ float Lsm[];
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= N) return;
  float* Ls = Lsm + (size_t)(threadIdx.x >> 5) * E;
  if (part2 != nullptr) {
    // logits from two K halves: (first + second) + bias, written back
    for (int e = threadIdx.x & 31; e < E; e += 32) {
      const size_t i = (size_t)t * E + e;
      const float v = (__ldcg(logits + i) + __ldcg(part2 + i)) + (bias ? bias[e] : 0.f);
      logits[i] = v;
      Ls[e] = v;
    }
    __syncwarp();
  } else {
    stage_logits(logits, t, E, Ls);
  }
  rt::topk_row_many(Ls, E, k, norm_topk, idx + (size_t)t * k, gates + (size_t)t * k);
}

}  // namespace

cudaError_t launch_router_split(const Geo& g, const float* Wr, __nv_bfloat16* Wp, cudaStream_t st) {
  const size_t n = (size_t)g.E * g.d;
  router_split_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(Wr, n, Wp);
  return cudaGetLastError();
}

cudaError_t launch_router(const Geo& g, const __nv_bfloat16* x, int N, const float* Wr,
                          const __nv_bfloat16* Whl, const float* bias, float* logits, int* idx,
                          float* gates, int* xexp, unsigned int* counter, int* errw, float* part2,
                          cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  if (Whl == nullptr || counter == nullptr) return cudaErrorInvalidValue;
  if (N > 64) {
    // large batches: tensor-core logits (tcgen05 where the shape allows,
    // else mma.sync), then the top-k kernel
    int split = 1;
    cudaError_t err = errw ? launch_router_tc5(g, x, N, Whl, bias, logits, part2, &split, xexp, errw, st)
                           : cudaErrorNotSupported;
    if (err == cudaErrorNotSupported) {
      const size_t smem = (size_t)2 * kTcStage * sizeof(__nv_bfloat16);
      cudaError_t e = ensure_smem_limit((const void*)router_tc_kernel, (int)smem);
      if (e != cudaSuccess) return e;
      const dim3 grid((N + kTcM - 1) / kTcM, (g.E + kTcN - 1) / kTcN);
      router_tc_kernel<<<grid, 256, smem, st>>>(x, N, g.d, g.E, Whl, bias, logits, xexp);
      err = cudaGetLastError();
    }
    if (err != cudaSuccess) return err;
    router_topk_kernel<<<(N + 7) / 8, 256, (size_t)8 * g.E * sizeof(float), st>>>(
        logits, split > 1 ? part2 : nullptr, bias, N, g.E, g.k, g.norm_topk, idx, gates);
    return cudaGetLastError();
  }
  // decode sizes: one CTA per expert and token tile, top-k fused (router_dec_kernel)
  // token tiles of at most 4 up to 16 tokens: more, shorter CTAs (batch 16: 102.5 -> 101.5 us)
  const int TN = N <= 1 ? 1 : N <= 2 ? 2 : N <= 16 ? 4 : 8;
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

}  // namespace moe
