// Device pieces of the router shared by the router kernels and the fused
// decode step: the decode-size dot products (one expert's K split over 8
// warps), the per-token f16 exponent of x, and the warp top-k with gates.
//
// The pages do not define the router (they only say routing picks a few
// experts per token and varies per layer and token: "FreeToken：把 284B MoE
// 塞进游戏 PC", zhichai.net, §二 "Decode" paragraph; ananclaw.com explainer,
// §核心方法 1); this is the standard softmax top-k router.  Both the chained
// decode path and the fused step call these functions, so their logits, ids
// and gates agree bit for bit.
#pragma once
#include "common.cuh"

namespace moe {
namespace rt {

constexpr int kRouterWarps = 8;

// Order-preserving 32-bit key of a logit: a > b (as floats) <=> key(a) >
// key(b), equal floats give equal keys (-0 is +0), and a NaN ranks as -inf.
MOE_DEV uint32_t logit_key(float v) {
  if (!(v == v)) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp: the k largest of the logits row L (shared memory, E <= 1024
// entries; ties to the lower expert id), gates, written in ascending id order.
// Each of the k rounds takes the largest key a lane still holds, then two
// warp reductions (redux.sync): the largest key, and the lowest id holding it.
MOE_DEV void topk_gates(const float* L, int E, int k, int norm_topk, int my_e, int* idx, float* gates);

MOE_DEV void topk_row(const float* L, int E, int k, int norm_topk, int* idx, float* gates) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit i: entry lane + 32 i already selected
  int my_e = -1;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int be = 0x7fffffff;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      const uint32_t key = logit_key(L[e]);
      if (key > bk) { bk = key; be = e; }   // ascending e: the first of equal keys is kept
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int w = (int)__reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)be : 0xffffffffu);
    if ((w & 31) == lane) taken |= 1u << (w >> 5);
    if (lane == j) my_e = w;
  }
  topk_gates(L, E, k, norm_topk, my_e, idx, gates);
}

// The same selection for E <= 32 P: each lane sorts its P entries (lane + 32 i,
// ascending id) once by key, descending and stable, so its head is the
// largest key it holds with the lowest id among equal ones -- what the scan of
// topk_row finds in every round -- and the winner of a round drops its head.
template <int P>
MOE_DEV void topk_row_sorted(const float* L, int E, int k, int norm_topk, int* idx, float* gates) {
  const int lane = threadIdx.x & 31;
  uint32_t ks[P];
  int es[P];
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const int e = lane + 32 * i;
    ks[i] = e < E ? logit_key(L[e]) : 0u;   // no entry: below every key (as the scan's start)
    es[i] = e < E ? e : 0x7fffffff;
  }
#pragma unroll
  for (int i = 1; i < P; ++i)
#pragma unroll
    for (int j = i; j > 0; --j)
      if (ks[j] > ks[j - 1]) {   // strict: equal keys keep ascending ids
        const uint32_t tk = ks[j];
        ks[j] = ks[j - 1];
        ks[j - 1] = tk;
        const int te = es[j];
        es[j] = es[j - 1];
        es[j - 1] = te;
      }
  int my_e = -1;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, ks[0]);
    const int w = (int)__reduce_min_sync(0xffffffffu, ks[0] == m ? (uint32_t)es[0] : 0xffffffffu);
    if ((w & 31) == lane) {
#pragma unroll
      for (int i = 0; i + 1 < P; ++i) {
        ks[i] = ks[i + 1];
        es[i] = es[i + 1];
      }
      ks[P - 1] = 0u;
      es[P - 1] = 0x7fffffff;
    }
    if (lane == j) my_e = w;
  }
  topk_gates(L, E, k, norm_topk, my_e, idx, gates);
}

// topk_row with the presorted selection for E <= 256: the same ids and gates.
// The prefill-sized top-k uses it (one warp per token, thousands of tokens);
// inside the fused decode step the scan measured faster.
MOE_DEV void topk_row_many(const float* L, int E, int k, int norm_topk, int* idx, float* gates) {
  if (E <= 32) return topk_row_sorted<1>(L, E, k, norm_topk, idx, gates);
  if (E <= 64) return topk_row_sorted<2>(L, E, k, norm_topk, idx, gates);
  if (E <= 128) return topk_row_sorted<4>(L, E, k, norm_topk, idx, gates);
  if (E <= 256) return topk_row_sorted<8>(L, E, k, norm_topk, idx, gates);
  topk_row(L, E, k, norm_topk, idx, gates);
}

// The selected experts' gates (one warp): lane j < k holds my_e = the j-th
// largest logit's expert (selection order); writes idx and gates in ascending
// expert order.  Gates (fp32) = softmax over the selected logits, or the full
// softmax probabilities.  Every top-k of the library ends here, so the
// chained and the fused decode paths compute the same gates bit for bit.
MOE_DEV void topk_gates(const float* L, int E, int k, int norm_topk, int my_e, int* idx, float* gates) {
  const int lane = threadIdx.x & 31;
  const float top = L[__shfl_sync(0xffffffffu, my_e, 0)];
  const float my_v = lane < k ? L[my_e] : 0.f;
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

// Power-of-two exponent s of one token row (d bf16 values) with
// max|x| 2^-s in [2^14, 2^15) (0 for a zero row), computed by one warp; every
// lane returns it.  The decode expert GEMV converts x 2^-s to f16, which then
// neither overflows nor loses precision to subnormals.
MOE_DEV int token_exp(const __nv_bfloat16* __restrict__ xr, int d) {
  const int lane = threadIdx.x & 31;
  const uint4* x4 = reinterpret_cast<const uint4*>(xr);
  const int n = d / 8;
  float m = 0.f;
  // eight 16-byte loads per lane in flight before any use (one round trip
  // for d <= 2048); zero padding leaves the maximum unchanged
  for (int i0 = lane; i0 < n; i0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + 32 * u;
      v[u] = i < n ? x4[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xffff0000u))));
    }
  }
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int s = 0;
  if (m > 0.f) {
    int ex;
    frexpf(m, &ex);
    s = max(-100, min(100, ex - 15));
  }
  return s;
}

// Warp `warp` (of kRouterWarps) of one expert's dot products with tokens
// t0 .. t0 + nt - 1 (nt <= TN): the warp's K slice d / 8 (a multiple of 16),
// every W_r load of the slice issued before any use (2 float4 per lane for
// d = 2048), x straight from L2.  sum[t] (every lane) = the warp's partial
// dot product of token t0 + t; the caller adds the 8 partials in warp order.
template <int TN>
MOE_DEV void router_dot(const __nv_bfloat16* __restrict__ x, int t0, int nt, int d, const float* __restrict__ wrow,
                        int warp, float (&sum)[TN]) {
  const int lane = threadIdx.x & 31;
  const int ks = d / kRouterWarps;
  const int k0 = warp * ks;
  const float4* w4 = reinterpret_cast<const float4*>(wrow + k0);
  const int nv = ks / 4;
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
    sum[t] = v;
  }
}

// The logit of expert e from its 8 warp partials part[w] (warp order) and
// the bias: the same sum on every path.
MOE_DEV float logit_from_parts(const float* part, int stride, float bias) {
  float sum = 0.f;
#pragma unroll
  for (int w = 0; w < kRouterWarps; ++w) sum += part[w * stride];
  return sum + bias;
}

}  // namespace rt
}  // namespace moe
