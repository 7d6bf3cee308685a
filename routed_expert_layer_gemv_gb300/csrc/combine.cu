// Combine: y[t] = sum_{j < k} gate[t, j] * O[row_of[t, j]] (+ O[N*k + t] for
// the shared expert, weight 1), accumulated in fp32 in ascending j (= ascending
// expert id) and rounded once to bf16.  A fixed summation order with no
// atomics makes the output reproducible bit for bit.  (The pages do not define
// the combine; a shared, always-on expert is one of the architecture axes of
// the ananclaw.com explainer, §核心方法 4.)
#include "common.cuh"

namespace moe {

namespace {

// O rows are fp32 (decode) or f16 with a power-of-two exponent per row and
// 128-column block (prefill: half the bytes of the largest intermediate);
// either way the sum is formed in fp32.  A thread takes one 16-byte piece of
// each O row: V = 4 (fp32) or 8 (f16) columns.  fetch() only issues the loads
// (so a thread has all of its rows in flight at once); unpack() converts.
struct OF32 {
  static constexpr int V = 4;
  struct Raw { float4 v; };
  const float* O;
  MOE_DEV Raw fetch(size_t row, int d, int cv) const { return {reinterpret_cast<const float4*>(O + row * d)[cv]}; }
  MOE_DEV static void unpack(const Raw& r, float (&o)[4]) {
    o[0] = r.v.x; o[1] = r.v.y; o[2] = r.v.z; o[3] = r.v.w;
  }
};
struct OF16 {
  static constexpr int V = 8;
  struct Raw { uint4 v; int e; };
  const __half* O;
  const int8_t* e;
  MOE_DEV Raw fetch(size_t row, int d, int cv) const {
    return {reinterpret_cast<const uint4*>(O + row * d)[cv], e[row * (d / 128) + cv / 16]};
  }
  MOE_DEV static void unpack(const Raw& r, float (&o)[8]) {
    const float s = __int_as_float((127 + r.e) << 23);
    const uint32_t w[4] = {r.v.x, r.v.y, r.v.z, r.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x * s;
      o[2 * i + 1] = f.y * s;
    }
  }
};

// Rows of one token fetched together, kBatch per round trip.  Four rows
// (64 B in flight per thread at 56 registers) measured best on the 35B-A3B
// prefill chunk: 76 -> 57 us against one row at a time; eight rows need 85
// registers and ran slower (85 us) for the lost occupancy.
constexpr int kBatch = 4;

template <typename OT>
__global__ void combine_kernel(const OT O, const float* __restrict__ gates,
                               const int* __restrict__ row_of, int N, int k, int d, int shared,
                               __nv_bfloat16* __restrict__ y) {
  constexpr int V = OT::V;
  pdl_wait();
  const int q = d / V;
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= N * q) return;
  const int t = v / q, cv = v % q;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    int r[kBatch];
    float gj[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const bool in = j0 + u < k;
      r[u] = in ? __ldg(row_of + (size_t)t * k + j0 + u) : 0;
      gj[u] = in ? __ldg(gates + (size_t)t * k + j0 + u) : 0.f;
    }
    typename OT::Raw raw[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (j0 + u < k) raw[u] = O.fetch((size_t)r[u], d, cv);
    // ascending j, one fma per term: the summation order of the definition
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + u < k) {
        float o[V];
        OT::unpack(raw[u], o);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(gj[u], o[i], acc[i]);
      }
    }
  }
  if (shared) {
    float o[V];
    OT::unpack(O.fetch((size_t)N * k + t, d, cv), o);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += o[i];
  }
  uint32_t out[V / 2];
#pragma unroll
  for (int i = 0; i < V / 2; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    out[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  if constexpr (V == 8)
    reinterpret_cast<uint4*>(y + (size_t)t * d)[cv] = make_uint4(out[0], out[1], out[2], out[3]);
  else
    reinterpret_cast<uint2*>(y + (size_t)t * d)[cv] = make_uint2(out[0], out[1]);
}

}  // namespace

cudaError_t launch_combine(const Geo& g, const float* O, bool o_f16, const float* gates, const int* row_of,
                           int N, __nv_bfloat16* y, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  if (o_f16) {
    // 128-thread blocks measured faster than 256 (57 vs 60 us, 35B-A3B chunk)
    const int total = N * (g.d / OF16::V);
    return launch_pdl(combine_kernel<OF16>, dim3((total + 127) / 128), dim3(128), 0, st,
                      OF16{reinterpret_cast<const __half*>(O), prefill_o_exp(g, O, N)}, gates, row_of, N, g.k, g.d,
                      g.has_shared, y);
  }
  const int total = N * (g.d / OF32::V);
  return launch_pdl(combine_kernel<OF32>, dim3((total + 255) / 256), dim3(256), 0, st, OF32{O}, gates, row_of, N,
                    g.k, g.d, g.has_shared, y);
}

}  // namespace moe
