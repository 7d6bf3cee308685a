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
// each O row: V = 4 (fp32) or 8 (f16) columns.
struct OF32 {
  static constexpr int V = 4;
  const float* O;
  MOE_DEV void load(size_t row, int d, int cv, float (&o)[4]) const {
    const float4 v = reinterpret_cast<const float4*>(O + row * d)[cv];
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
struct OF16 {
  static constexpr int V = 8;
  const __half* O;
  const int8_t* e;
  MOE_DEV void load(size_t row, int d, int cv, float (&o)[8]) const {
    const uint4 v = reinterpret_cast<const uint4*>(O + row * d)[cv];
    const float s = __int_as_float((127 + e[row * (d / 128) + cv / 16]) << 23);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      o[2 * i] = f.x * s;
      o[2 * i + 1] = f.y * s;
    }
  }
};

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
  for (int j = 0; j < k; ++j) {
    const float gj = gates[(size_t)t * k + j];
    float o[V];
    O.load((size_t)row_of[(size_t)t * k + j], d, cv, o);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(gj, o[i], acc[i]);
  }
  if (shared) {
    float o[V];
    O.load((size_t)N * k + t, d, cv, o);
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
    const int total = N * (g.d / OF16::V);
    return launch_pdl(combine_kernel<OF16>, dim3((total + 255) / 256), dim3(256), 0, st,
                      OF16{reinterpret_cast<const __half*>(O), prefill_o_exp(g, O, N)}, gates, row_of, N, g.k, g.d,
                      g.has_shared, y);
  }
  const int total = N * (g.d / OF32::V);
  return launch_pdl(combine_kernel<OF32>, dim3((total + 255) / 256), dim3(256), 0, st, OF32{O}, gates, row_of, N,
                    g.k, g.d, g.has_shared, y);
}

}  // namespace moe
