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
// either way the sum is formed in fp32.
struct OF32 {
  const float* O;
  MOE_DEV float4 load(size_t row, int d, int c4) const { return reinterpret_cast<const float4*>(O + row * d)[c4]; }
};
struct OF16 {
  const __half* O;
  const int8_t* e;
  MOE_DEV float4 load(size_t row, int d, int c4) const {
    const uint2 v = reinterpret_cast<const uint2*>(O + row * d)[c4];
    const float s = __int_as_float((127 + e[row * (d / 128) + c4 / 32]) << 23);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    return make_float4(a.x * s, a.y * s, b.x * s, b.y * s);
  }
};

template <typename OT>
__global__ void combine_kernel(const OT O, const float* __restrict__ gates,
                               const int* __restrict__ row_of, int N, int k, int d, int shared,
                               __nv_bfloat16* __restrict__ y) {
  pdl_wait();
  const int q = d / 4;
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= N * q) return;
  const int t = v / q, c4 = v % q;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const float gj = gates[(size_t)t * k + j];
    const float4 o = O.load((size_t)row_of[(size_t)t * k + j], d, c4);
    acc.x = fmaf(gj, o.x, acc.x);
    acc.y = fmaf(gj, o.y, acc.y);
    acc.z = fmaf(gj, o.z, acc.z);
    acc.w = fmaf(gj, o.w, acc.w);
  }
  if (shared) {
    const float4 o = O.load((size_t)N * k + t, d, c4);
    acc.x += o.x;
    acc.y += o.y;
    acc.z += o.z;
    acc.w += o.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 out;
  out.x = *reinterpret_cast<uint32_t*>(&lo);
  out.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(y + (size_t)t * d)[c4] = out;
}

}  // namespace

cudaError_t launch_combine(const Geo& g, const float* O, bool o_f16, const float* gates, const int* row_of,
                           int N, __nv_bfloat16* y, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int total = N * (g.d / 4);
  if (o_f16)
    return launch_pdl(combine_kernel<OF16>, dim3((total + 255) / 256), dim3(256), 0, st,
                      OF16{reinterpret_cast<const __half*>(O), prefill_o_exp(g, O, N)}, gates, row_of, N, g.k, g.d,
                      g.has_shared, y);
  return launch_pdl(combine_kernel<OF32>, dim3((total + 255) / 256), dim3(256), 0, st, OF32{O}, gates, row_of, N,
                    g.k, g.d, g.has_shared, y);
}

}  // namespace moe
