// Test hooks: dequantise one slot's matrix, and run the activation quantiser
// on given rows.  They exercise the same device decoding / quantising code
// the forward path uses, so tests can compare them bit for bit.
#include "actquant.cuh"
#include "common.cuh"

namespace moe {

namespace {

__global__ void dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                               float tscale, int rows, int K, int fmt, float* __restrict__ out) {
  const int blk = fmt == MOE_MXFP4 ? 32 : 16;
  const size_t nbytes = (size_t)rows * (K / 2);
  const size_t p = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= nbytes) return;
  const int r = (int)(p / (K / 2));
  const int i = (int)(p % (K / 2)) * 2;     // even K index
  const uint32_t h2 = e2m1x2_to_f16x2(codes[p]);
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  const uint32_t sb = scales[(size_t)r * (K / blk) + i / blk];
  const float s = fmt == MOE_MXFP4 ? e8m0_to_f32(sb) : e4m3_to_f32(sb) * tscale;
  out[(size_t)r * K + i] = __low2float(hv) * s;
  out[(size_t)r * K + i + 1] = __high2float(hv) * s;
}

// MXFP8 / BF16 matrices: one thread per element (E4M3 x E8M0, or the bf16 value).
__global__ void dequant8_16_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int rows,
                                   int K, int fmt, float* __restrict__ out) {
  const size_t p = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= (size_t)rows * K) return;
  const int r = (int)(p / K), i = (int)(p % K);
  if (fmt == MOE_BF16) {
    const uint32_t lo = codes[2 * p], hi = codes[2 * p + 1];
    out[p] = __uint_as_float((lo | (hi << 8)) << 16);
  } else {
    out[p] = e4m3_to_f32(codes[p]) * e8m0_to_f32(scales[(size_t)r * (K / 32) + i / 32]);
  }
}

// Rows of 32-element blocks through the MXFP8 quantiser, or rounded to bf16.
__global__ void actquant8_16_kernel(const float* __restrict__ v, int rows, int K, int fmt,
                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int nb = K / 32;
  const size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= (size_t)rows * nb) return;
  const int r = (int)(b / nb), c = (int)(b % nb);
  const float* src = v + (size_t)r * K + (size_t)c * 32;
  if (fmt == MOE_BF16) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(codes) + (size_t)r * K + (size_t)c * 32;
    for (int i = 0; i < 32; ++i) dst[i] = __float2bfloat16_rn(src[i]);
    return;
  }
  float vals[32];
  for (int i = 0; i < 32; ++i) vals[i] = src[i];
  uint32_t words[8];
  scales[b] = (uint8_t)quant_mx8_32(vals, words);
  uint32_t* dst = reinterpret_cast<uint32_t*>(codes + (size_t)r * K + (size_t)c * 32);
  for (int w = 0; w < 8; ++w) dst[w] = words[w];
}

__global__ void actquant_kernel(const float* __restrict__ v, int rows, int K, int fmt, float g,
                                uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int blk = fmt == MOE_MXFP4 ? 32 : 16;
  const int nb = K / blk;
  const size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= (size_t)rows * nb) return;
  const int r = (int)(b / nb), c = (int)(b % nb);
  const float* src = v + (size_t)r * K + (size_t)c * blk;
  float vals[32];
  for (int i = 0; i < blk; ++i) vals[i] = src[i];
  uint32_t words[4];
  uint8_t* dst = codes + (size_t)r * (K / 2) + (size_t)c * (blk / 2);
  if (fmt == MOE_MXFP4) {
    scales[b] = (uint8_t)quant_mx32(vals, words);
    for (int w = 0; w < 4; ++w) reinterpret_cast<uint32_t*>(dst)[w] = words[w];
  } else {
    scales[b] = (uint8_t)quant_nv16(vals, g, words);
    for (int w = 0; w < 2; ++w) reinterpret_cast<uint32_t*>(dst)[w] = words[w];
  }
}

}  // namespace

cudaError_t launch_dequant(const Geo& g, const uint8_t* expert, int m, float* out, cudaStream_t st) {
  const int rows = m == 2 ? g.d : g.f;
  const int K = m == 2 ? g.f : g.d;
  const float* ts = reinterpret_cast<const float*>(expert + g.off_tscale);
  // the tensor scale is read on the host side of the copy below
  float tscale = 1.0f;
  cudaError_t err = cudaMemcpyAsync(&tscale, ts + m, sizeof(float), cudaMemcpyDeviceToHost, st);
  if (err != cudaSuccess) return err;
  err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return err;
  if (g.fmt == MOE_MXFP8 || g.fmt == MOE_BF16) {
    const size_t n = (size_t)rows * K;
    dequant8_16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(expert + g.off_codes[m],
                                                                    expert + g.off_scales[m], rows, K, g.fmt, out);
    return cudaGetLastError();
  }
  const size_t nbytes = (size_t)rows * (K / 2);
  dequant_kernel<<<(unsigned)((nbytes + 255) / 256), 256, 0, st>>>(
      expert + g.off_codes[m], expert + g.off_scales[m], tscale, rows, K, g.fmt, out);
  return cudaGetLastError();
}

cudaError_t launch_actquant(const Geo& g, const float* v, int rows, int K, uint8_t* codes,
                            uint8_t* scales, float gscale, cudaStream_t st) {
  const int af = g.afmt;   // the prefill regime's activation format
  if (af == MOE_MXFP8 || af == MOE_BF16) {
    const size_t total = (size_t)rows * (K / 32);
    if (total == 0) return cudaSuccess;
    actquant8_16_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(v, rows, K, af, codes, scales);
    return cudaGetLastError();
  }
  const int nb = K / fmt_block(af);
  const size_t total = (size_t)rows * nb;
  if (total == 0) return cudaSuccess;
  actquant_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(v, rows, K, af, gscale, codes,
                                                                  scales);
  return cudaGetLastError();
}

}  // namespace moe
