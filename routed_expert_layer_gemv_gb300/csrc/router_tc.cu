// Router logits of large batches on the 5th-generation tensor cores.
//
// The arithmetic of the mma.sync router (router.cu): W_r split once into
// three bf16 parts W = W0 + W1 + W2 (+ |r| <= 2^-24 |W|), x exact in bf16, so
// x W^T = sum_p x W_p^T.  Each 64-wide K stage sums its twelve products
// (three parts, smallest first, four 16-wide steps each) from zero in a TMEM
// accumulator (tcgen05.mma kind::f16, fp32 accumulation), and the stage's
// result is added to the running sums with ordinary fp32 adds in ascending K,
// so no long chain of tensor-core accumulations drifts.  (The pages do not
// define the router: the standard softmax top-k router, see router.cu.)
//
// One CTA per 128 tokens and K half (the halves only when the token tiles
// fill less than half of the SMs; the top-k kernel adds the two partial sums,
// first half first, and the bias) (MMA M = 128, N = E <= 256): warp 0 streams x and
// the three parts of W_r by TMA through a ring of K = 64 stages, warp 1 issues
// each stage's twelve MMAs into one of several accumulator slots, the
// epilogue warps (one or two per lane quarter) drain each stage's slot and
// add it to their rows' sums, then write the logits.  Every wait is bounded;
// on a timeout the CTA records an error, stops, waits for its own copies and
// MMAs (bounded again), frees its TMEM and returns.
#include <algorithm>

#include "common.cuh"
#include "router_dev.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kRM = 128;          // tokens per CTA (MMA M)
constexpr int kRK = 64;           // K per stage: one 128-byte row of bf16
constexpr int kRParts = 3;
constexpr int kRMaxStages = 4;
constexpr int kRMaxSlots = 4;
constexpr int kRSmemMin = 120 * 1024;   // one CTA per SM (each allocates all of TMEM)

__device__ __forceinline__ bool rwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (*abort_flag) return false;
  if (tc::mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  atomicExch(err, 1);
  return false;
}

__device__ __forceinline__ void rarrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::su32(bar)) : "memory");
}

// EW epilogue warps: 4 (E <= 128: one per lane quarter, all columns) or 8
// (two per quarter, 128 columns each).
template <int EW>
__global__ void __launch_bounds__(64 + 32 * EW, 1)
router_tc5_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, int N, int d,
                  int E, int stages, const float* __restrict__ bias, float* __restrict__ logits,
                  float* __restrict__ part2, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kRMaxStages], empty[kRMaxStages], accf[kRMaxSlots], acce[kRMaxSlots], fin;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t a_bytes = kRM * 128, st_bytes = a_bytes + (uint32_t)kRParts * E * 128;
  const int ncols = E <= 128 ? 128 : 256;           // TMEM columns of one accumulator slot
  const int nslot = 512 / ncols;
  const int m0 = blockIdx.x * kRM;
  // this CTA's K stages [kb, kb + nk) (blockIdx.y: the K half when split)
  const int nk_all = d / kRK, ns = gridDim.y;
  const int kb = (int)((long long)nk_all * blockIdx.y / ns);
  const int nk = (int)((long long)nk_all * (blockIdx.y + 1) / ns) - kb;
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kRMaxStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kRMaxSlots; ++a) {
      tc::mbar_init(&accf[a], 1);
      tc::mbar_init(&acce[a], EW);
    }
    tc::mbar_init(&fin, 1);
    s_abort = 0;
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kt = 0;
      for (; kt < nk; ++kt) {
        const int s = kt % stages;
        const uint32_t u = kt / stages;
        if (u > 0 && !rwait(&empty[s], (u - 1) & 1, &s_abort, err)) break;
        uint8_t* st = smem + (size_t)s * st_bytes;
        tc::mbar_expect_tx(&full[s], st_bytes);
        tc::tma_load_2d(st, &tx, &full[s], (kb + kt) * kRK, m0);   // rows past N read as zeros
        for (int p = 0; p < kRParts; ++p)
          tc::tma_load_2d(st + a_bytes + (size_t)p * E * 128, &tw, &full[s], (kb + kt) * kRK, p * E);
      }
      // copies in flight land before the CTA exits (bounded)
      const int first = kt > stages ? kt - stages : 0;
      for (int i = first; i < kt; ++i)
        if (!tc::mbar_wait(&full[i % stages], (i / stages) & 1)) { atomicExch(err, 1); break; }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(E);
      uint32_t step = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % stages;
        if (!rwait(&full[s], (kt / stages) & 1, &s_abort, err)) break;
        tc::fence_after();
        const uint32_t a_s = tc::su32(smem + (size_t)s * st_bytes), b_s = a_s + a_bytes;
        const int a = (int)(step % nslot);
        const uint32_t u = step / nslot;
        if (u > 0 && !rwait(&acce[a], (u - 1) & 1, &s_abort, err)) break;
        tc::fence_after();
        // the stage's twelve products from zero: the parts smallest first,
        // each over the four 16-wide steps
        for (int p = kRParts - 1; p >= 0; --p)
          for (int k16 = 0; k16 < kRK / 16; ++k16)
            tc::mma_bf16(tb + ncols * a, tc::sdesc_sw128(a_s + 32 * k16),
                         tc::sdesc_sw128(b_s + (uint32_t)p * E * 128 + 32 * k16), idesc,
                         p != kRParts - 1 || k16 > 0);
        tc::mma_commit(&accf[a]);
        tc::mma_commit(&empty[s]);   // the stage is free once its MMAs finish
        ++step;
      }
      tc::mma_commit(&fin);
      if (!tc::mbar_wait(&fin, 0)) atomicExch(err, 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2, hh = ew >> 2;
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
    const int row = 32 * (warp & 3) + lane;          // token m0 + row
    const int c0 = 128 * hh;                          // this warp's first column (expert)
    float sum[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) sum[i] = 0.f;
    const uint32_t nsteps = (uint32_t)nk;   // one accumulator slot per stage
    bool ok = true;
    for (uint32_t step = 0; step < nsteps && ok; ++step) {
      const int a = (int)(step % nslot);
      if (!rwait(&accf[a], (step / nslot) & 1, &s_abort, err)) { ok = false; break; }
      tc::fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tb + lq + ncols * a + c0 + 32 * c, v);   // columns past E: unused
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) sum[32 * c + i] += __uint_as_float(v[i]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) rarrive(&acce[a]);
    }
    const int t = m0 + row;
    if (ok && t < N) {
      // one K range: the logits; two: this half's partial sums (no bias)
      float* out = (blockIdx.y == 0 ? logits : part2) + (size_t)t * E + c0;
      const bool whole = ns == 1;
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (c0 + i < E) out[i] = whole ? sum[i] + (bias ? bias[c0 + i] : 0.f) : sum[i];
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 512);
}

// Per-token f16 exponent of x (the decode GEMV's conversion), one warp per token.
__global__ void token_exp_kernel(const __nv_bfloat16* __restrict__ x, int N, int d, int* __restrict__ xexp) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= N) return;
  const int s = rt::token_exp(x + (size_t)t * d, d);
  if ((threadIdx.x & 31) == 0) xexp[t] = s;
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// bf16 rows [rows][d], boxes of 64 elements x box_rows rows, 128B swizzle.
bool map_bf16(CUtensorMap* m, const void* base, int d, int rows, int box_rows) {
  EncodeFn fn = encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {(cuuint32_t)kRK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool router_tc5_shape_ok(const Geo& g) {
  return g.E >= 16 && g.E <= 256 && g.E % 16 == 0 && g.d % kRK == 0;
}

cudaError_t launch_router_tc5(const Geo& g, const __nv_bfloat16* x, int N, const __nv_bfloat16* Whl,
                              const float* bias, float* logits, float* part2, int* split, int* xexp, int* err,
                              cudaStream_t st) {
  if (!router_tc5_shape_ok(g) || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(Whl) & 15))
    return cudaErrorNotSupported;
  CUtensorMap tx, tw;
  if (!map_bf16(&tx, x, g.d, N, kRM) || !map_bf16(&tw, Whl, g.d, kRParts * g.E, g.E)) return cudaErrorNotSupported;
  const size_t st_bytes = (size_t)kRM * 128 + (size_t)kRParts * g.E * 128;
  const int stages = (int)std::min<size_t>(kRMaxStages, (226 * 1024) / st_bytes);
  if (stages < 2) return cudaErrorNotSupported;
  const int smem = (int)std::max<size_t>(kRSmemMin, 1024 + stages * st_bytes);
  const int mt = (N + kRM - 1) / kRM;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ns = part2 != nullptr && 2 * mt <= sms && g.d / kRK >= 2 ? 2 : 1;   // K halves
  *split = ns;
  const dim3 grid(mt, ns);
  cudaError_t e;
  if (g.E <= 128) {
    e = ensure_smem_limit((const void*)router_tc5_kernel<4>, smem);
    if (e != cudaSuccess) return e;
    router_tc5_kernel<4><<<grid, 64 + 32 * 4, smem, st>>>(tx, tw, N, g.d, g.E, stages, bias, logits, part2, err);
  } else {
    e = ensure_smem_limit((const void*)router_tc5_kernel<8>, smem);
    if (e != cudaSuccess) return e;
    router_tc5_kernel<8><<<grid, 64 + 32 * 8, smem, st>>>(tx, tw, N, g.d, g.E, stages, bias, logits, part2, err);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || xexp == nullptr) return e;
  token_exp_kernel<<<(N + 7) / 8, 256, 0, st>>>(x, N, g.d, xexp);
  return cudaGetLastError();
}

}  // namespace moe
