// Miss fills by copy kernels: each reads the step record on the GPU and pulls
// missed experts from the pinned host pool (reached over NVLink-C2C through
// unified addressing) into the buffers the record names.  fill_copy_kernel
// (MOE_FILL_DEVICE) spreads one step's misses over the whole GPU;
// fill_sm_kernel (MOE_FILL_KERNEL) copies one chunk of the miss list on a few
// SMs the expert GEMV leaves free.  Both follow the pages' decode path: misses
// are loaded into the GPU's expert cache from host memory ("FreeToken：把 284B
// MoE 塞进游戏 PC", zhichai.net, §二 "Decode" paragraph).
#include <algorithm>

#include "common.cuh"

namespace moe {

namespace {

constexpr int kFillThreads = 256;
constexpr size_t kFillChunk = 64 * 1024;

// Copy chunk `ch` of one expert, 4 x 16 bytes in flight per thread.
__device__ __forceinline__ void copy_chunk(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                           size_t ebytes, int ch) {
  const size_t off = (size_t)ch * kFillChunk;
  if (off >= ebytes) return;
  const size_t n16 = (min(kFillChunk, ebytes - off)) / 16;
  const uint4* s = reinterpret_cast<const uint4*>(src + off);
  uint4* d = reinterpret_cast<uint4*>(dst + off);
  for (size_t v = threadIdx.x; v < n16; v += 4 * kFillThreads) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (v + u * kFillThreads < n16) r[u] = s[v + u * kFillThreads];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (v + u * kFillThreads < n16) d[v + u * kFillThreads] = r[u];
  }
}

// A buffer a fill may write: an LRU slot's or a spare, never the shared expert's.
__device__ __forceinline__ bool fill_buf_ok(int b, int S, int X) { return b >= 0 && b <= S + X && b != S; }

// CTA (miss m, chunk ch): access n_hit + m, from the pool to its buffer.
__global__ void __launch_bounds__(kFillThreads)
fill_copy_kernel(const StepRecord* __restrict__ rec, int E, int S, int X, const uint8_t* __restrict__ pool,
                 uint8_t* __restrict__ slots, size_t ebytes, int chunks) {
  const int U = min(max(rec->U, 0), E), nh = min(max(rec->n_hit, 0), U);
  const int i = nh + blockIdx.x / chunks, ch = blockIdx.x % chunks;
  if (i >= U || i - S >= X) return;
  const int ex = rec_expert(const_cast<StepRecord*>(rec))[i];
  const int b = rec_buf(const_cast<StepRecord*>(rec), E)[i];
  if (ex < 0 || ex >= E || !fill_buf_ok(b, S, X)) return;
  copy_chunk(pool + (size_t)ex * ebytes, slots + (size_t)b * ebytes, ebytes, ch);
}

// SM fill of one chunk of the miss list: kFillSms CTAs, one per SM (the
// shared memory they reserve, more than half an SM's, keeps two off one SM and
// keeps the expert GEMV, which takes nearly all of it, off theirs), copy the
// chunk's misses from the pinned host pool to their buffers.  The m = U - n_hit
// misses form miss_chunks(m) chunks split by miss_chunk -- the split the host
// makes from its copy of the record -- and a launch for a chunk past them
// copies nothing.  Each expert is cut into pieces of kFillPiece bytes dealt
// round-robin to the CTAs; a piece is one load of kFillSmUnroll x 16 bytes per
// thread, all in flight before the stores.
constexpr int kFillSmThreads = 1024;
constexpr int kFillSmUnroll = 8;
constexpr size_t kFillPiece = (size_t)kFillSmThreads * kFillSmUnroll * 16;
constexpr int kFillSmSmem = 120 * 1024;

__global__ void __launch_bounds__(kFillSmThreads, 1)
fill_sm_kernel(const StepRecord* __restrict__ rec, int E, int S, int X, int chunk,
               const uint8_t* __restrict__ pool, uint8_t* __restrict__ slots, size_t ebytes) {
  const int U = min(max(rec->U, 0), E), nh = min(max(rec->n_hit, 0), U);
  const int m = U - nh;
  const int nch = miss_chunks(m);
  if (chunk >= nch) return;
  int lo, hi;
  miss_chunk(m, chunk, nch, &lo, &hi);
  const int i0 = nh + lo;
  const int i1 = min(nh + hi, S + X);
  if (i1 <= i0) return;
  const int* ab = rec_buf(const_cast<StepRecord*>(rec), E);
  const int* ae = rec_expert(const_cast<StepRecord*>(rec));
  const long long P = (long long)((ebytes + kFillPiece - 1) / kFillPiece);
  const long long total = (long long)(i1 - i0) * P;
  for (long long q = blockIdx.x; q < total; q += gridDim.x) {
    const int i = i0 + (int)(q / P);
    const size_t off = (size_t)(q % P) * kFillPiece;
    const int ex = ae[i], b = ab[i];
    if (ex < 0 || ex >= E || !fill_buf_ok(b, S, X)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(pool + (size_t)ex * ebytes + off);
    uint4* dst = reinterpret_cast<uint4*>(slots + (size_t)b * ebytes + off);
    const int n16 = (int)(min(kFillPiece, ebytes - off) / 16);
    uint4 r[kFillSmUnroll];
#pragma unroll
    for (int u = 0; u < kFillSmUnroll; ++u) {
      const int v = threadIdx.x + u * kFillSmThreads;
      if (v < n16) r[u] = src[v];
    }
#pragma unroll
    for (int u = 0; u < kFillSmUnroll; ++u) {
      const int v = threadIdx.x + u * kFillSmThreads;
      if (v < n16) dst[v] = r[u];
    }
  }
}

// dst <- src, bytes a multiple of 16, both 16-byte aligned (src may be host
// memory reached through unified addressing).
__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<size_t>((n16 + 255) / 256, 64);
  copy16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

cudaError_t launch_fill_copy(const Geo& g, const StepRecord* rec, int max_misses,
                             const uint8_t* pool_dev, uint8_t* slots, cudaStream_t st) {
  const int chunks = (int)((g.ebytes + kFillChunk - 1) / kFillChunk);
  const long long grid = (long long)chunks * max_misses;
  if (grid <= 0) return cudaSuccess;
  fill_copy_kernel<<<(unsigned)grid, kFillThreads, 0, st>>>(rec, g.E, g.S, g.X, pool_dev, slots, g.ebytes,
                                                            chunks);
  return cudaGetLastError();
}

cudaError_t launch_fill_sm(const Geo& g, const StepRecord* rec, int chunk, const uint8_t* pool_dev,
                           uint8_t* slots, cudaStream_t st) {
  cudaError_t e = ensure_smem_limit((const void*)fill_sm_kernel, kFillSmSmem);
  if (e != cudaSuccess) return e;
  fill_sm_kernel<<<kFillSms, kFillSmThreads, kFillSmSmem, st>>>(rec, g.E, g.S, g.X, chunk, pool_dev, slots,
                                                               g.ebytes);
  return cudaGetLastError();
}

}  // namespace moe
