// Device-driven miss fill: a copy kernel reads the step record on the GPU and
// pulls each missed expert of one wave from the pinned host pool (reached over
// NVLink-C2C through unified addressing) into its slot.  The host never waits
// for the routing, so a decode step runs without a host round trip.  This is
// the variant of the default fill (cudaMemcpyAsync from pinned host memory on
// side streams), which follows the pages' decode path: misses are loaded into
// the GPU's expert cache from host memory ("FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).
#include "common.cuh"

namespace moe {

namespace {

constexpr int kFillThreads = 256;
constexpr size_t kFillChunk = 64 * 1024;

__global__ void __launch_bounds__(kFillThreads)
fill_copy_kernel(const StepRecord* __restrict__ rec, int E, int S, int wave,
                 const uint8_t* __restrict__ pool, uint8_t* __restrict__ slots, size_t ebytes,
                 int chunks) {
  const int U = rec->U, nh = rec->n_hit;
  const int b = max(nh, wave * S), e = min((wave + 1) * S, U);
  const int m = blockIdx.x / chunks, ch = blockIdx.x % chunks;
  if (b + m >= e) return;
  const int i = b + m;
  const int ex = rec_expert(const_cast<StepRecord*>(rec))[i];
  const int sl = rec_slot(const_cast<StepRecord*>(rec), E)[i];
  if (ex < 0 || ex >= E || sl < 0 || sl >= S) return;
  const size_t off = (size_t)ch * kFillChunk;
  if (off >= ebytes) return;
  const size_t n16 = (min(kFillChunk, ebytes - off)) / 16;
  const uint4* src = reinterpret_cast<const uint4*>(pool + (size_t)ex * ebytes + off);
  uint4* dst = reinterpret_cast<uint4*>(slots + (size_t)sl * ebytes + off);
  for (size_t v = threadIdx.x; v < n16; v += 4 * kFillThreads) {
    uint4 r[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (v + u * kFillThreads < n16) r[u] = src[v + u * kFillThreads];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (v + u * kFillThreads < n16) dst[v + u * kFillThreads] = r[u];
  }
}

}  // namespace

cudaError_t launch_fill_copy(const Geo& g, const StepRecord* rec, int wave, int max_misses,
                             const uint8_t* pool_dev, uint8_t* slots, cudaStream_t st) {
  const int chunks = (int)((g.ebytes + kFillChunk - 1) / kFillChunk);
  const long long grid = (long long)chunks * max_misses;
  if (grid <= 0) return cudaSuccess;
  fill_copy_kernel<<<(unsigned)grid, kFillThreads, 0, st>>>(rec, g.E, g.S, wave, pool_dev, slots,
                                                            g.ebytes, chunks);
  return cudaGetLastError();
}

}  // namespace moe
