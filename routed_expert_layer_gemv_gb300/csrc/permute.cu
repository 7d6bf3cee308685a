// Permutation of routed (token, expert) pairs into expert-contiguous rows,
// atomic-free and deterministic.
//
// counts[e] = number of tokens routed to e; offsets = exclusive prefix sum
// over ascending e; the rows of expert e hold its tokens in ascending token
// order, so row_of[t*k+j] = offsets[e] + #{t' < t : t' routed to e}.  This
// placement is unique, so it is reproducible bit for bit.  (The pages do not
// describe this step; grouping tokens by expert is what lets each expert's
// weights be read once per step, the point of the expert cache in
// "FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二.)
//
// Block b owns tokens [b*128, b*128+128) (ballot scheme: permute_dev.cuh); a
// scan over blocks and experts turns block histograms and in-block ranks into
// the final rows.  No atomics anywhere.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "permute_dev.cuh"

namespace moe {

namespace {

using perm::kTokPerBlock;
using perm::kPermWarps;
using perm::block_excl_scan;

// Step 1 (multi-block): block histogram hist[b][e] and in-block ranks.
__global__ void __launch_bounds__(kTokPerBlock)
perm_hist_kernel(const int* __restrict__ idx, int N, int k, int E, int* __restrict__ hist,
                 int* __restrict__ rank) {
  extern __shared__ uint32_t sm[];
  uint32_t* cm = sm;                                              // [E][kPermWarps]
  int* rows = reinterpret_cast<int*>(sm + E * kPermWarps);        // [128][k]
  uint32_t* tb = reinterpret_cast<uint32_t*>(rows + kTokPerBlock * k);   // [128][ceil(E/32)]
  const int t_base = blockIdx.x * kTokPerBlock;
  perm::stage_rows(idx, N, k, t_base, rows);
  __syncthreads();
  perm::build_ballots_par(rows, k, E, min(kTokPerBlock, N - t_base), tb, cm);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = perm::block_count(cm, e);
  const int t = t_base + threadIdx.x;
  if (t < N)
    for (int j = 0; j < k; ++j) {
      const int e = rows[threadIdx.x * k + j];
      rank[(size_t)t * k + j] = e >= 0 && e < E ? perm::rank_in_block(cm, e) : 0;
    }
}

// Step 2 (one CTA of 1024 threads): per-expert block prefix, counts, offsets.
__global__ void __launch_bounds__(1024)
perm_scan_kernel(int* __restrict__ hist, int nblk, int E, int* __restrict__ counts,
                 int* __restrict__ offsets) {
  __shared__ int sh[33];
  perm::scan_hist(hist, nblk, E, counts, offsets, sh);
}

// Step 3: rows.
__global__ void perm_scatter_kernel(const int* __restrict__ idx, int N, int k, int E,
                                    const int* __restrict__ base, const int* __restrict__ rank,
                                    const int* __restrict__ offsets, int* __restrict__ row_of,
                                    int* __restrict__ tok_of) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= N * k) return;
  const int t = p / k;
  const int e = idx[p];
  if (e < 0 || e >= E) {   // invalid id: no row (the outputs are then unspecified, but in bounds)
    row_of[p] = -1;
    return;
  }
  const int b = t / kTokPerBlock;
  const int r = offsets[e] + base[(size_t)b * E + e] + rank[p];
  row_of[p] = r;
  if (r >= 0 && r < N * k) tok_of[r] = t;
}

// Whole permutation in one CTA (N <= 128 tokens).
__global__ void __launch_bounds__(kTokPerBlock)
perm_single_kernel(const int* __restrict__ idx, int N, int k, int E, int* __restrict__ counts,
                   int* __restrict__ offsets, int* __restrict__ row_of, int* __restrict__ tok_of) {
  extern __shared__ uint32_t sm[];
  uint32_t* cm = sm;                                           // [E][kPermWarps]
  int* off = reinterpret_cast<int*>(sm + E * kPermWarps);      // [E]
  int* sh = off + E;                                           // [33]
  int* rows = sh + 33;                                         // [128][k]
  uint32_t* tb = reinterpret_cast<uint32_t*>(rows + kTokPerBlock * k);   // [128][ceil(E/32)]
  perm::stage_rows(idx, N, k, 0, rows);
  __syncthreads();
  perm::build_ballots_par(rows, k, E, N, tb, cm);
  // exclusive scan of counts over e, kTokPerBlock experts at a time
  int carry = 0;
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int c = e < E ? perm::block_count(cm, e) : 0;
    int tot;
    const int ex = block_excl_scan(c, &tot, sh);
    if (e < E) {
      counts[e] = c;
      offsets[e] = carry + ex;
      off[e] = carry + ex;
    }
    carry += tot;
  }
  if (threadIdx.x == 0) offsets[E] = carry;
  __syncthreads();
  const int t = threadIdx.x;
  if (t < N) {
    for (int j = 0; j < k; ++j) {
      const int e = rows[t * k + j];
      if (e < 0 || e >= E) {   // invalid id: no row (outputs unspecified, but in bounds)
        row_of[(size_t)t * k + j] = -1;
        continue;
      }
      const int r = off[e] + perm::rank_in_block(cm, e);
      row_of[(size_t)t * k + j] = r;
      if (r >= 0 && r < N * k) tok_of[r] = t;
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(const Geo& g, int max_tokens) {
  size_t nblk = (max_tokens + kTokPerBlock - 1) / kTokPerBlock;
  return (nblk * g.E + (size_t)max_tokens * g.k) * sizeof(int);
}

cudaError_t launch_permute(const Geo& g, const int* idx, int N, int* counts, int* offsets,
                           int* row_of, int* tok_of, void* scratch, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  if (N <= kTokPerBlock) {
    size_t smem = (size_t)g.E * kPermWarps * 4 + (size_t)g.E * 4 + 33 * 4 + (size_t)kTokPerBlock * g.k * 4 +
                  (size_t)kTokPerBlock * ((g.E + 31) / 32) * 4;
    // up to 53 KB at E = 1024, k = 32
    cudaError_t e = ensure_smem_limit((const void*)perm_single_kernel, 64 * 1024);
    if (e != cudaSuccess) return e;
    perm_single_kernel<<<1, kTokPerBlock, smem, st>>>(idx, N, g.k, g.E, counts, offsets, row_of,
                                                      tok_of);
    return cudaGetLastError();
  }
  const int nblk = (N + kTokPerBlock - 1) / kTokPerBlock;
  cudaError_t err = launch_perm_hist(g, idx, N, scratch, st);
  if (err != cudaSuccess) return err;
  perm_scan_kernel<<<1, 1024, 0, st>>>(static_cast<int*>(scratch), nblk, g.E, counts, offsets);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_perm_scatter(g, idx, N, offsets, scratch, row_of, tok_of, st);
}

cudaError_t launch_perm_hist(const Geo& g, const int* idx, int N, void* scratch, cudaStream_t st) {
  const int nblk = (N + kTokPerBlock - 1) / kTokPerBlock;
  int* hist = static_cast<int*>(scratch);
  int* rank = hist + (size_t)nblk * g.E;
  perm_hist_kernel<<<nblk, kTokPerBlock, (size_t)g.E * kPermWarps * 4 + (size_t)kTokPerBlock * g.k * 4 +
                                          (size_t)kTokPerBlock * ((g.E + 31) / 32) * 4,
                     st>>>(idx, N, g.k, g.E, hist, rank);
  return cudaGetLastError();
}

cudaError_t launch_perm_scatter(const Geo& g, const int* idx, int N, const int* offsets, void* scratch,
                                int* row_of, int* tok_of, cudaStream_t st) {
  const int nblk = (N + kTokPerBlock - 1) / kTokPerBlock;
  const int* hist = static_cast<const int*>(scratch);
  const int* rank = hist + (size_t)nblk * g.E;
  perm_scatter_kernel<<<(N * g.k + 255) / 256, 256, 0, st>>>(idx, N, g.k, g.E, hist, rank, offsets, row_of,
                                                            tok_of);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------- no-alloc entry
// Scratch of moe_permute_noalloc (block histograms, then in-block ranks) lives
// in a file-scope device array, so the call never allocates.  In host code the
// array's name is only a host-side stand-in; each device's real address is
// looked up once with cudaGetSymbolAddress and passed to the kernels.
namespace {

constexpr size_t kNoAllocInts = 2u * 262144u;  // 2 MiB of int
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocInts];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};   // context the address belongs to

// Unique id of the current CUDA context (cuCtxGetId, through the runtime's
// driver entry points), 0 if it cannot be had.  A device's context can be
// destroyed and re-created (cudaDeviceReset), and the array's address in the
// new context need not be the old one, so the cached address is keyed by it.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
    cudaGetLastError();
    looked_up = true;
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int noalloc_fail(int code, const char* msg, char* errbuf, size_t errbuf_len) {
  if (errbuf && errbuf_len > 0) snprintf(errbuf, errbuf_len, "%s", msg);
  return code;
}

}  // namespace

extern "C" int moe_permute_noalloc(const int* idx, int N, int k, int E, int* counts, int* offsets,
                                   int* row_of, int* tok_of, void* stream, char* errbuf,
                                   size_t errbuf_len) {
  if (errbuf && errbuf_len > 0) errbuf[0] = '\0';
  if (E < 1 || E > moe::kMaxE)
    return noalloc_fail(MOE_ERR_ARG, "E must be in [1, 1024]", errbuf, errbuf_len);
  if (k < 1 || k > E || k > moe::kMaxK)
    return noalloc_fail(MOE_ERR_ARG, "k must be in [1, min(E, 32)]", errbuf, errbuf_len);
  if (N < 0) return noalloc_fail(MOE_ERR_ARG, "N must be >= 0", errbuf, errbuf_len);
  if (N == 0) return MOE_OK;
  if ((long long)N * k > 262144)
    return noalloc_fail(MOE_ERR_ARG, "N * k exceeds the 262144 pairs the static scratch holds",
                        errbuf, errbuf_len);
  const long long nblk = (N + 127) / 128;
  if (nblk * E > 262144)
    return noalloc_fail(MOE_ERR_ARG,
                        "ceil(N / 128) * E exceeds the 262144 histogram entries of the static scratch",
                        errbuf, errbuf_len);
  if (!idx || !counts || !offsets || !row_of || !tok_of)
    return noalloc_fail(MOE_ERR_ARG, "NULL pointer", errbuf, errbuf_len);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return noalloc_fail(MOE_ERR_CUDA, "cudaGetDevice failed or device index too large", errbuf,
                        errbuf_len);
  }
  int* scratch = nullptr;
  {
    // set-up, once per device (and again after its context was re-created),
    // with that device current
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    // (0 before the runtime created the device's context, or when the id
    // cannot be read: then the address is looked up on every call)
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // creates the context if needed
      if (e != cudaSuccess) {
        cudaGetLastError();
        return noalloc_fail(MOE_ERR_CUDA, cudaGetErrorString(e), errbuf, errbuf_len);
      }
      g_noalloc_ptr[dev] = static_cast<int*>(p);
      g_noalloc_ctx[dev] = current_context_id();
    }
    scratch = g_noalloc_ptr[dev];
  }
  moe::Geo g{};
  g.E = E;
  g.k = k;
  cudaError_t e = moe::launch_permute(g, idx, N, counts, offsets, row_of, tok_of, scratch,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, cudaGetErrorString(e), errbuf, errbuf_len);
  return MOE_OK;
}
