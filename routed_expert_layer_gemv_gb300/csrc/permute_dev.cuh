// Device pieces of the atomic-free permutation, shared by the permutation
// kernels and the fused decode routing tail.
//
// Block b owns 128 consecutive tokens.  For every expert e and warp-sized
// group of 32 tokens the block holds the ballot of the tokens routed to e
// (built from per-token expert bitmaps, no loop over the experts).  Popcounts
// of the ballots give the block histogram and each pair's rank among the
// block's earlier tokens routed to the same expert.
#pragma once
#include "common.cuh"

namespace moe {
namespace perm {

constexpr int kTokPerBlock = 128;
constexpr int kPermWarps = kTokPerBlock / 32;

// Stage the id rows of tokens [t_base, t_base + 128) into shared memory
// (threads of the first 128 cover one token each; k <= 32).
MOE_DEV void stage_rows(const int* __restrict__ idx, int N, int k, int t_base, int* rows) {
  for (int v = threadIdx.x; v < kTokPerBlock * k; v += blockDim.x) {
    const int t = t_base + v / k;
    rows[v] = t < N ? idx[(size_t)t_base * k + v] : 0x7fffffff;
  }
}

// Ballots of the block's tokens per expert: cm[e * kPermWarps + w] bit l =
// token 32 w + l is routed to e.  Built by the whole CTA (any blockDim)
// without a loop over the experts: each token's expert set becomes a bitmap
// tb[t][E/32] (one thread per token word, k compares), then thread (e, w)
// gathers bit e of warp w's tokens.  nt = tokens of the block (<= 128); tb: 128 * ceil(E/32)
// words of scratch.  Ends with the CTA synchronised.
MOE_DEV void build_ballots_par(const int* rows, int k, int E, int nt, uint32_t* tb, uint32_t* cm) {
  const int W = (E + 31) >> 5;
  for (int v = threadIdx.x; v < nt * W; v += blockDim.x) {
    const int t = v / W, wd = v % W;
    uint32_t b = 0;
    for (int j = 0; j < k; ++j) {
      const int e = rows[t * k + j];
      if ((e >> 5) == wd) b |= 1u << (e & 31);
    }
    tb[t * W + wd] = b;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < E * kPermWarps; v += blockDim.x) {
    const int e = v % E, w = v / E;   // consecutive threads: consecutive experts, one broadcast word
    const int l1 = min(32, nt - 32 * w);
    uint32_t b = 0;
    for (int l = 0; l < l1; ++l) b |= ((tb[(32 * w + l) * W + (e >> 5)] >> (e & 31)) & 1u) << l;
    cm[e * kPermWarps + w] = b;
  }
  __syncthreads();
}

// Rank of this thread's token among the block's earlier tokens routed to e
// (thread t of the first 128 = token t of the block).
MOE_DEV int rank_in_block(const uint32_t* cm, int e) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int r = 0;
  for (int w = 0; w < warp; ++w) r += __popc(cm[e * kPermWarps + w]);
  return r + __popc(cm[e * kPermWarps + warp] & ((1u << lane) - 1u));
}

MOE_DEV int block_count(const uint32_t* cm, int e) {
  int c = 0;
  for (int w = 0; w < kPermWarps; ++w) c += __popc(cm[e * kPermWarps + w]);
  return c;
}

// Block-wide exclusive scan over blockDim.x (<= 1024) threads; *total gets
// the sum.  sh: >= 33 ints of shared memory.
MOE_DEV int block_excl_scan(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int s = lane < nw ? sh[lane] : 0;
    int si = s;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += u;
    }
    if (lane < nw) sh[lane] = si - s;
    if (lane == 31) sh[32] = si;
  }
  __syncthreads();
  const int res = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return res;
}

// Thread e (< E) of a CTA of >= E threads: the block histograms hist[b][e]
// (nblk blocks) become their exclusive prefixes over b, counts[e] gets the
// expert's total and offsets the exclusive prefix over e (offsets[E]: all
// rows).  Returns thread e's count (0 for e >= E).  sh: >= 33 ints.
MOE_DEV int scan_hist(int* __restrict__ hist, int nblk, int E, int* __restrict__ counts, int* __restrict__ offsets,
                      int* sh) {
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E) {
    // exclusive prefix over blocks, 16 loads in flight at a time
    for (int b0 = 0; b0 < nblk; b0 += 16) {
      int c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = b0 + i < nblk ? hist[(size_t)(b0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (b0 + i < nblk) hist[(size_t)(b0 + i) * E + e] = tot;
        tot += c[i];
      }
    }
  }
  int all;
  const int off = block_excl_scan(e < E ? tot : 0, &all, sh);
  if (e < E) {
    counts[e] = tot;
    offsets[e] = off;
  }
  if (e == 0) offsets[E] = all;
  return tot;
}

}  // namespace perm
}  // namespace moe
