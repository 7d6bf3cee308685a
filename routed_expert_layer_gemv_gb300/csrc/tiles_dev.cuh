// The prefill GEMM's tile list, shared by its own launch (build_tiles_kernel)
// and the routing CTA of large batches, which builds the hits' tiles right
// after its LRU step.
#pragma once
#include "common.cuh"

namespace moe {
namespace tl {

struct Tile {
  int slot;       // pool buffer of the expert (Geo::shb: the shared expert)
  int row_start;  // first permuted row of the tile
  int row_end;    // one past the expert's last row
  int pb;         // padded 128-row block of the tile's activation scales
  int ent;        // the expert's entry in the launch (its interleaved weight scales)
  int pad[3];
};

constexpr int kSharedKey = -2;   // weight key of the shared expert's buffer (never an expert's)

// One CTA (any blockDim): the tiles of one launch range (mode: the step's
// hits, its misses, or all; with_shared: the shared expert's rows last) from
// the step record, 128 rows each by expert in access order; n_tiles[0] = the
// tile count, n_tiles[1] = the entry count.  sh (33 ints) and carry: shared
// memory of the caller.  Ends with the CTA synchronised.
MOE_DEV void build_tiles(const StepRecord* __restrict__ rec, const int* __restrict__ offsets,
                         const int* __restrict__ pbase, int E, int S, int X, int shb, int key0, int N, int k,
                         int mode, int with_shared, Tile* __restrict__ tiles, int* __restrict__ ents,
                         int* __restrict__ n_tiles, int* sh, int* carry) {
  // entries: buffer ents[i], then the key of its weights ekey[i] (key0 +
  // expert; kSharedKey for the shared expert) and efresh[i] = 1 where the
  // buffer was (re)filled by this step (a miss)
  int* ekey = ents + (E + 1);
  int* efresh = ekey + (E + 1);
  int& cr = *carry;
  const int U = min(max(rec->U, 0), E), nh = min(max(rec->n_hit, 0), U);
  const int b = mode == kRangeHits ? 0 : nh, e = mode == kRangeHits ? nh : U;
  const int nr = max(0, e - b);
  const int n_ent = nr + (with_shared ? 1 : 0);
  if (threadIdx.x == 0) cr = 0;
  __syncthreads();
  const int* ae = reinterpret_cast<const int*>(rec + 1);
  const int* as = ae + E;
  const int* abuf = ae + 3 * E;
  for (int e0 = 0; e0 < n_ent; e0 += blockDim.x) {
    const int i = e0 + threadIdx.x;
    int slot = -1, r0 = 0, nrows = 0, pb0 = 0, key = -1, fresh = 0;
    if (i < nr) {
      const int ex = ae[b + i], ls = as[b + i], bb = abuf[b + i];
      if (ex >= 0 && ex < E && ls >= 0 && ls < S && b + i - S < X && bb >= 0 && bb <= S + X && bb != S) {
        slot = bb;
        r0 = offsets[ex];
        nrows = offsets[ex + 1] - r0;
        pb0 = pbase[ex];
        key = key0 + ex;
        fresh = b + i >= nh;
      }
    } else if (i < n_ent) {
      slot = shb;
      r0 = N * k;
      nrows = N;
      pb0 = pbase[E];
      key = kSharedKey;
    }
    if (i < n_ent) {
      ents[i] = nrows > 0 ? slot : -1;
      ekey[i] = key;
      efresh[i] = fresh;
    }
    const int nt = (nrows + kPrefillTileRows - 1) / kPrefillTileRows;
    // block exclusive scan of nt
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = nt;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
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
    const int base = cr + sh[warp] + inc - nt;
    for (int t = 0; t < nt; ++t) {
      Tile tile;
      tile.slot = slot;
      tile.row_start = r0 + t * kPrefillTileRows;
      tile.row_end = r0 + nrows;
      tile.pb = pb0 + t;
      tile.ent = i;
      tile.pad[0] = tile.pad[1] = tile.pad[2] = 0;
      tiles[base + t] = tile;
    }
    __syncthreads();
    if (threadIdx.x == 0) cr += sh[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    n_tiles[0] = cr;
    n_tiles[1] = n_ent;
  }
  __syncthreads();
}

}  // namespace tl
}  // namespace moe
