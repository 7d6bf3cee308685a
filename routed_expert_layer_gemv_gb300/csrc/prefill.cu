// Prefill expert FFN: grouped GEMM on tcgen05 block-scaled FP4 MMAs.
//
// A prefill chunk gives each expert hundreds of tokens, so the expert FFN is a
// dense contraction (FreeToken's prefill streams whole layers of experts and
// is bound by compute once they are resident: "FreeToken：把 284B MoE 塞进游戏
// PC", zhichai.net, §二 "Prefill" paragraph).  FP4 x FP4 MMAs need FP4
// activations, so x and h go through the block quantiser of the weight format
// (actquant.cuh).  Steps:
//  1. gather_quant: row r of the permuted activations = quant(x[tok_of[r]]);
//     rows N*k .. N*k+N-1 hold every token for the shared expert.
//  2. build_tiles: the launch's experts (hits, or all misses, + shared) cut
//     into M tiles of 128 rows; the last tile of an expert is ragged (its extra
//     rows are computed and dropped).
//  3. gemm_gateup: CTA = (M tile, 128 rows of d_ff); per K tile of 256 codes
//     TMA brings A (128 x 128 B), B_gate and B_up (128 x 128 B each) into
//     shared memory (128B swizzle), cp.async brings the block scales; four
//     warps write the scales to TMEM; one thread issues the MMAs into two TMEM
//     accumulators (gate, up).  Epilogue: h = SiLU(a) * u, re-quantised to FP4.
//  4. gemm_down: CTA = (M tile, 128 rows of d_model), O = h W_d^T in fp32.
// Every wait is bounded (~2 s); on a timeout the CTA records an error, waits
// for its own copies and MMAs (bounded again), frees its TMEM and returns.
#include <cstdio>

#include "actquant.cuh"
#include "common.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kStages = 3;
constexpr int kTileRows = 128;          // M and N of one MMA tile
constexpr int kKTileBytes = 128;        // 256 FP4 codes per K tile
constexpr int kOpBytes = kTileRows * kKTileBytes;   // 16 KB per operand tile

struct Tile {
  int slot;       // slot of the expert (n_slots = the shared expert)
  int row_start;  // first permuted row of the tile
  int row_end;    // one past the expert's last row
  int pad;
};

// ---------------------------------------------------------------- step 1
__global__ void gather_quant_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ tok_of,
                                    int N, int k, int d, int fmt, float gx, int with_shared,
                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int nb = d / 32;                       // 32-value groups per row
  const size_t rows = (size_t)N * k + (with_shared ? N : 0);
  const size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= rows * nb) return;
  const size_t r = v / nb;
  const int c = (int)(v % nb);
  const int tok = r < (size_t)N * k ? tok_of[r] : (int)(r - (size_t)N * k);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * d + (size_t)c * 32);
  float vals[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = src[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      vals[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      vals[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  uint32_t words[4];
  uint8_t* dst = codes + r * (d / 2) + (size_t)c * 16;
  if (fmt == MOE_MXFP4) {
    scales[r * (d / 32) + c] = (uint8_t)quant_mx32(vals, words);
  } else {
    uint32_t w2[2];
    scales[r * (d / 16) + 2 * c] = (uint8_t)quant_nv16(vals, gx, words);
    scales[r * (d / 16) + 2 * c + 1] = (uint8_t)quant_nv16(vals + 16, gx, w2);
    words[2] = w2[0];
    words[3] = w2[1];
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

// ---------------------------------------------------------------- step 2
__global__ void __launch_bounds__(1024)
build_tiles_kernel(const StepRecord* __restrict__ rec, const int* __restrict__ offsets, int E, int S,
                   int X, int N, int k, int mode, int with_shared, Tile* __restrict__ tiles,
                   int* __restrict__ n_tiles) {
  __shared__ int sh[33];
  __shared__ int carry;
  const int U = min(max(rec->U, 0), E), nh = min(max(rec->n_hit, 0), U);
  const int b = mode == kRangeHits ? 0 : nh, e = mode == kRangeHits ? nh : U;
  const int nr = max(0, e - b);
  const int n_ent = nr + (with_shared ? 1 : 0);
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int* ae = reinterpret_cast<const int*>(rec + 1);
  const int* as = ae + E;
  for (int e0 = 0; e0 < n_ent; e0 += blockDim.x) {
    const int i = e0 + threadIdx.x;
    int slot = -1, r0 = 0, nrows = 0;
    if (i < nr) {
      const int ex = ae[b + i], ls = as[b + i];
      if (ex >= 0 && ex < E && ls >= 0 && ls < S && b + i - S < X) {
        slot = access_slot(as, S, b + i);
        r0 = offsets[ex];
        nrows = offsets[ex + 1] - r0;
      }
    } else if (i < n_ent) {
      slot = S;
      r0 = N * k;
      nrows = N;
    }
    const int nt = (nrows + kTileRows - 1) / kTileRows;
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
    const int base = carry + sh[warp] + inc - nt;
    for (int t = 0; t < nt; ++t) {
      Tile tl;
      tl.slot = slot;
      tl.row_start = r0 + t * kTileRows;
      tl.row_end = r0 + nrows;
      tl.pad = 0;
      tiles[base + t] = tl;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += sh[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_tiles = carry;
}

// ---------------------------------------------------------------- GEMM pieces
struct GemmArgs {
  const Tile* tiles;
  const int* n_tiles;
  const uint8_t* a_scales;     // [rows, K/blk] of the A operand (activations)
  const uint8_t* slots;        // slot pool (n_slots + 1 experts; the last is shared)
  size_t ebytes;
  size_t w_scales_off[3];
  int K;                       // contraction length
  int rows_out;                // d_ff (phase 1) or d_model (phase 2)
  int fmt;
  float act_scale;             // NVFP4 static activation scale of A (1 for MXFP4)
  float w_tscale_default;
  int* err;
  // phase 1 outputs
  uint8_t* h_codes;
  uint8_t* h_scales;
  float act_scale_h;
  // phase 2 output
  float* O;
  int O_ld;
};

// bytes of one row's block scales in a K tile of 256 codes
__device__ __forceinline__ int scale_bytes(int fmt) { return fmt == MOE_MXFP4 ? 8 : 16; }

// Copy `bytes` (8 or 16) from global to shared asynchronously.
__device__ __forceinline__ void cp_async(void* dst, const void* src, int bytes) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(tc::su32(dst)), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(tc::su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Write the scale groups of one operand tile (128 rows, staged in shared
// memory as [row][sb bytes]) into TMEM at column `col0`: group g goes to
// columns col0 + 4g .. + 3, lane 32w + i, column 4g + j = row 32j + i.
__device__ __forceinline__ void scales_to_tmem(const uint8_t* st, int sb, uint32_t tmem_lane_base,
                                               uint32_t col0) {
  const int i = threadIdx.x & 31;
  const int groups = sb / 4;
  for (int g = 0; g < groups; ++g) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint32_t*>(st + (32 * j + i) * sb + 4 * g);
    tc::tmem_st4(tmem_lane_base + col0 + 4 * g, w[0], w[1], w[2], w[3]);
  }
}

// Issue the MMAs of one K tile: nb B operands (1 or 2) into accumulators at
// columns 0, 128 (each N = 128).
__device__ __forceinline__ void issue_mmas(int fmt, uint32_t tb, uint32_t a_smem, const uint32_t* b_smem,
                                           int nb, uint32_t sfa_col, const uint32_t* sfb_col,
                                           bool acc_first) {
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t ad = tc::sdesc_sw128(a_smem + 32 * kk);
    for (int bi = 0; bi < nb; ++bi) {
      const uint64_t bd = tc::sdesc_sw128(b_smem[bi] + 32 * kk);
      const bool acc = acc_first || kk > 0;
      if (fmt == MOE_MXFP4) {
        const uint32_t sf = 2 * (kk & 1), g = kk >> 1;
        tc::mma_mxf4(tb + 128 * bi, ad, bd, tc::idesc_fp4(128, true, sf, sf), tb + sfa_col + 4 * g,
                     tb + sfb_col[bi] + 4 * g, acc);
      } else {
        tc::mma_nvf4(tb + 128 * bi, ad, bd, tc::idesc_fp4(128, false, 0, 0), tb + sfa_col + 4 * kk,
                     tb + sfb_col[bi] + 4 * kk, acc);
      }
    }
  }
}

// The shared mainloop of both phases: A = activations (tensor map ta, rows
// row_start..), nb weight operands (tensor maps tw[bi], rows n0.., slot z).
// On return the accumulators hold the full-K products (or *bad is set).
template <int NB>
__device__ bool gemm_mainloop(const GemmArgs& p, const CUtensorMap* ta, const CUtensorMap* const* tw,
                              const Tile& tile, int n0, uint8_t* smem, uint64_t* full, uint64_t* done,
                              uint32_t tb, uint32_t scol0, int* n_committed) {
  const int nkt = p.K / 256;
  const int sb = scale_bytes(p.fmt);
  const int stage_bytes = (1 + NB) * kOpBytes;
  uint8_t* sc_base = smem + kStages * stage_bytes;           // [stage][1+NB][128][sb]
  const int sc_stage = (1 + NB) * kTileRows * 16;
  const uint32_t lane_base = (uint32_t)(32 * (threadIdx.x >> 5)) << 16;
  const uint32_t scols = (uint32_t)(1 + NB) * (uint32_t)(sb);  // TMEM columns per stage (4 per group)
  const int row = threadIdx.x;                                // one scale row per thread
  const uint8_t* wbase = p.slots + (size_t)tile.slot * p.ebytes;
  bool ok = true;

  auto issue_loads = [&](int kt) {
    const int s = kt % kStages;
    uint8_t* st = smem + s * stage_bytes;
    if (threadIdx.x == 0) {
      tc::mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
      tc::tma_load_2d(st, ta, &full[s], kt * kKTileBytes, tile.row_start);
      for (int bi = 0; bi < NB; ++bi)
        tc::tma_load_3d(st + (1 + bi) * kOpBytes, tw[bi], &full[s], kt * kKTileBytes, n0, tile.slot);
    }
    // block scales of this K tile: A rows, then each weight operand's rows
    uint8_t* sst = sc_base + s * sc_stage;
    cp_async(sst + row * sb, p.a_scales + (size_t)(tile.row_start + row) * (p.K / (p.fmt == MOE_MXFP4 ? 32 : 16)) +
                                 (size_t)kt * sb, sb);
    for (int bi = 0; bi < NB; ++bi) {
      const uint8_t* ws = wbase + p.w_scales_off[bi] + (size_t)(n0 + row) * (p.K / (p.fmt == MOE_MXFP4 ? 32 : 16)) +
                          (size_t)kt * sb;
      cp_async(sst + (1 + bi) * kTileRows * sb + row * sb, ws, sb);
    }
    cp_async_commit();
  };

  for (int kt = 0; kt < kStages - 1 && kt < nkt; ++kt) issue_loads(kt);
  for (int kt = 0; kt < nkt; ++kt) {
    const int s = kt % kStages;
    // keep the pipeline kStages - 1 tiles ahead: refill the stage of tile kt-1
    if (kt + kStages - 1 < nkt) {
      if (kt >= 1) {
        const int ps = (kt - 1) % kStages;
        bool w = true;
        if (threadIdx.x == 0) w = tc::mbar_wait(&done[ps], (uint32_t)(((kt - 1) / kStages) & 1));
        if (!__syncthreads_and(w)) { ok = false; break; }
      }
      issue_loads(kt + kStages - 1);
      cp_async_wait<kStages - 1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // scales of tile kt -> TMEM (its stage's previous MMAs finished: waited above)
    const uint8_t* sst = sc_base + s * sc_stage;
    const uint32_t c0 = scol0 + (uint32_t)s * scols;
    scales_to_tmem(sst, sb, tb + lane_base, c0);
    for (int bi = 0; bi < NB; ++bi)
      scales_to_tmem(sst + (1 + bi) * kTileRows * sb, sb, tb + lane_base, c0 + (uint32_t)(1 + bi) * (uint32_t)(sb));
    tc::tmem_st_wait();
    tc::fence_before();
    __syncthreads();
    bool w = true;
    if (threadIdx.x == 0) {
      tc::fence_after();
      w = tc::mbar_wait(&full[s], (uint32_t)((kt / kStages) & 1));
      if (w) {
        uint8_t* st = smem + s * stage_bytes;
        uint32_t bs[2], sfb[2];
        for (int bi = 0; bi < NB; ++bi) {
          bs[bi] = tc::su32(st + (1 + bi) * kOpBytes);
          sfb[bi] = c0 + (uint32_t)(1 + bi) * (uint32_t)(sb);
        }
        issue_mmas(p.fmt, tb, tc::su32(st), bs, NB, c0, sfb, kt > 0);
        tc::mma_commit(&done[s]);
        ++*n_committed;
      }
    }
    if (!__syncthreads_and(w)) { ok = false; break; }
  }
  // all MMAs: wait for the last commit (they complete in order)
  if (ok && nkt > 0) {
    const int last = nkt - 1;
    const bool w = tc::mbar_wait(&done[last % kStages], (uint32_t)((last / kStages) & 1));
    ok = __syncthreads_and(w);
  }
  tc::fence_after();
  return ok;
}

// Bounded clean-up after an error: let copies and MMAs in flight finish.
__device__ void drain(uint64_t* full, uint64_t* done) {
  cp_async_wait<0>();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < 200000000LL) {
    }
  }
  __syncthreads();
}

template <int FMT>
__global__ void __launch_bounds__(128, 1)
gemm_gateup_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tg,
                   const __grid_constant__ CUtensorMap tu, GemmArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kStages], done[kStages];
  __shared__ uint32_t tmem_base;
  if ((int)blockIdx.x >= *p.n_tiles) return;
  const Tile tile = p.tiles[blockIdx.x];
  const int n0 = blockIdx.y * kTileRows;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&done[s], 1); }
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = tmem_base;
  const CUtensorMap* tw[2] = {&tg, &tu};
  int n_committed = 0;
  const bool ok = gemm_mainloop<2>(p, &ta, tw, tile, n0, smem, full, done, tb, 256, &n_committed);
  if (!ok) {
    if (threadIdx.x == 0) atomicExch(p.err, 1);
    drain(full, done);
  } else {
    // epilogue: row m of the tile, 128 gate and 128 up columns
    const int m = threadIdx.x;
    const int r = tile.row_start + m;
    const bool live = r < tile.row_end;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float* ts = reinterpret_cast<const float*>(p.slots + (size_t)tile.slot * p.ebytes +
                                                     p.w_scales_off[2]);  // tensor scales
    const float sg = FMT == MOE_MXFP4 ? 1.0f : ts[0] * p.act_scale;
    const float su = FMT == MOE_MXFP4 ? 1.0f : ts[1] * p.act_scale;
    const int f = p.rows_out;
    for (int c = 0; c < 4; ++c) {
      uint32_t gv[32], uv[32];
      tc::tmem_ld32(tb + lane_base + 32 * c, gv);
      tc::tmem_ld32(tb + lane_base + 128 + 32 * c, uv);
      tc::tmem_ld_wait();
      float h[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float a = __uint_as_float(gv[i]) * sg, u = __uint_as_float(uv[i]) * su;
        h[i] = a / (1.0f + expf(-a)) * u;
      }
      if (live) {
        const int col = n0 + 32 * c;
        uint32_t words[4];
        if (FMT == MOE_MXFP4) {
          p.h_scales[(size_t)r * (f / 32) + col / 32] = (uint8_t)quant_mx32(h, words);
        } else {
          uint32_t w2[2];
          p.h_scales[(size_t)r * (f / 16) + col / 16] = (uint8_t)quant_nv16(h, p.act_scale_h, words);
          p.h_scales[(size_t)r * (f / 16) + col / 16 + 1] = (uint8_t)quant_nv16(h + 16, p.act_scale_h, w2);
          words[2] = w2[0];
          words[3] = w2[1];
        }
        *reinterpret_cast<uint4*>(p.h_codes + (size_t)r * (f / 2) + col / 2) =
            make_uint4(words[0], words[1], words[2], words[3]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 512);
}

template <int FMT>
__global__ void __launch_bounds__(128, 1)
gemm_down_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tdn,
                 GemmArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kStages], done[kStages];
  __shared__ uint32_t tmem_base;
  if ((int)blockIdx.x >= *p.n_tiles) return;
  const Tile tile = p.tiles[blockIdx.x];
  const int n0 = blockIdx.y * kTileRows;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&done[s], 1); }
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = tmem_base;
  const CUtensorMap* tw[1] = {&tdn};
  int n_committed = 0;
  const bool ok = gemm_mainloop<1>(p, &ta, tw, tile, n0, smem, full, done, tb, 128, &n_committed);
  if (!ok) {
    if (threadIdx.x == 0) atomicExch(p.err, 1);
    drain(full, done);
  } else {
    const int m = threadIdx.x;
    const int r = tile.row_start + m;
    const bool live = r < tile.row_end;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const float* ts = reinterpret_cast<const float*>(p.slots + (size_t)tile.slot * p.ebytes +
                                                     p.w_scales_off[2]);
    const float sd = FMT == MOE_MXFP4 ? 1.0f : ts[2] * p.act_scale;
    for (int c = 0; c < 4; ++c) {
      uint32_t v[32];
      tc::tmem_ld32(tb + lane_base + 32 * c, v);
      tc::tmem_ld_wait();
      if (live) {
        float4* dst = reinterpret_cast<float4*>(p.O + (size_t)r * p.O_ld + n0 + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(v[4 * i]) * sd, __uint_as_float(v[4 * i + 1]) * sd,
                               __uint_as_float(v[4 * i + 2]) * sd, __uint_as_float(v[4 * i + 3]) * sd);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 256);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {kKTileBytes, kTileRows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                 uint64_t slot_stride) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {kKTileBytes, kTileRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t gemm_smem(int nb) {
  return 1024 + (size_t)kStages * (1 + nb) * kOpBytes + (size_t)kStages * (1 + nb) * kTileRows * 16;
}

}  // namespace

// ---------------------------------------------------------------- host side
struct PrefillPlan {
  CUtensorMap xq, hq, wg, wu, wd;
  bool ready;
};

bool prefill_shape_ok(const Geo& g) {
  return g.d % 256 == 0 && g.f % 256 == 0 && g.d >= 256 && g.f >= 256;
}

PrefillPlan* prefill_plan_create(const Geo& g, const uint8_t* slots, const uint8_t* xq_codes, size_t xq_rows,
                                 const uint8_t* hq_codes) {
  PrefillPlan* pl = new PrefillPlan();
  pl->ready = make_map_2d(&pl->xq, xq_codes, g.d / 2, xq_rows) &&
              make_map_2d(&pl->hq, hq_codes, g.f / 2, xq_rows) &&
              make_map_3d(&pl->wg, slots + g.off_codes[0], g.d / 2, g.f, g.S + 1 + g.X, g.ebytes) &&
              make_map_3d(&pl->wu, slots + g.off_codes[1], g.d / 2, g.f, g.S + 1 + g.X, g.ebytes) &&
              make_map_3d(&pl->wd, slots + g.off_codes[2], g.f / 2, g.d, g.S + 1 + g.X, g.ebytes);
  return pl;
}

void prefill_plan_destroy(PrefillPlan* pl) { delete pl; }
bool prefill_plan_ready(const PrefillPlan* pl) { return pl && pl->ready; }

cudaError_t launch_gather_quant(const Geo& g, const __nv_bfloat16* x, const int* tok_of, int N, float gx,
                                uint8_t* codes, uint8_t* scales, cudaStream_t st) {
  const size_t rows = (size_t)N * g.k + (g.has_shared ? N : 0);
  const size_t total = rows * (g.d / 32);
  if (total == 0) return cudaSuccess;
  gather_quant_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(x, tok_of, N, g.k, g.d, g.fmt, gx,
                                                                      g.has_shared, codes, scales);
  return cudaGetLastError();
}

int prefill_max_tiles(const Geo& g, int N) {
  const long long rows = (long long)N * g.k + (g.has_shared ? N : 0);
  return (int)((rows + kTileRows - 1) / kTileRows + g.E + 1);
}

cudaError_t launch_prefill_gemms(const Geo& g, const PrefillPlan* pl, const StepRecord* rec,
                                 const int* offsets, int N, int mode, int with_shared,
                                 void* tiles, int* n_tiles, const uint8_t* slots,
                                 const uint8_t* xq_scales, uint8_t* hq_codes, uint8_t* hq_scales,
                                 float* O, float gx, float gh, int* err, cudaStream_t st,
                                 const cudaEvent_t* ev) {
  Tile* tl = static_cast<Tile*>(tiles);
  build_tiles_kernel<<<1, 1024, 0, st>>>(rec, offsets, g.E, g.S, g.X, N, g.k, mode, with_shared, tl,
                                         n_tiles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int max_tiles = prefill_max_tiles(g, N);
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(gemm_gateup_kernel<MOE_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem(2));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_gateup_kernel<MOE_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem(2));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_down_kernel<MOE_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem(1));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_down_kernel<MOE_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem(1));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  GemmArgs p{};
  p.tiles = tl;
  p.n_tiles = n_tiles;
  p.slots = slots;
  p.ebytes = g.ebytes;
  p.fmt = g.fmt;
  p.err = err;
  // phase 1
  p.a_scales = xq_scales;
  p.w_scales_off[0] = g.off_scales[0];
  p.w_scales_off[1] = g.off_scales[1];
  p.w_scales_off[2] = g.off_tscale;
  p.K = g.d;
  p.rows_out = g.f;
  p.act_scale = g.fmt == MOE_MXFP4 ? 1.0f : gx;
  p.h_codes = hq_codes;
  p.h_scales = hq_scales;
  p.act_scale_h = gh;
  dim3 grid1(max_tiles, g.f / kTileRows);
  if (ev) cudaEventRecord(ev[0], st);
  if (g.fmt == MOE_MXFP4)
    gemm_gateup_kernel<MOE_MXFP4><<<grid1, 128, gemm_smem(2), st>>>(pl->xq, pl->wg, pl->wu, p);
  else
    gemm_gateup_kernel<MOE_NVFP4><<<grid1, 128, gemm_smem(2), st>>>(pl->xq, pl->wg, pl->wu, p);
  e = cudaGetLastError();
  if (ev) cudaEventRecord(ev[1], st);
  if (e != cudaSuccess) return e;
  // phase 2
  p.a_scales = hq_scales;
  p.w_scales_off[0] = g.off_scales[2];
  p.w_scales_off[2] = g.off_tscale;
  p.K = g.f;
  p.rows_out = g.d;
  p.act_scale = g.fmt == MOE_MXFP4 ? 1.0f : gh;
  p.O = O;
  p.O_ld = g.d;
  dim3 grid2(max_tiles, g.d / kTileRows);
  if (ev) cudaEventRecord(ev[2], st);
  if (g.fmt == MOE_MXFP4)
    gemm_down_kernel<MOE_MXFP4><<<grid2, 128, gemm_smem(1), st>>>(pl->hq, pl->wd, p);
  else
    gemm_down_kernel<MOE_NVFP4><<<grid2, 128, gemm_smem(1), st>>>(pl->hq, pl->wd, p);
  e = cudaGetLastError();
  if (ev) cudaEventRecord(ev[3], st);
  return e;
}

size_t prefill_tile_bytes(const Geo& g, int N) { return (size_t)prefill_max_tiles(g, N) * sizeof(Tile); }

}  // namespace moe
