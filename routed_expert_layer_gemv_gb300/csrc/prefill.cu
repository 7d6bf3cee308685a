// Prefill expert FFN: grouped GEMM on tcgen05 block-scaled MMAs.
//
// A prefill chunk gives each expert hundreds of tokens, so the expert FFN is a
// dense contraction (FreeToken's prefill streams whole layers of experts and
// is bound by compute once they are resident: "FreeToken：把 284B MoE 塞进游戏
// PC", zhichai.net, §二 "Prefill" paragraph).  Low-precision MMAs need
// low-precision activations, so x and h go through the block quantiser of the
// prefill activation format (the weights' own, or MXFP8 on MXFP4 weights:
// W4A8; actquant.cuh).  Steps:
//  1. gather_quant: row r of the permuted activations = quant(x[tok_of[r]]);
//     rows N*k .. N*k+N-1 hold every token for the shared expert; block
//     scales by padded 128-row block in the layout tcgen05.cp reads.
//  2. build_tiles: the launch's experts (hits, or all misses, + shared) cut
//     into M tiles of 128 rows; the last tile of an expert is ragged (its extra
//     rows are computed and dropped).  interleave_wscales: the launch's
//     weight scales into the tcgen05.cp layout.
//  3. phase 1 (gemm_ws_kernel<fmt, 1>): tiles of 128 rows x 128 d_ff columns;
//     B stacks the 128 gate rows over the same 128 up rows, so one N = 256 MMA
//     yields both halves of SwiGLU; epilogue h = SiLU(a) * u, re-quantised.
//  4. phase 2 (gemm_ws_kernel<fmt, 2>): tiles of 128 rows x 256 d_model
//     columns, O = h W_d^T, written as scaled f16.
// Both phases run the persistent warp-specialised kernel below (TMA warp, MMA
// warp, epilogue warps).  Every wait is bounded (~2 s); on a timeout the CTA
// records an error, skips its remaining waits, waits for its own copies and
// MMAs (bounded again), frees its TMEM and returns.
#include <algorithm>
#include <cstdio>

#include "actquant.cuh"
#include "common.cuh"
#include "tc.cuh"
#include "tiles_dev.cuh"

namespace moe {

namespace {

constexpr int kTileRows = kPrefillTileRows;   // M of one MMA tile, rows of one TMA box
using tl::Tile;
using tl::kSharedKey;

// Kernel variant of W4A8: MXFP4 weights under MXFP8 activations.  The MMA is
// kind::mxf8f6f4 with E4M3 A and E2M1 B; the FP4 weight tiles are loaded by
// TMA as 16 x U4 packed values per 16-byte shared-memory chunk (the unpacked
// layout that kind reads), so both operands have 128-byte rows of 128
// elements per stage and one E8M0 scale per 32 along K.
constexpr int kW4A8 = 100;
// The activation (A) operand's format of a kernel variant.
__host__ __device__ constexpr int act_op_fmt(int F) { return F == kW4A8 ? MOE_MXFP8 : F; }
constexpr int kKTileBytes = 128;        // 256 FP4 codes per K tile
constexpr int kOpBytes = kTileRows * kKTileBytes;   // 16 KB per 128-row operand box

// Block scales in the layout tcgen05.cp copies into TMEM (32x128b, one copy
// per lane quarter): per 128-row block and per group of 4 scale bytes along
// K, 512 bytes, byte 16 i + 4 j + b holding the scale of block row 32 j + i
// and K-block 4 g + b.  ng: groups per row.
__host__ __device__ inline size_t sf_off(size_t blk, int ng, int g, int row, int b) {
  return (blk * ng + g) * 512 + 16 * (row & 31) + 4 * (row >> 5) + b;
}
__host__ __device__ constexpr int sf_groups(int fmt, int K) { return fmt_block(fmt) ? K / fmt_block(fmt) / 4 : 0; }

// Exclusive scan of one int per thread over a block of up to 1024 threads;
// returns the thread's prefix, *total gets the sum.
__device__ int block_excl_scan(int v, int* sh33, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) sh33[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const int x = lane < nw ? sh33[lane] : 0;
    int xi = x;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += u;
    }
    if (lane < nw) sh33[lane] = xi - x;
    if (lane == 31) sh33[32] = xi;
  }
  __syncthreads();
  const int r = sh33[warp] + inc - v;
  *total = sh33[32];
  __syncthreads();
  return r;
}

// pbase[e]: the first padded 128-row block of expert e's rows (experts in
// ascending order, each taking ceil(count / 128) blocks); pbase[E]: the
// shared expert's first block; pbase[E + 1]: the total.
__global__ void __launch_bounds__(1024)
pad_base_kernel(const int* __restrict__ counts, int E, int N, int with_shared, int* __restrict__ pbase) {
  __shared__ int sh[33];
  const int e = threadIdx.x;
  const int nb = e < E ? (max(counts[e], 0) + kTileRows - 1) / kTileRows : 0;
  int total;
  const int pre = block_excl_scan(nb, sh, &total);
  if (e < E) pbase[e] = pre;
  if (e == 0) {
    pbase[E] = total;
    pbase[E + 1] = total + (with_shared ? (N + kTileRows - 1) / kTileRows : 0);
  }
}

// ---------------------------------------------------------------- step 1
// FP4 activations of every (token, expert) row: each token's 32-value groups
// are quantised once and the codes and scales written to the token's k
// permuted rows (row_of) and its shared-expert row N k + t.  Thread = (token,
// group).
// The scales go to the tcgen05.cp layout (sf_off) by padded block: row r of
// expert e is row (r - offsets[e]) % 128 of block pbase[e] + (r - offsets[e]) / 128.
__global__ void gather_quant_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ idx,
                                    const int* __restrict__ row_of, const int* __restrict__ offsets,
                                    const int* __restrict__ pbase, int N, int k, int E, int d, int fmt,
                                    float gx, int with_shared, uint8_t* __restrict__ codes,
                                    uint8_t* __restrict__ scales) {
  const int nb = d / 32;                       // 32-value groups per row
  const size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= (size_t)N * nb) return;
  const int t = (int)(v / nb), c = (int)(v % nb);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + (size_t)c * 32);
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
  const int nr = k + (with_shared ? 1 : 0);
  const int ng = sf_groups(fmt, d);
  // (padded block, row in the block) of the j-th row of token t
  auto place = [&](int j, size_t* blk, int* rib) {
    int local, b0;
    if (j < k) {
      const int e = idx[(size_t)t * k + j];
      local = row_of[(size_t)t * k + j] - offsets[e];
      b0 = pbase[e];
    } else {
      local = t;
      b0 = pbase[E];
    }
    *blk = (size_t)b0 + local / kTileRows;
    *rib = local % kTileRows;
  };
  if (fmt == MOE_MXFP8 || fmt == MOE_BF16) {
    // W8A8: the group as 32 E4M3 bytes + an E8M0 byte; W16A16: x as it is
    uint4 cw[4];
    uint32_t s8 = 0;
    if (fmt == MOE_MXFP8) {
      uint32_t w8[8];
      s8 = quant_mx8_32(vals, w8);
      cw[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
      cw[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) cw[q] = src[q];
    }
    const int nv = fmt == MOE_MXFP8 ? 2 : 4;            // 16-byte pieces of the group
    const size_t rowb = (size_t)d * (fmt == MOE_MXFP8 ? 1 : 2);
    for (int j = 0; j < nr; ++j) {
      const size_t r = j < k ? (size_t)row_of[(size_t)t * k + j] : (size_t)N * k + t;
      uint4* dst = reinterpret_cast<uint4*>(codes + r * rowb + (size_t)c * 16 * nv);
      for (int q = 0; q < nv; ++q) dst[q] = cw[q];
      if (fmt == MOE_MXFP8) {
        size_t blk;
        int rib;
        place(j, &blk, &rib);
        scales[sf_off(blk, ng, c >> 2, rib, c & 3)] = (uint8_t)s8;
      }
    }
    return;
  }
  uint32_t words[4];
  uint32_t s0, s1 = 0;
  if (fmt == MOE_MXFP4) {
    s0 = quant_mx32(vals, words);
  } else {
    uint32_t w2[2];
    s0 = quant_nv16(vals, gx, words);
    s1 = quant_nv16(vals + 16, gx, w2);
    words[2] = w2[0];
    words[3] = w2[1];
  }
  const uint4 cw = make_uint4(words[0], words[1], words[2], words[3]);
  for (int j = 0; j < nr; ++j) {
    const size_t r = j < k ? (size_t)row_of[(size_t)t * k + j] : (size_t)N * k + t;
    *reinterpret_cast<uint4*>(codes + r * (d / 2) + (size_t)c * 16) = cw;
    size_t blk;
    int rib;
    place(j, &blk, &rib);
    if (fmt == MOE_MXFP4) {
      scales[sf_off(blk, ng, c >> 2, rib, c & 3)] = (uint8_t)s0;
    } else {   // K-blocks 2c and 2c + 1 of 16 values
      scales[sf_off(blk, ng, c >> 1, rib, (2 * c) & 3)] = (uint8_t)s0;
      scales[sf_off(blk, ng, c >> 1, rib, (2 * c + 1) & 3)] = (uint8_t)s1;
    }
  }
}

// ---------------------------------------------------------------- step 2
__global__ void __launch_bounds__(1024)
build_tiles_kernel(const StepRecord* __restrict__ rec, const int* __restrict__ offsets,
                   const int* __restrict__ pbase, int E, int S, int X, int shb, int key0, int N, int k, int mode,
                   int with_shared, Tile* __restrict__ tiles, int* __restrict__ ents, int* __restrict__ n_tiles) {
  __shared__ int sh[33];
  __shared__ int carry;
  tl::build_tiles(rec, offsets, pbase, E, S, X, shb, key0, N, k, mode, with_shared, tiles, ents, n_tiles, sh,
                  &carry);
}

// Weight block scales of the launch's experts in the tcgen05.cp layout, by
// pool buffer (the scales of buffer b at wsf + b ent_bytes): phase 1 first
// (per block q of 128 gate rows and the same 128 up rows, per group g: the
// gate block's 512 bytes, then the up block's, K = d), then phase 2 (per
// block of 256 down rows, per group: its two 128-row halves' 512 bytes,
// K = f).  A block is 128 rows of one matrix (phase 1's (q, gate / up)
// blocks, then the down matrix's), staged through shared memory (rows padded
// to an odd word count) so that both the row reads and the 16-byte writes are
// coalesced; a CTA takes kIlvBlocks consecutive blocks of one buffer
// (blockIdx.y: the launch entry).
constexpr int kIlvBlocks = 4;

__global__ void __launch_bounds__(256)
interleave_wscales_kernel(const uint8_t* __restrict__ slots, size_t ebytes, size_t off_g, size_t off_u,
                          size_t off_d, const int* __restrict__ ents, const int* __restrict__ n_tiles, int E, int d,
                          int f, int blk, uint8_t* __restrict__ wsf, int* __restrict__ wtag, int nb) {
  extern __shared__ uint32_t smw[];
  const int ent = blockIdx.y;
  if (ent >= n_tiles[1]) return;
  const int slot = ents[ent];
  if (slot < 0) return;
  // wtag[b]: key of the weights whose scales wsf holds for buffer b (-1:
  // none); wtag[nb + b]: CTAs of buffer b done in this launch.  A buffer that
  // holds the same weights as when its scales were last laid out is skipped;
  // the tag changes only once every CTA of the buffer has written its blocks,
  // so all CTAs of one buffer take the same decision.
  const int key = ents[(E + 1) + ent], fresh = ents[2 * (E + 1) + ent];
  if (!fresh && key != -1 && wtag[slot] == key) return;
  const uint8_t* w = slots + (size_t)slot * ebytes;
  const int nb1 = 2 * (f / kTileRows), nblk = nb1 + d / kTileRows;
  for (int b = blockIdx.x * kIlvBlocks; b < min(nblk, (int)(blockIdx.x + 1) * kIlvBlocks); ++b) {
    uint8_t* out = wsf + (size_t)slot * (3 * (size_t)d * f / blk);
    int K, hi, hh;
    const uint8_t* src;
    if (b < nb1) {
      hi = b >> 1;
      hh = b & 1;
      K = d;
      src = w + (hh ? off_u : off_g) + (size_t)kTileRows * hi * (K / blk);
    } else {
      const int rb = b - nb1;   // 128-row block of the down matrix
      hi = rb >> 1;
      hh = rb & 1;
      K = f;
      src = w + off_d + (size_t)kTileRows * rb * (K / blk);
      out += 2 * (size_t)d * f / blk;
    }
    const int ng = K / blk / 4, ngp = ng | 1;   // words per row, padded to odd
    const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
    __syncthreads();   // the previous block's reads of smw are done
    for (int v = threadIdx.x; v < kTileRows * ng; v += blockDim.x) smw[(v / ng) * ngp + v % ng] = s4[v];
    __syncthreads();
    for (int v = threadIdx.x; v < ng * 32; v += blockDim.x) {
      const int i = v & 31, g = v >> 5;
      *reinterpret_cast<uint4*>(out + (((size_t)hi * ng + g) * 2 + hh) * 512 + 16 * i) =
          make_uint4(smw[i * ngp + g], smw[(32 + i) * ngp + g], smw[(64 + i) * ngp + g], smw[(96 + i) * ngp + g]);
    }
  }
  // the buffer's last CTA records the key (and resets the count)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&wtag[nb + slot], 1) == (int)gridDim.x - 1) {
      wtag[nb + slot] = 0;
      wtag[slot] = key;
    }
  }
}

// Block scales of h back to rows [rows][f / blk] (test hook): row r of
// expert e (offsets) sits in block pbase[e] + (r - offsets[e]) / 128.
__global__ void untile_scales_kernel(const uint8_t* __restrict__ tiled, const int* __restrict__ offsets,
                                     const int* __restrict__ pbase, int E, int Nk, int rows, int K, int blk,
                                     uint8_t* __restrict__ out) {
  const int nq = K / blk, ng = nq / 4;
  const size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= (size_t)rows * nq) return;
  const int r = (int)(v / nq), q = (int)(v % nq);
  int b0, local;
  if (r < Nk) {
    int lo = 0, hi = E - 1;   // the expert whose rows hold r: largest e with offsets[e] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
    }
    b0 = pbase[lo];
    local = r - offsets[lo];
  } else {
    b0 = pbase[E];
    local = r - Nk;
  }
  out[v] = tiled[sf_off((size_t)b0 + local / kTileRows, ng, q >> 2, local % kTileRows, q & 3)];
}

// ---------------------------------------------------------------- GEMM pieces
struct GemmArgs {
  const Tile* tiles;
  const int* n_tiles;
  const uint8_t* a_scales;     // block scales of the A operand (activations), tcgen05.cp layout by padded block
  const uint8_t* w_scales;     // the launch's weight scales, tcgen05.cp layout (this phase's part of entry 0)
  size_t ent_bytes;            // bytes of one entry's weight scales (both phases)
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
  float* O;                    // phase 2: f16 rows [rows][O_ld] (the buffer's first half)
  int8_t* O_exp;               // phase 2: power-of-two exponent per row and 128-column block
  int O_ld;
};

// ---------------------------------------------------------------- persistent warp-specialised GEMM
// One CTA per SM walks the launch's (M tile, N tile) pairs.  Warps with one
// job each, meeting only at mbarriers:
//   warp 0     TMA: A (128 token rows x one 128-byte K stage) and B (phase 1:
//              128 gate rows over the same 128 up rows; phase 2: 128 down
//              rows) per stage, and with them the stage's block scales of A
//              and B (512-byte groups already in the layout tcgen05.cp reads:
//              activations quantised into it, weight scales interleaved per
//              launch), all on one barrier;
//   warp 1     one thread copies the stage's scales into its TMEM ring slot
//              (tcgen05.cp, every lane quarter gets all 128 rows) and issues
//              four block-scaled MMAs per stage (M = 128, N = 256 in phase 1
//              into its one accumulator, N = 128 in phase 2 into one of two);
//              copies and MMAs run in issue order, so no other warp touches
//              the scales;
//   warps 2-9  epilogue (phase 2: warps 2-5), by lane quarter (32 rows; in
//              phase 1 two warps per quarter, one per half of the columns):
//              drain the accumulator into registers, release it, then SiLU *
//              mul + quantisation of h (phase 1) or the scaled f16 O rows
//              (phase 2), while the MMAs of the next tile proceed.
constexpr int kEpiWarp0 = 2;
constexpr int kSfBase = 256;            // TMEM columns 0..255: the accumulator(s); then the scale ring

// Phase 2 keeps room to stage O for its epilogue: per epilogue warp 32 rows
// x 32 f16 columns at a time, rows padded by 8 so the row writes and reads
// spread over the banks.
// Both phases multiply each A tile by 256 weight rows in one N = 256 MMA
// (phase 1: 128 gate over the same 128 up rows; phase 2: 256 down rows),
// twice the MMA work per staged byte of a 128-row B tile; the single
// accumulator takes 256 TMEM columns (two would leave none for the scales;
// the epilogue hides behind the operand ring either way, measured), drained
// by eight epilogue warps.  Ring stages: 4 of 48 KB of operands, 3 for
// NVFP4's phase 2 (its larger scales and the O staging fill the rest).
template <int FMT, int PH> constexpr int ws_stages() { return PH == 2 && FMT == MOE_NVFP4 ? 3 : 4; }
template <int PH> constexpr int ws_nb() { return 256; }        // B rows = MMA N
template <int PH> constexpr int ws_epi_warps() { return 8; }
template <int PH> constexpr int ws_threads() { return 32 * (2 + ws_epi_warps<PH>()); }
constexpr int kOStrideB = 40;   // f16 elements per staged O row piece (32 columns + 8 of padding)
constexpr size_t kOStage = 8 * 32 * kOStrideB * 2;

// Scale groups of 4 bytes per row per stage: MXFP4 2 (8 blocks of 32 over
// 256 K), NVFP4 4 (16 blocks of 16), MXFP8 / W4A8 1 (4 blocks of 32 over 128
// K), bf16 0.
__host__ __device__ constexpr int stage_groups(int FMT) {
  return FMT == MOE_MXFP4 ? 2 : FMT == MOE_NVFP4 ? 4 : (FMT == MOE_MXFP8 || FMT == kW4A8) ? 1 : 0;
}
// Shared memory: the operand ring (1024-byte aligned stages), then each
// stage's scales (A groups, then B groups), then (phase 2) the O staging.
template <int FMT, int PH>
size_t ws_smem() {
  constexpr int BA = ws_nb<PH>() / 128;   // 128-row blocks of B
  return 1024 + (size_t)ws_stages<FMT, PH>() * ((1 + BA) * kOpBytes + (1 + BA) * 512 * stage_groups(FMT)) +
         (PH == 2 ? kOStage : 0);
}

__device__ __forceinline__ bool ws_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (*abort_flag) return false;
  if (tc::mbar_wait(bar, parity)) return true;
  *abort_flag = 1;
  atomicExch(err, 1);
  return false;
}

__device__ __forceinline__ void ws_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::su32(bar)) : "memory");
}

template <int FMT, int PH>
__global__ void __launch_bounds__(ws_threads<PH>(), 1)
gemm_ws_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb0,
               const __grid_constant__ CUtensorMap tb1, GemmArgs p) {
  // K elements per 128-byte stage row and 4-byte scale groups per row per stage:
  // MXFP4 256 / 2, NVFP4 256 / 4, MXFP8 128 / 1, bf16 64 / 0 (no scales)
  constexpr int AF = act_op_fmt(FMT);
  constexpr int KST = 1024 / fmt_code_bits(AF);
  constexpr int G = stage_groups(FMT);
  constexpr int NB = ws_nb<PH>(), BA = NB / 128;  // B rows (MMA N), their 128-row blocks
  constexpr int EW = ws_epi_warps<PH>();
  constexpr int NACC = 1;                         // accumulators (NB TMEM columns each)
  constexpr uint32_t kStageOp = (1 + BA) * kOpBytes;            // A, then B, of a stage
  constexpr uint32_t kSfStage = (1 + BA) * 512 * G;             // its scales: A groups, then B (group, block)
  constexpr int SFC = 4 * (1 + BA) * (G > 0 ? G : 1);           // TMEM columns of one scale slot
  constexpr int NCOL = PH == 1 ? 128 : 256;       // output columns of one tile (phase 1: h columns)
  constexpr int kWsStages = ws_stages<FMT, PH>();
  static_assert(kSfBase + kWsStages * SFC <= 512, "TMEM columns");
  // bytes the B loads of a stage count on its barrier: the 16 x U4 loads of
  // W4A8 count the packed bytes they read (8 KB of codes for each 16 KB they
  // fill with their padding)
  constexpr uint32_t kBTxBytes = BA * (FMT == kW4A8 ? kOpBytes / 2 : kOpBytes);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kWsStages], empty[kWsStages], accf[2], acce[2], fin;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kWsStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], EW);
    }
    tc::mbar_init(&fin, 1);
    s_abort = 0;
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = tmem_base;
  const int n_m = *p.n_tiles;
  const int NT = p.rows_out / NCOL;
  const long long T = (long long)n_m * NT;
  const int nkt = p.K / KST;
  const int ng = G > 0 ? nkt * G : 0;          // scale groups per row (A and B alike)
  uint8_t* sf_smem = smem + (size_t)kWsStages * kStageOp;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (long long t = blockIdx.x; t < T && !stop; t += gridDim.x) {
        const Tile tile = p.tiles[t / NT];
        const int n0 = (int)(t % NT) * NCOL;
        for (int kt = 0; kt < nkt; ++kt, ++it) {
          const int s = it % kWsStages;
          const uint32_t k = it / kWsStages;
          if (k > 0 && !ws_wait(&empty[s], (k - 1) & 1, &s_abort, p.err)) { stop = true; break; }
          uint8_t* st = smem + (size_t)s * kStageOp;
          tc::mbar_expect_tx(&full[s], kOpBytes + kBTxBytes + kSfStage);
          if (G > 0) {
            uint8_t* ss = sf_smem + (size_t)s * kSfStage;
            tc::bulk_load(ss, p.a_scales + ((size_t)tile.pb * ng + (size_t)kt * G) * 512, 512 * G, &full[s]);
            tc::bulk_load(ss + 512 * G,
                          p.w_scales + (size_t)tile.slot * p.ent_bytes +
                              ((size_t)(n0 / NCOL) * ng + (size_t)kt * G) * 512 * BA,
                          512 * G * BA, &full[s]);
          }
          tc::tma_load_2d(st, &ta, &full[s], kt * kKTileBytes, tile.row_start);
          if (PH == 1) {   // 128 gate rows over the same 128 up rows
            tc::tma_load_3d(st + kOpBytes, &tb0, &full[s], kt * kKTileBytes, n0, tile.slot);
            tc::tma_load_3d(st + 2 * kOpBytes, &tb1, &full[s], kt * kKTileBytes, n0, tile.slot);
          } else {         // 256 down rows as two 128-row boxes
            tc::tma_load_3d(st + kOpBytes, &tb0, &full[s], kt * kKTileBytes, n0, tile.slot);
            tc::tma_load_3d(st + 2 * kOpBytes, &tb0, &full[s], kt * kKTileBytes, n0 + 128, tile.slot);
          }
        }
      }
      // copies in flight land before the CTA exits (bounded)
      const uint32_t first = it > (uint32_t)kWsStages ? it - kWsStages : 0;
      for (uint32_t i = first; i < it; ++i)
        if (!tc::mbar_wait(&full[i % kWsStages], (i / kWsStages) & 1)) { atomicExch(p.err, 1); break; }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, nt_done = 0;
      bool stop = false;
      for (long long t = blockIdx.x; t < T && !stop; t += gridDim.x, ++nt_done) {
        const int b = NACC == 2 ? (int)(nt_done & 1) : 0;
        const uint32_t u = NACC == 2 ? nt_done >> 1 : nt_done;
        if (u > 0 && !ws_wait(&acce[b], (u - 1) & 1, &s_abort, p.err)) { stop = true; break; }
        tc::fence_after();
        for (int kt = 0; kt < nkt; ++kt, ++it) {
          const int s = it % kWsStages;
          const uint32_t ph = (it / kWsStages) & 1;
          if (!ws_wait(&full[s], ph, &s_abort, p.err)) {
            stop = true;
            break;
          }
          tc::fence_after();
          const uint32_t a_s = tc::su32(smem + (size_t)s * kStageOp), b_s = a_s + kOpBytes;
          // scale slot: A groups (4 columns each), then B groups of BA
          // 128-row blocks (4 columns per block, the blocks of a group side by side)
          const uint32_t sfa = tb + kSfBase + (uint32_t)(s * SFC), sfb = sfa + 4 * G;
          if (G > 0) {
            const uint32_t ss = tc::su32(sf_smem + (size_t)s * kSfStage);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              tc::cp_sf(sfa + 4 * g, tc::sdesc_rows16(ss + 512 * g));
#pragma unroll
              for (int h = 0; h < BA; ++h)
                tc::cp_sf(sfb + 4 * (BA * g + h), tc::sdesc_rows16(ss + 512 * (G + BA * g + h)));
            }
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = tc::sdesc_sw128(a_s + 32 * kk), bd = tc::sdesc_sw128(b_s + 32 * kk);
            const bool acc = kt > 0 || kk > 0;
            const uint32_t dacc = tb + NB * b;
            if (FMT == MOE_MXFP4) {
              const uint32_t id = 2 * (kk & 1), g = kk >> 1;
              tc::mma_mxf4(dacc, ad, bd, tc::idesc_fp4(NB, true, id, id), sfa + 4 * g, sfb + 4 * BA * g, acc);
            } else if (FMT == MOE_NVFP4) {
              tc::mma_nvf4(dacc, ad, bd, tc::idesc_fp4(NB, false, 0, 0), sfa + 4 * kk, sfb + 4 * BA * kk, acc);
            } else if (AF == MOE_MXFP8) {
              // one E8M0 scale per 32-K MMA: byte kk of the stage's group;
              // B E4M3 (W8A8) or E2M1 (W4A8)
              tc::mma_mxf8(dacc, ad, bd, tc::idesc_mxf8(NB, kk, kk, FMT == kW4A8), sfa, sfb, acc);
            } else {
              tc::mma_bf16(dacc, ad, bd, tc::idesc_bf16(NB), acc);
            }
          }
          tc::mma_commit(&empty[s]);   // the stage's smem and scale slot are free once these MMAs finish
        }
        if (stop) break;
        tc::mma_commit(&accf[b]);
      }
      // every MMA issued (also of a tile cut short) has finished before the CTA
      // frees TMEM (bounded)
      tc::mma_commit(&fin);
      if (!tc::mbar_wait(&fin, 0)) atomicExch(p.err, 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp 2 + e: lane quarter warp & 3 (the TMEM lanes a warp may read);
    // two warps per quarter split the tile's columns in halves (hh)
    const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
    const int rl = 32 * (warp & 3) + lane;   // tile row of this thread
    const int hh = (warp - kEpiWarp0) >> 2;
    uint32_t nt_done = 0;
    for (long long t = blockIdx.x; t < T; t += gridDim.x, ++nt_done) {
      const Tile tile = p.tiles[t / NT];
      const int n0 = (int)(t % NT) * NCOL;
      const int b = NACC == 2 ? (int)(nt_done & 1) : 0;
      if (!ws_wait(&accf[b], (NACC == 2 ? nt_done >> 1 : nt_done) & 1, &s_abort, p.err)) continue;
      tc::fence_after();
      const int r = tile.row_start + rl;
      const bool live = r < tile.row_end;
      const float* ts = reinterpret_cast<const float*>(p.slots + (size_t)tile.slot * p.ebytes + p.w_scales_off[2]);
      uint32_t v0[32], v1[32], v2[32], v3[32];
      const uint32_t acc = tb + lq + NB * b;
      // phase 1: gate columns 64 hh .. + 63 (v0, v1) and the same up columns
      // (128 + 64 hh .., v2, v3); phase 2: O columns 128 hh .. + 127 (v0 .. v3)
      const uint32_t c0 = PH == 1 ? 64 * hh : 128 * hh, c2 = PH == 1 ? 128 + 64 * hh : 128 * hh + 64;
      tc::tmem_ld32(acc + c0, v0);
      tc::tmem_ld32(acc + c0 + 32, v1);
      tc::tmem_ld32(acc + c2, v2);
      tc::tmem_ld32(acc + c2 + 32, v3);
      tc::tmem_ld_wait();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ws_arrive(&acce[b]);   // the accumulator is free for a later tile
      // Rows past the expert's last (the tail of its last tile) carry another
      // expert's codes under stale scale bytes, which may decode to NaN: they
      // are never stored, so phase 1 skips their SiLU and quantisation (whose
      // special-value paths would cost more than the live rows)
      if (PH == 1 && live) {
        // h columns n0 + 64 hh .. + 63 of this thread's row
        const float sg = FMT == MOE_NVFP4 ? ts[0] * p.act_scale : 1.0f;
        const float su = FMT == MOE_NVFP4 ? ts[1] * p.act_scale : 1.0f;
        const int f = p.rows_out;
        const int ngh = sf_groups(AF, f);   // scale groups per row of h
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t* gv = c == 0 ? v0 : v1;
          const uint32_t* uv = c == 0 ? v2 : v3;
          float hv[32];
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) {
            const float a = __uint_as_float(gv[i2]) * sg, u = __uint_as_float(uv[i2]) * su;
            hv[i2] = a / (1.0f + __expf(-a)) * u;
          }
          if (live && (AF == MOE_MXFP8 || AF == MOE_BF16)) {
            const int col = n0 + 64 * hh + 32 * c;
            if (AF == MOE_MXFP8) {
              uint32_t w8[8];
              const int q = col / 32;
              p.h_scales[sf_off(tile.pb, ngh, q >> 2, rl, q & 3)] = (uint8_t)quant_mx8_32(hv, w8);
              uint4* dst = reinterpret_cast<uint4*>(p.h_codes + (size_t)r * f + col);
              dst[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
              dst[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
            } else {
              uint32_t wb[16];
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[2 * i2], hv[2 * i2 + 1]);
                wb[i2] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              uint4* dst = reinterpret_cast<uint4*>(p.h_codes + ((size_t)r * f + col) * 2);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = make_uint4(wb[4 * q], wb[4 * q + 1], wb[4 * q + 2], wb[4 * q + 3]);
            }
          } else if (live) {
            const int col = n0 + 64 * hh + 32 * c;
            uint32_t words[4];
            if (FMT == MOE_MXFP4) {
              const int q = col / 32;
              p.h_scales[sf_off(tile.pb, ngh, q >> 2, rl, q & 3)] = (uint8_t)quant_mx32(hv, words);
            } else {
              uint32_t w2[2];
              const int q = col / 16;   // K-blocks q and q + 1 (q even)
              p.h_scales[sf_off(tile.pb, ngh, q >> 2, rl, q & 3)] = (uint8_t)quant_nv16(hv, p.act_scale_h, words);
              p.h_scales[sf_off(tile.pb, ngh, q >> 2, rl, (q & 3) + 1)] = (uint8_t)quant_nv16(hv + 16, p.act_scale_h, w2);
              words[2] = w2[0];
              words[3] = w2[1];
            }
            *reinterpret_cast<uint4*>(p.h_codes + (size_t)r * (f / 2) + col / 2) =
                make_uint4(words[0], words[1], words[2], words[3]);
          }
        }
      } else if (PH == 2) {
        // lane = row in TMEM; O is written as f16 scaled by 2^-s, s per row
        // and 128-column block (max |O| * 2^-s in [2^14, 2^15), so nothing
        // overflows and the rounding is relative to the block's largest
        // value); the combine multiplies by 2^s and accumulates in fp32.
        // This warp's block is columns nb0 .. nb0 + 127.  Rows go through
        // shared memory 32 columns at a time, so that each store instruction
        // writes eight whole 64-byte row pieces
        const int nb0 = n0 + 128 * hh;
        const float sd = FMT == MOE_NVFP4 ? ts[2] * p.act_scale : 1.0f;
        __half* Oh = reinterpret_cast<__half*>(p.O);
        float mx = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2)
          mx = fmaxf(fmaxf(fmaxf(mx, fabsf(__uint_as_float(v0[i2]))), fabsf(__uint_as_float(v1[i2]))),
                     fmaxf(fabsf(__uint_as_float(v2[i2])), fabsf(__uint_as_float(v3[i2]))));
        mx *= fabsf(sd);
        int se = 0;
        if (mx > 0.f && mx < 3.0e38f) {
          int ex;
          frexpf(mx, &ex);
          se = max(-100, min(100, ex - 15));
        }
        const float sc = sd * __int_as_float((127 - se) << 23);   // sd * 2^-se
        if (live) p.O_exp[(size_t)r * (p.O_ld / 128) + nb0 / 128] = (int8_t)se;
        __half* ost = reinterpret_cast<__half*>(sf_smem + (size_t)kWsStages * kSfStage) +
                      (size_t)(warp - kEpiWarp0) * 32 * kOStrideB;
        uint4* myrow = reinterpret_cast<uint4*>(ost + lane * kOStrideB);
        const int row0 = tile.row_start + 32 * (warp & 3);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t* vv = q4 == 0 ? v0 : q4 == 1 ? v1 : q4 == 2 ? v2 : v3;
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __half2 h2 = __floats2half2_rn(__uint_as_float(vv[8 * i2 + 2 * j]) * sc,
                                                   __uint_as_float(vv[8 * i2 + 2 * j + 1]) * sc);
              w[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            myrow[i2] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          __syncwarp();
          // eight rows per instruction: lanes 4j .. 4j + 3 take row rr + j
          for (int rr = 0; rr < 32; rr += 8) {
            const int rw = rr + (lane >> 2), rg = row0 + rw;
            if (rg < tile.row_end)
              reinterpret_cast<uint4*>(Oh + (size_t)rg * p.O_ld + nb0 + 32 * q4)[lane & 3] =
                  reinterpret_cast<const uint4*>(ost + rw * kOStrideB)[lane & 3];
          }
          __syncwarp();
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 512);
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

// Packed FP4 rows [slots][rows][K] (K / 2 bytes per row) loaded unpacked for
// kind::mxf8f6f4: boxes of 128 codes x box_rows rows, each 16 codes landing
// in a 16-byte chunk (128 shared-memory bytes per box row), 128B swizzle.
// The encoder checks what this type needs: a 32-byte aligned base, K a
// multiple of 128, strides multiples of 32 bytes.
bool make_map_3d_u4(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t slots,
                    uint64_t slot_stride, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {K, rows, slots};
  cuuint64_t strides[2] = {K / 2, slot_stride};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                 uint64_t slot_stride, uint32_t box_rows = kTileRows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {kKTileBytes, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace

// ---------------------------------------------------------------- host side
struct PrefillPlan {
  CUtensorMap xq, hq, wd;
  CUtensorMap wg, wu;       // gate / up in 128-row boxes (stacked into one 256-row B tile)
  bool ready;
};

bool prefill_shape_ok(const Geo& g) {
  return g.d % 256 == 0 && g.f % 256 == 0 && g.d >= 256 && g.f >= 256;
}

PrefillPlan* prefill_plan_create(const Geo& g, const uint8_t* slots, const uint8_t* xq_codes, size_t xq_rows,
                                 const uint8_t* hq_codes) {
  PrefillPlan* pl = new PrefillPlan();
  // activation rows in the prefill activation format, weight rows in the
  // weights' own (W4A8: FP4 weights loaded unpacked)
  const uint64_t da = (uint64_t)g.d * fmt_code_bits(g.afmt) / 8, fa = (uint64_t)g.f * fmt_code_bits(g.afmt) / 8;
  pl->ready = make_map_2d(&pl->xq, xq_codes, da, xq_rows) && make_map_2d(&pl->hq, hq_codes, fa, xq_rows);
  if (g.afmt != g.fmt) {
    pl->ready = pl->ready && g.fmt == MOE_MXFP4 && g.afmt == MOE_MXFP8 &&
                make_map_3d_u4(&pl->wd, slots + g.off_codes[2], g.f, g.d, g.nbuf, g.ebytes, kTileRows) &&
                make_map_3d_u4(&pl->wg, slots + g.off_codes[0], g.d, g.f, g.nbuf, g.ebytes, kTileRows) &&
                make_map_3d_u4(&pl->wu, slots + g.off_codes[1], g.d, g.f, g.nbuf, g.ebytes, kTileRows);
    return pl;
  }
  const uint64_t db = (uint64_t)g.d * fmt_code_bits(g.fmt) / 8, fb = (uint64_t)g.f * fmt_code_bits(g.fmt) / 8;
  pl->ready = pl->ready &&
              make_map_3d(&pl->wd, slots + g.off_codes[2], fb, g.d, g.nbuf, g.ebytes) &&
              make_map_3d(&pl->wg, slots + g.off_codes[0], db, g.f, g.nbuf, g.ebytes) &&
              make_map_3d(&pl->wu, slots + g.off_codes[1], db, g.f, g.nbuf, g.ebytes);
  return pl;
}

void prefill_plan_destroy(PrefillPlan* pl) { delete pl; }
bool prefill_plan_ready(const PrefillPlan* pl) { return pl && pl->ready; }

cudaError_t launch_gather_quant(const Geo& g, const __nv_bfloat16* x, const int* idx, const int* row_of,
                                const int* counts, const int* offsets, int N, float gx, int* pbase,
                                bool pbase_ready, uint8_t* codes, uint8_t* scales, cudaStream_t st) {
  const size_t total = (size_t)N * (g.d / 32);
  if (total == 0) return cudaSuccess;
  if (!pbase_ready) {
    pad_base_kernel<<<1, 1024, 0, st>>>(counts, g.E, N, g.has_shared, pbase);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  gather_quant_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(x, idx, row_of, offsets, pbase, N, g.k,
                                                                      g.E, g.d, g.afmt, gx, g.has_shared,
                                                                      codes, scales);
  return cudaGetLastError();
}

int prefill_max_tiles(const Geo& g, int N) {
  const long long rows = (long long)N * g.k + (g.has_shared ? N : 0);
  return (int)((rows + kTileRows - 1) / kTileRows + g.E + 1);
}

// Pool buffers that can hold an expert's weights: the pool's own count, at
// least E + 1 (a resized lone layer stays within E + 1).
static int wscale_entries(const Geo& g) { return std::max(g.nbuf, g.E + 1); }

// Block scales of the activations (x or h, K = d or f) by padded 128-row block.
size_t prefill_act_scale_bytes(const Geo& g, int N, int K) {
  return std::max<size_t>(16, (size_t)prefill_max_tiles(g, N) * kTileRows * fmt_scale_row(g.afmt, K));
}
// The interleaved weight scales, one entry per pool buffer.
size_t prefill_wscale_bytes(const Geo& g) {
  return std::max<size_t>(16, (size_t)wscale_entries(g) * 3 * fmt_scale_row(g.afmt, g.d) * (size_t)g.f);
}
// Their tags and per-launch counts (ints; all tags -1 = nothing laid out).
size_t prefill_wtag_ints(const Geo& g) { return 2 * (size_t)wscale_entries(g); }

cudaError_t launch_untile_hscales(const Geo& g, const uint8_t* tiled, const int* offsets, const int* pbase, int N,
                                  uint8_t* out, cudaStream_t st) {
  const int blk = fmt_block(g.afmt);
  const int rows = N * g.k + (g.has_shared ? N : 0);
  const size_t total = (size_t)rows * (blk ? g.f / blk : 0);
  if (total == 0) return cudaSuccess;
  untile_scales_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(tiled, offsets, pbase, g.E, N * g.k, rows,
                                                                       g.f, blk, out);
  return cudaGetLastError();
}

cudaError_t launch_prefill_gemms(const Geo& g, const PrefillPlan* pl, const StepRecord* rec,
                                 const int* offsets, const int* pbase, int N, int mode, int with_shared,
                                 void* tiles, int* n_tiles, const uint8_t* slots,
                                 const uint8_t* xq_scales, uint8_t* hq_codes, uint8_t* hq_scales, uint8_t* wsf,
                                 int* wtag, float* O, float gx, float gh, int* err, int num_sms, cudaStream_t st,
                                 const cudaEvent_t* ev, bool tiles_ready) {
  const int max_tiles = prefill_max_tiles(g, N);
  Tile* tl = static_cast<Tile*>(tiles);
  int* ents = reinterpret_cast<int*>(tl + max_tiles);
  cudaError_t e = cudaSuccess;
  if (!tiles_ready) {   // (else built by the routing CTA: launch_scan_lru)
    build_tiles_kernel<<<1, 1024, 0, st>>>(rec, offsets, pbase, g.E, g.S, g.X, g.shb, g.key0, N, g.k, mode,
                                           with_shared, tl, ents, n_tiles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int blk = fmt_block(g.afmt);   // scale block of both operands (W4A8: 32 on either side)
  const size_t ent_bytes = blk ? 3 * (size_t)g.d * g.f / blk : 0;
  if (blk) {
    const int ngp_max = std::max(g.d, g.f) / blk / 4 | 1;
    const int ismem = kTileRows * ngp_max * 4;
    e = ensure_smem_limit((const void*)interleave_wscales_kernel, ismem);
    if (e != cudaSuccess) return e;
    const int nblk = 2 * (g.f / kTileRows) + g.d / kTileRows;
    const dim3 grid((unsigned)((nblk + kIlvBlocks - 1) / kIlvBlocks), (unsigned)(g.E + 1));
    interleave_wscales_kernel<<<grid, 256, ismem, st>>>(slots, g.ebytes, g.off_scales[0], g.off_scales[1],
                                                        g.off_scales[2], ents, n_tiles, g.E, g.d, g.f, blk, wsf,
                                                        wtag, wscale_entries(g));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_MXFP4, 1>, (int)ws_smem<MOE_MXFP4, 1>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_NVFP4, 1>, (int)ws_smem<MOE_NVFP4, 1>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_MXFP8, 1>, (int)ws_smem<MOE_MXFP8, 1>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_BF16, 1>, (int)ws_smem<MOE_BF16, 1>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<kW4A8, 1>, (int)ws_smem<kW4A8, 1>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<kW4A8, 2>, (int)ws_smem<kW4A8, 2>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_MXFP4, 2>, (int)ws_smem<MOE_MXFP4, 2>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_NVFP4, 2>, (int)ws_smem<MOE_NVFP4, 2>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_MXFP8, 2>, (int)ws_smem<MOE_MXFP8, 2>());
    if (e == cudaSuccess) e = ensure_smem_limit((const void*)gemm_ws_kernel<MOE_BF16, 2>, (int)ws_smem<MOE_BF16, 2>());
    if (e != cudaSuccess) return e;
  }
  GemmArgs p{};
  p.tiles = tl;
  p.n_tiles = n_tiles;
  p.slots = slots;
  p.ebytes = g.ebytes;
  p.fmt = g.fmt;
  p.err = err;
  p.ent_bytes = ent_bytes;
  // phase 1
  p.a_scales = xq_scales;
  p.w_scales = wsf;
  p.w_scales_off[0] = g.off_scales[0];
  p.w_scales_off[1] = g.off_scales[1];
  p.w_scales_off[2] = g.off_tscale;
  p.K = g.d;
  p.rows_out = g.f;
  p.act_scale = g.fmt == MOE_NVFP4 ? gx : 1.0f;
  p.h_codes = hq_codes;
  p.h_scales = hq_scales;
  p.act_scale_h = gh;
  const int grid1 = (int)std::min<long long>(num_sms, (long long)max_tiles * (g.f / kTileRows));
  if (ev) cudaEventRecord(ev[0], st);
  if (g.afmt != g.fmt)
    gemm_ws_kernel<kW4A8, 1><<<grid1, ws_threads<1>(), ws_smem<kW4A8, 1>(), st>>>(pl->xq, pl->wg, pl->wu, p);
  else if (g.fmt == MOE_MXFP4)
    gemm_ws_kernel<MOE_MXFP4, 1><<<grid1, ws_threads<1>(), ws_smem<MOE_MXFP4, 1>(), st>>>(pl->xq, pl->wg, pl->wu, p);
  else if (g.fmt == MOE_NVFP4)
    gemm_ws_kernel<MOE_NVFP4, 1><<<grid1, ws_threads<1>(), ws_smem<MOE_NVFP4, 1>(), st>>>(pl->xq, pl->wg, pl->wu, p);
  else if (g.fmt == MOE_MXFP8)
    gemm_ws_kernel<MOE_MXFP8, 1><<<grid1, ws_threads<1>(), ws_smem<MOE_MXFP8, 1>(), st>>>(pl->xq, pl->wg, pl->wu, p);
  else
    gemm_ws_kernel<MOE_BF16, 1><<<grid1, ws_threads<1>(), ws_smem<MOE_BF16, 1>(), st>>>(pl->xq, pl->wg, pl->wu, p);
  e = cudaGetLastError();
  if (ev) cudaEventRecord(ev[1], st);
  if (e != cudaSuccess) return e;
  // phase 2
  p.a_scales = hq_scales;
  p.w_scales = wsf + (blk ? 2 * (size_t)g.d * g.f / blk : 0);
  p.w_scales_off[0] = g.off_scales[2];
  p.w_scales_off[2] = g.off_tscale;
  p.K = g.f;
  p.rows_out = g.d;
  p.act_scale = g.fmt == MOE_NVFP4 ? gh : 1.0f;
  p.O = O;
  p.O_ld = g.d;
  p.O_exp = prefill_o_exp(g, O, N);
  const int grid2 = (int)std::min<long long>(num_sms, (long long)max_tiles * (g.d / 256));
  if (ev) cudaEventRecord(ev[2], st);
  if (g.afmt != g.fmt)
    gemm_ws_kernel<kW4A8, 2><<<grid2, ws_threads<2>(), ws_smem<kW4A8, 2>(), st>>>(pl->hq, pl->wd, pl->wd, p);
  else if (g.fmt == MOE_MXFP4)
    gemm_ws_kernel<MOE_MXFP4, 2><<<grid2, ws_threads<2>(), ws_smem<MOE_MXFP4, 2>(), st>>>(pl->hq, pl->wd, pl->wd, p);
  else if (g.fmt == MOE_NVFP4)
    gemm_ws_kernel<MOE_NVFP4, 2><<<grid2, ws_threads<2>(), ws_smem<MOE_NVFP4, 2>(), st>>>(pl->hq, pl->wd, pl->wd, p);
  else if (g.fmt == MOE_MXFP8)
    gemm_ws_kernel<MOE_MXFP8, 2><<<grid2, ws_threads<2>(), ws_smem<MOE_MXFP8, 2>(), st>>>(pl->hq, pl->wd, pl->wd, p);
  else
    gemm_ws_kernel<MOE_BF16, 2><<<grid2, ws_threads<2>(), ws_smem<MOE_BF16, 2>(), st>>>(pl->hq, pl->wd, pl->wd, p);
  e = cudaGetLastError();
  if (ev) cudaEventRecord(ev[3], st);
  return e;
}

size_t prefill_tile_bytes(const Geo& g, int N) {
  // tiles, then the entries' buffers, keys and refill flags
  return (size_t)prefill_max_tiles(g, N) * sizeof(Tile) + (size_t)3 * (g.E + 2) * sizeof(int);
}

}  // namespace moe
