// Decode expert FFN: a persistent, warp-specialised grouped GEMV over the
// experts of one work range, weights read through the slot table and
// dequantised in registers.
//
// Decode moves each routed expert's weights once per step for a handful of
// tokens, so the kernel is bound by HBM bandwidth (the pages' decode is bound
// by the bytes each step must move: "FreeToken：把 284B MoE 塞进游戏 PC",
// zhichai.net, §二 "Decode" paragraph).  Design:
//  * work unit = one expert entry x one matrix x a 64-row block (all of K);
//    one CTA per SM, persistent, each taking an equal contiguous range of
//    the launch's units, so every SM streams from the first cycle;
//  * three roles that only meet at mbarriers, so loads, math and reductions
//    overlap and no warp waits for a CTA-wide barrier:
//    - a producer warp streams the unit's codes as TMA boxes of 64 rows x
//      256 K (128 bytes per row, 128-byte swizzle), four boxes per stage,
//      plus their scale bytes (one more TMA box, or one bulk copy), into a
//      ring of shared-memory stages; tall boxes and a handful of copy
//      instructions per 32 KB keep the copy engine near the HBM rate;
//    - 16 compute warps: warp (b, q) takes the 16-row quarter q of box b of
//      every stage, so a unit's K splits four ways and each warp accumulates
//      its share across the unit's stages;
//    - 3 epilogue warps stage the next token group's activations and add the
//      four partial sums of each output in a fixed order (deterministic);
//  * the token dimension goes through tensor-core MMAs (mma.sync m16n8k16,
//    f16 x f16 -> f32): a lane's 32-bit word of codes becomes four f16x2 A
//    registers with cvt.rn.f16x2.e2m1x2 (exact); the activations are staged
//    once per token group as f16 (power-of-two scaled per token so nothing
//    overflows) in B-fragment order, so each B load is one contiguous 256-byte
//    warp access; each MMA stays inside one scale block, whose scale is
//    applied to the MMA sum in fp32; the swizzle makes the A loads
//    conflict-free.
// Phase 1: a = W_g x and u = W_u x (separate units), fp32 [rows, 2 d_ff].
// Phase 2: O = W_d h with h = SiLU(a) * u formed while staging, fp32 [rows, d_model].

#include "gemv_dev.cuh"

namespace moe {

namespace {

using namespace gv;

// HOST: the launch may stream misses from the host pool (GemvArgs::host_pool);
// launches over resident weights only use the variant without that path.
template <int FMT, int PH, bool HOST>
__global__ void __launch_bounds__(kThreads, 1)
gemv_stream_kernel(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
                   const __grid_constant__ CUtensorMap smap0, const __grid_constant__ CUtensorMap smap1,
                   Geo g, GemvArgs a, SG p, const __nv_bfloat16* __restrict__ x,
                   const int* __restrict__ xexp, float* __restrict__ h, float* __restrict__ O) {
  extern __shared__ uint8_t smem_raw[];
  Smem S;
  S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  S.full = reinterpret_cast<uint64_t*>(S.base + p.off_bar);
  S.empty = S.full + p.D;
  S.rfull = S.empty + p.D;
  S.rempty = S.rfull + 2;
  S.xfull = S.rempty + 2;
  S.xempty = S.xfull + 2;
  __shared__ Small sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // operational waits give up after wl cycles; the final wait for the
  // producer's own copies in flight keeps the default limit
  const long long wl = a.wait_cycles > 0 ? a.wait_cycles : tc::kWaitCycles;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.D; ++i) {
      tc::mbar_init(&S.full[i], 1);
      tc::mbar_init(&S.empty[i], kCW);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&S.rfull[i], kCW);
      tc::mbar_init(&S.rempty[i], kEW);
      tc::mbar_init(&S.xfull[i], kEW);
      tc::mbar_init(&S.xempty[i], kCW);
    }
    sm.abort = 0;
    tc::mbar_init_fence();
  }
  __syncthreads();
  // launched as a dependent of the previous kernel: phase 2's producer only
  // reads the step record and weights, both final before phase 1 got past its
  // own wait, so it starts streaming at once; everything else waits for the
  // predecessor.  The successor is released only after this wait, so what
  // the successor's producer reads without waiting is final by then.
  if (warp == kProd && lane == 0) {
    // descriptor fetches overlap the wait for the predecessor
    tc::prefetch_tmap(&map0);
    tc::prefetch_tmap(&map1);
    if (p.smode) {
      tc::prefetch_tmap(&smap0);
      tc::prefetch_tmap(&smap1);
    }
  }
  const bool ALL = PH == 1 && p.all;
  if (ALL && warp != kProd) {
    // every token of the step, before the wait: x is final before the router starts
    const int tid = warp < kCW ? threadIdx.x : threadIdx.x - 32;
    stage_all<FMT>(p, a.N, x, reinterpret_cast<uint2*>(S.base + p.off_x), &sm.sexp[0][0], tid, kThreads - 32, 2);
  }
  if (PH == 1 || warp != kProd) pdl_wait();
  pdl_trigger();
  // the launch's work: the access range its mode selects (+ the shared expert)
  EntryTable T{};
  {
    const StepRecord* rec = a.rec;
    const int U = min(max(rec->U, 0), g.E), nh = min(max(rec->n_hit, 0), U);
    int b = 0, e = nh;
    if (a.mode == kRangeAll) {
      e = U;
    } else if (a.mode != kRangeHits) {
      // misses [nh, U), or chunk `chunk` of n_chunks of them
      const int C = max(a.n_chunks, 1), c = min(max(a.chunk, 0), C - 1);
      int lo, hi;
      miss_chunk(U - nh, c, C, &lo, &hi);
      b = nh + lo;
      e = nh + hi;
    }
    T.ent = rec_entry(const_cast<StepRecord*>(rec), g.E);
    T.expert = rec_expert(const_cast<StepRecord*>(rec));
    T.base = b;
    T.nr = max(0, e - b);
    T.n_hit = nh;
    T.shared = a.with_shared ? 1 : 0;
  }
  const Range rr = cta_range(T, p, blockIdx.x, gridDim.x);
  // the first token group is staged by every warp but the producer (its
  // latency is on the critical path); the epilogue stages later ones ahead
  bool first_staged = false;
  if (!ALL && warp != kProd) {
    Cursor c0;
    cursor_init(c0, rr);
    if (cursor_next(c0, g, a, T, p, rr)) {
      const int tid = warp < kCW ? threadIdx.x : threadIdx.x - 32;
      stage_block<FMT, PH>(g, a, p, c0.en, c0.tg, reinterpret_cast<uint2*>(S.base + p.off_x), sm.sexp[0], sm.stok,
                           x, xexp, h, tid, kThreads - 32, 2);
      asm volatile("bar.sync 2, %0;" :: "n"(kThreads - 32) : "memory");
      if (warp > kCW && lane == 0) mbar_arrive(&S.xfull[0]);
      first_staged = true;
    }
  }
  Ring ring;
  if (warp == kProd) {
    produce<FMT, PH, HOST>(g, a, p, T, rr, S, sm, ring, &map0, &map1, &smap0, &smap1, wl);
    produce_drain(S, p.D, ring, a.err);
  } else if (warp < kCW) {
    compute<FMT, PH, HOST>(g, a, p, T, rr, S, sm, ring, wl);
  } else {
    reduce<FMT, PH, HOST>(g, a, p, T, rr, S, sm, ring, first_staged, x, xexp, h, O, wl);
  }
  __syncthreads();
}

template <int FMT, int PH, bool HOST>
cudaError_t launch_phase(const Geo& g, const GemvPlan* pl, const GemvArgs& a, const SG& p,
                         const __nv_bfloat16* x, const int* xexp, float* h, float* O, int n_ent_max,
                         int num_sms, cudaStream_t st) {
  cudaError_t e = ensure_smem_limit((const void*)gemv_stream_kernel<FMT, PH, HOST>, kSmemBudget + 1024);
  if (e != cudaSuccess) return e;
  const long long units = (long long)n_ent_max * p.UE;
  // phase 1 is launched while the one-CTA routing tail still holds an SM, and
  // a CTA of this size cannot share it: leave that SM out rather than have
  // one CTA start after the tail and finish last
  const int grid = (int)std::min<long long>(PH == 1 ? std::max(1, num_sms - 1) : num_sms, units);
  if (grid <= 0) return cudaSuccess;
  const CUtensorMap& m0 = PH == 1 ? pl->w[0] : pl->w[2];
  const CUtensorMap& m1 = PH == 1 ? pl->w[1] : pl->w[2];
  const CUtensorMap& s0 = PH == 1 ? pl->s[0] : pl->s[2];
  const CUtensorMap& s1 = PH == 1 ? pl->s[1] : pl->s[2];
  return launch_pdl(gemv_stream_kernel<FMT, PH, HOST>, dim3(grid), dim3(kThreads), (size_t)p.smem, st, m0, m1, s0,
                    s1, g, a, p, x, xexp, h, O);
}

template <int FMT>
cudaError_t launch_fmt(const Geo& g, const GemvPlan* pl, const GemvArgs& a, const __nv_bfloat16* x,
                       const int* xexp, float* h, float* O, int n_ent_max, int num_sms,
                       cudaStream_t st, const cudaEvent_t* ev, int phases) {
  cudaError_t e = cudaSuccess;
  if (phases & 1) {
    const SG p1 = make_sg(g, 1, a.N);
    if (ev) cudaEventRecord(ev[0], st);
    e = a.host_pool ? launch_phase<FMT, 1, true>(g, pl, a, p1, x, xexp, h, O, n_ent_max, num_sms, st)
                    : launch_phase<FMT, 1, false>(g, pl, a, p1, x, xexp, h, O, n_ent_max, num_sms, st);
    if (ev) cudaEventRecord(ev[1], st);
    if (e != cudaSuccess) return e;
  }
  if (phases & 2) {
    const SG p2 = make_sg(g, 2, a.N);
    if (ev) cudaEventRecord(ev[2], st);
    e = a.host_pool ? launch_phase<FMT, 2, true>(g, pl, a, p2, x, xexp, h, O, n_ent_max, num_sms, st)
                    : launch_phase<FMT, 2, false>(g, pl, a, p2, x, xexp, h, O, n_ent_max, num_sms, st);
    if (ev) cudaEventRecord(ev[3], st);
  }
  return e;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
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

// Codes of one matrix in every slot: [slot][row][K/2 bytes], boxes of
// 64 rows x 128 bytes, 128-byte swizzle; a box past the row end reads zeros.
bool make_box_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                  uint64_t slot_stride) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {kBoxRowBytes, kBoxRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale bytes of one matrix in every slot: [slot][row][scale_row], boxes of
// 64 rows x (4 code boxes' scale bytes), no swizzle.
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
                    uint64_t slot_stride, uint32_t box_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, slots};
  cuuint64_t strides[2] = {row_bytes, slot_stride};
  cuuint32_t box[3] = {box_bytes, kBoxRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Shapes the decode kernels accept: d_model and d_ff multiples of 128 (so
// the 64-row blocks tile both) up to 8192, and a ring of at least two stages
// next to the staged activations.
bool gemv_shape_ok(const Geo& g) {
  if (g.d > 8192 || g.f > 8192 || g.d % 128 || g.f % 128) return false;
  return make_sg(g, 1, 0).D >= 2 && make_sg(g, 2, 0).D >= 2;
}

GemvPlan* gemv_plan_create(const Geo& g, const uint8_t* slots) {
  GemvPlan* pl = new GemvPlan();
  const int ns = g.nbuf;   // LRU slots' buffers, the shared expert's, the spares (+ a stack's other shared experts)
  const int cb = fmt_code_bits(g.fmt);   // row bytes = K * cb / 8
  pl->ready = make_box_map(&pl->w[0], slots + g.off_codes[0], (size_t)g.d * cb / 8, g.f, ns, g.ebytes) &&
              make_box_map(&pl->w[1], slots + g.off_codes[1], (size_t)g.d * cb / 8, g.f, ns, g.ebytes) &&
              make_box_map(&pl->w[2], slots + g.off_codes[2], (size_t)g.f * cb / 8, g.d, ns, g.ebytes);
  // scale maps only where a scale row is a 16-byte multiple (the phase uses them then)
  const SG p1 = make_sg(g, 1, 0), p2 = make_sg(g, 2, 0);
  const uint32_t sb = kBoxes * p1.SBB;
  if (sb == 0) return pl;   // no block scales
  if (pl->ready && p1.smode)
    pl->ready = make_scale_map(&pl->s[0], slots + g.off_scales[0], p1.scale_row, g.f, ns, g.ebytes, sb) &&
                make_scale_map(&pl->s[1], slots + g.off_scales[1], p1.scale_row, g.f, ns, g.ebytes, sb);
  if (pl->ready && p2.smode)
    pl->ready = make_scale_map(&pl->s[2], slots + g.off_scales[2], p2.scale_row, g.d, ns, g.ebytes, sb);
  return pl;
}

void gemv_plan_destroy(GemvPlan* pl) { delete pl; }
bool gemv_plan_ready(const GemvPlan* pl) { return pl && pl->ready; }

cudaError_t launch_gemv_decode(const Geo& g, const GemvPlan* pl, const GemvArgs& a,
                               const __nv_bfloat16* x, const int* xexp, float* h, float* O,
                               int n_ent_max, int num_sms, cudaStream_t st, const cudaEvent_t* ev,
                               int phases) {
  if (g.fmt == MOE_MXFP4)
    return launch_fmt<MOE_MXFP4>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
  if (g.fmt == MOE_NVFP4)
    return launch_fmt<MOE_NVFP4>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
  if (g.fmt == MOE_MXFP8)
    return launch_fmt<MOE_MXFP8>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
  return launch_fmt<MOE_BF16>(g, pl, a, x, xexp, h, O, n_ent_max, num_sms, st, ev, phases);
}

}  // namespace moe
