// Blackwell (sm_100 family) primitives used by the prefill grouped GEMM:
// mbarriers with bounded waits, TMA tensor loads, tcgen05 TMEM allocation,
// block-scaled FP4 and MXFP8 MMAs, bf16 MMAs, TMEM loads/stores.  All inline
// PTX.  Every kind takes 128-byte operand rows per K tile (256 FP4, 128 FP8
// or 64 bf16 elements) and 32 bytes of them per MMA (K = 64, 32, 16).
//
// Layouts these wrappers assume (checked on GB300 against a CPU product of
// a 128x128x256 tile, both FP4 kinds):
//  * operands: K-major, 128-byte rows (256 FP4 codes), TMA 128B swizzle;
//    matrix descriptor: SBO = 1024 B (8 rows), 128B-swizzle layout, version 1;
//    the k-th MMA of K = 64 codes starts 32 bytes further into the rows;
//  * block scales in TMEM: a group of 4 scale bytes per row (4 blocks along K)
//    occupies 4 columns starting at a multiple of 4; lane 32w + i, column
//    4g + j holds the 4 bytes of row 32j + i (each lane quarter reads its own
//    column), so every quarter holds all 128 rows' group g; the scale-factor id
//    selects the first byte (MXFP4: 2 scales per MMA, id 0 or 2; NVFP4: 4 per
//    MMA, id 0).  tcgen05.cp.32x128b.warpx4 writes exactly this from 512
//    bytes of shared memory (byte 16 i + 4 j + b: row 32 j + i, block b);
//  * an N = 256 MMA reads B's scales for rows 128 h + r from the 4 columns
//    4 h further on (the two 128-row blocks of a group side by side; checked
//    on GB300 by the layer parity tests of every block-scaled kind).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace moe {
namespace tc {

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(su32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(su32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(su32(bar)), "r"(phase) : "memory");
  return ok != 0;
}

// Non-blocking test of the barrier's phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(su32(bar)), "r"(phase) : "memory");
  return ok != 0;
}

// Default limit of a bounded wait: ~2 s of SM clock.
constexpr long long kWaitCycles = 4000000000LL;

// Wait for `phase` of the barrier, at most `limit` SM clock cycles; false on
// timeout.  try_wait may suspend the thread inside the instruction until the
// phase completes, so a short limit (a test's) polls with test_wait, which
// returns at once.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, long long limit = kWaitCycles) {
  const long long t0 = clock64();
  if (limit < 1000000) {
    while (!mbar_test(bar, phase))
      if (clock64() - t0 > limit) return false;
    return true;
  }
  while (!mbar_try(bar, phase))
    if (clock64() - t0 > limit) return false;
  return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3}], [%4];"
               :: "r"(su32(dst)), "l"(map), "r"(x), "r"(y), "r"(su32(bar)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3, %4}], [%5];"
               :: "r"(su32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(su32(bar)) : "memory");
}

// Non-tensor bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completing on `bar` like a tensor load.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar)) : "memory");
}

// whole warp
// Fetch a tensor map (a __grid_constant__ parameter) into the descriptor cache.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(su32(dst_smem)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile of 128-byte rows, 128B swizzle, 1024-byte aligned base.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;                 // leading offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128B swizzle
  return d;
}

// Descriptor of a plain (unswizzled) shared-memory matrix of 16-byte rows
// stored back to back: core matrices of 8 rows x 16 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;        // leading offset (one core matrix wide: unused)
  d |= (uint64_t)(128 >> 4) << 32;        // stride offset: the next 8 rows
  d |= (uint64_t)1 << 46;                 // descriptor version
  return d;                               // no swizzle
}

// Block scales into TMEM: 32 rows of 16 bytes from shared memory (sdesc_rows16)
// to columns taddr .. taddr + 3, row i into lane i of every lane quarter
// (lanes i, 32 + i, 64 + i, 96 + i).  Asynchronous; ordered before the MMAs
// the same thread issues after it, and tracked by its later commits.
__device__ __forceinline__ void cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc));
}

// Instruction descriptor of a block-scaled FP4 MMA (M = 128, dense, K-major).
__device__ __forceinline__ uint32_t idesc_fp4(int N, bool ue8m0, uint32_t sf_a, uint32_t sf_b) {
  uint32_t d = (1u << 7) | (1u << 10);            // E2M1 A and B
  d |= (uint32_t)(N >> 3) << 17;
  if (ue8m0) d |= 1u << 23;
  d |= (128u >> 4) << 24;
  d |= (sf_b & 3u) << 4;
  d |= (sf_a & 3u) << 29;
  return d;
}

// D (+)= A x B^T with block scales; single thread.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
               :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
                  "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
               :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
                  "r"((uint32_t)accumulate));
}

// Instruction descriptor of a block-scaled kind::mxf8f6f4 MMA (A E4M3; B
// E4M3, or E2M1 when b_e2m1; UE8M0 scales, M = 128, dense, K-major); sf_a /
// sf_b select the scale byte of the 4-byte group (one scale per 32-K MMA).
// An E2M1 operand sits in shared memory unpacked, 16 codes (8 bytes) per
// 16-byte chunk as the TMA's 16 x U4 load writes them, so its rows have the
// byte extent of an E4M3 tile (128 elements per 128-byte row).
__device__ __forceinline__ uint32_t idesc_mxf8(int N, uint32_t sf_a, uint32_t sf_b, bool b_e2m1 = false) {
  uint32_t d = 0;                                 // A E4M3 (type 0)
  if (b_e2m1) d |= 5u << 10;                      // B E2M1 (type 5 of this kind)
  d |= (uint32_t)(N >> 3) << 17;
  d |= 1u << 23;                                  // UE8M0 scales
  d |= (128u >> 4) << 24;
  d |= (sf_b & 3u) << 4;
  d |= (sf_a & 3u) << 29;
  return d;
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
               :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
                  "r"((uint32_t)accumulate));
}

// Instruction descriptor of a bf16 x bf16 -> fp32 MMA (M = 128, dense, K-major).
__device__ __forceinline__ uint32_t idesc_bf16(int N) {
  uint32_t d = 1u << 4;                           // D fp32
  d |= (1u << 7) | (1u << 10);                    // A and B bf16
  d |= (uint32_t)(N >> 3) << 17;
  d |= (128u >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
}

// Arrive on `bar` when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(su32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(taddr), "r"(a), "r"(b), "r"(c), "r"(d));
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
               "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                 "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
                 "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
                 "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
                 "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
                 "=r"(v[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace moe
