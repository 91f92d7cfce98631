// lsc_tc.h -- inline-PTX helpers of liblsc for the 5th-generation tensor cores
// of sm_103a: tensor-memory (TMEM) allocation, tcgen05.mma of kind tf32 with
// operands in shared memory (no swizzle, "interleaved" core matrices) or, for
// A, in TMEM, completion through tcgen05.commit on an mbarrier, and TMEM <->
// register moves.  One CTA per instruction (cta_group::1), no clusters.
//
// Shared-memory operand layout used with these descriptors (no swizzle): the
// matrix is cut into core matrices of 8 rows x 16 bytes (8 x 4 tf32), each
// stored as 128 contiguous bytes (row i of the core matrix at byte 16 i).
//  * K-major operand (rows = M or N, 16-byte groups along K): the descriptor's
//    leading byte offset (LBO) is the distance between core matrices adjacent
//    along K, the stride byte offset (SBO) between core matrices adjacent
//    along M/N (8-row groups).
//  * MN-major operand (16-byte groups along M/N, 8 K rows per core matrix):
//    SBO is the distance between core matrices adjacent along M/N, LBO the
//    distance between 8-row groups along K.
// A tile stored with element (row, col) at (row/8)*RG + (col/4)*128 +
// (row%8)*16 + (col%4)*4 is therefore a K-major operand with K = col
// (LBO 128, SBO RG) and, read the other way, an MN-major operand with
// MN = col, K = row (SBO 128, LBO RG).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lsc_ptx.h"

namespace lsc {
namespace tc {

// ---- descriptors -------------------------------------------------------------

// Shared-memory matrix descriptor: start address, LBO and SBO in bytes (all
// multiples of 16), version 1 (bits 46-48 = 0b001), base offset 0, relative
// LBO, no swizzle (bits 61-63 = 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::tf32 with an fp32 accumulator: D format f32
// (bits 4-5 = 1), A and B tf32 (bits 7-9, 10-12 = 2), A K-major (bit 15 = 0),
// B K-major or MN-major (bit 16), N / 8 at bits 17-22, M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---- TMEM allocation (one warp, .sync.aligned) -------------------------------

// Allocate ncols TMEM columns (a power of two >= 32); the base address is
// written to *dst_smem.  Called by every thread of one warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering ----------------------------------------------------------------

// Before a thread barrier that orders this thread's tcgen05 operations before
// other threads' later ones; after the barrier, in the threads that follow.
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- MMA (issued by one thread) ------------------------------------------------

// True on one lane of the calling (converged) warp.  Issuing MMAs under it
// from code that every lane of the warp runs keeps their operands
// warp-uniform, so they stay in uniform registers.
__device__ __forceinline__ bool elect_one() {
  uint32_t is = 0;
  asm volatile(
      "{\n\t.reg .b32 lid;\n\t.reg .pred p;\n\telect.sync lid|p, %1;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(is)
      : "r"(0xffffffffu));
  return is != 0;
}

// D[tmem] (+)= A[smem] x B[smem]^T  (A: M x K, B: N x K as seen by the descriptors)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem]^T  (A: M lanes x K columns of tf32 values)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- TMEM <-> registers (warp-wide; a warp reaches the 32 lanes of its
// sub-partition, warp index % 4) --------------------------------------------------

#define LSC_TC_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                     "=r"(v[i + 6]), "=r"(v[i + 7])
#define LSC_TC_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                     "r"(v[i + 6]), "r"(v[i + 7])

// 32 consecutive columns of this thread's lane -> v[0..31] (raw 32-bit words).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : LSC_TC_R8(0), LSC_TC_R8(8), LSC_TC_R8(16), LSC_TC_R8(24)
      : "r"(taddr)
      : "memory");
}

// v[0..31] -> 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      LSC_TC_W8(0), LSC_TC_W8(8), LSC_TC_W8(16), LSC_TC_W8(24)
      : "memory");
}
// 4 consecutive columns of this thread's lane -> v[0..3].
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr)
               : "memory");
}

// 16 consecutive columns of this thread's lane -> v[0..15].
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : LSC_TC_R8(0), LSC_TC_R8(8)
      : "r"(taddr)
      : "memory");
}

// v[0..15] -> 16 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      LSC_TC_W8(0), LSC_TC_W8(8)
      : "memory");
}

#undef LSC_TC_R8
#undef LSC_TC_W8

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of (lane, column) relative to an allocation base.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// ---- tf32 splitting ------------------------------------------------------------

// x rounded to tf32 (10 explicit mantissa bits, round to nearest, ties away),
// as the bits of an fp32 value whose low 13 bits are zero.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// x = hi + lo with hi = tf32(x) and lo = tf32(x - hi); x - hi is exact in
// fp32, so hi + lo carries about 22 significant bits of x.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}

}  // namespace tc
}  // namespace lsc
