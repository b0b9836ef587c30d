// tcgen05.cuh -- thin inline-PTX wrappers for the 5th-generation tensor cores (sm_100+):
// tensor-memory allocation, shared-memory matrix descriptors, bf16 MMA into TMEM,
// completion through an mbarrier, and TMEM <-> register moves.
//
// Operand convention used throughout this library: every MMA operand is a K-major bf16
// tile in shared memory with the 128-byte swizzle.  A tile of R rows x Kd elements
// (Kd a multiple of 64) is stored as Kd/64 column blocks of [R][64] elements; inside a
// block row r occupies 128 bytes and its 16-byte chunk c sits at chunk c ^ (r % 8).
// Tiles start on 1024-byte boundaries.  The accumulator of an M = 128 MMA holds row m in
// TMEM lane m and column n in TMEM column n (f32).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace gdn {
namespace tc {

// Byte offset of element (r, k) of a K-major, 128B-swizzled bf16 tile with R rows.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int R, int r, int k) {
  return uint32_t((k >> 6) * R * 128 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) +
                  ((k & 7) << 1));
}

// Shared-memory matrix descriptor: K-major, SWIZZLE_128B, 8-row groups 1024 B apart.
// `addr` is the shared-window address of the first element the MMA reads (the tile
// base plus the K offset of this instruction, within the 128-byte swizzle row).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= uint64_t((addr >> 4) & 0x3FFFu);          // start address
  d |= uint64_t(1u) << 16;                        // leading byte offset (unused here)
  d |= uint64_t((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1u) << 46;                        // descriptor version for sm_100
  d |= uint64_t(2u) << 61;                        // layout: SWIZZLE_128B
  return d;
}

// MN-major, SWIZZLE_128B: the operand is stored [K rows][MN elements] with 64-element
// (128-byte) MN blocks `lbo_bytes` apart; 8 K rows span 1024 bytes.  `addr` points at the
// first K row the instruction reads (advance 16 rows = 2048 bytes per K = 16 step).
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t lbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((addr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;  // stride between 64-element MN blocks
  d |= uint64_t((1024u >> 4) & 0x3FFFu) << 32;      // stride between 8-row K groups
  d |= uint64_t(1u) << 46;
  d |= uint64_t(2u) << 61;
  return d;
}

// Descriptor of the K sub-block starting at element k0 (a multiple of 16) of a tile.
__device__ __forceinline__ uint64_t desc_at(uint32_t tile_addr, int R, int k0) {
  return desc_sw128(tile_addr + uint32_t((k0 >> 6) * R * 128 + (k0 & 63) * 2));
}

// Instruction descriptor of kind::f16 with an f32 accumulator: A and B both bf16 (or both
// fp16 when `fp16`), K-major unless a_mn / b_mn select MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false,
                                                  bool b_mn = false, bool fp16 = false) {
  return (1u << 4)                       // D format: f32
         | (uint32_t(!fp16) << 7)        // A format: 1 = bf16, 0 = fp16
         | (uint32_t(!fp16) << 10)       // B format: 1 = bf16, 0 = fp16
         | (uint32_t(a_mn) << 15)        // A major-ness
         | (uint32_t(b_mn) << 16)        // B major-ness
         | (uint32_t(N >> 3) << 17)      // N / 8
         | (uint32_t(M >> 4) << 24);     // M / 16
}
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn = false,
                                                 bool b_mn = false) {
  return idesc_bf16(M, N, a_mn, b_mn, true);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K = 16 step of kind::f16 (bf16 or fp16
// operands as the instruction descriptor says), issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Tensor-memory allocation: executed by one whole warp.  The TMEM address lands in *slot.
__device__ __forceinline__ void alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns in one load: thread t of warp w gets lane
// 32*(w%4)+t.  The wait is part of the same statement, so no use of the values can
// precede it.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace tc
}  // namespace gdn
