// tc.cuh -- sm_103a tensor-core building blocks: 2-D TMA tile loads, TMEM allocation,
// tcgen05 MMA (bf16 x bf16 -> f32, operands K-major in 128-byte-swizzled shared
// memory), MMA completion to an mbarrier, and TMEM -> register loads.
//
// Encodings (PTX ISA, tcgen05 "Shared memory descriptor" and "Instruction
// descriptor" for .kind::f16):
//   shared memory descriptor (64 bits): start address >> 4 in bits 0-13, leading
//     byte offset >> 4 in bits 16-29, stride byte offset >> 4 in bits 32-45, the
//     fixed value 1 in bits 46-47, base offset 0 in bits 49-51, swizzle mode in
//     bits 61-63 (2 = 128-byte swizzle);
//   instruction descriptor (32 bits): D format in bits 4-5 (1 = f32), A format in
//     bits 7-9 and B format in bits 10-12 (1 = bf16), A/B major in bits 15/16
//     (0 = K-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
// A K-major tile of R rows x 64 bf16 loaded by TMA with 128-byte swizzling is R
// rows of 128 bytes, the 16-byte chunks of row r permuted by r mod 8; groups of 8
// rows are 1024 bytes apart (the stride byte offset), and the 16-element step of
// one MMA along K advances the start address by 32 bytes.  With 32 bf16 per row and
// 64-byte swizzling the rows are 64 bytes and the groups 512 bytes apart.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace adaflash {

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// One warp: allocate ncols TMEM columns (a power of two >= 32); the address goes to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major tile of rows of `row_bytes` (128 or 64) swizzled at that width: 8-row groups
// are 8 * row_bytes apart; swizzle mode 2 (128-byte) or 4 (64-byte).
template <int kRowBytes>
__device__ __forceinline__ uint64_t sdesc_swizzled(uint32_t saddr) {
  static_assert(kRowBytes == 128 || kRowBytes == 64, "128- or 64-byte swizzle");
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>((8 * kRowBytes) >> 4) << 32;  // stride byte offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                   // fixed value
  d |= static_cast<uint64_t>(kRowBytes == 128 ? 2 : 4) << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 16-deep step; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on bar once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 16 consecutive f32 columns of this thread's TMEM lane; the values are usable
// after tmem_wait16 on the same array.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Wait for this thread's TMEM loads; the registers are tied to the wait so that no
// use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

}  // namespace adaflash
