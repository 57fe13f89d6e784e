// tcgen05 (5th-generation tensor core) helpers for sm_103a: shared-memory
// matrix descriptors for 128-byte-swizzled K-major fp16 tiles, the kind::f16
// instruction descriptor, MMA issue/commit, TMEM allocation and loads, and
// bulk (TMA) shared->global stores.
//
// Tile convention ("SW128 image"): a K-major operand with R rows and K columns
// of fp16 is stored as K/64 column blocks, each [R rows][128 bytes]; inside a
// row the 16-byte chunk c sits at position c ^ (row % 8). Every tile starts on
// a 1024-byte boundary. The descriptor of column block kb, k-step ks (16
// columns = 32 bytes) starts at base + kb*R*128 + ks*32, with the 8-row group
// stride (SBO) 1024 bytes.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {

// Byte offset of element (row, col) in an SW128 image with R rows.
__device__ __forceinline__ uint32_t sw128_off(int R, int row, int col) {
  return (uint32_t)((col >> 6) * R * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}
// Byte offset of the 16-byte chunk holding columns [8*c8, 8*c8+8) of a row.
__device__ __forceinline__ uint32_t sw128_chunk(int R, int row, int c8) {
  return (uint32_t)((c8 >> 3) * R * 128 + row * 128 + (((c8 & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A(desc_a) * B(desc_b)^T over one K=16 step. One thread issues.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}

// Descriptor of an MN-major SW128 fp16 operand stored [K rows][MN columns]:
// 64-column MN blocks `lbo` bytes apart, each [rows][128 bytes] with the same
// chunk swizzle as a K-major image, 8-row K groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor with B read MN-major (A K-major).
__host__ __device__ constexpr uint32_t umma_idesc_f16_bmn(int M, int N) { return umma_idesc_f16(M, N) | (1u << 16); }

// D = A[0:M, 0:K] * B[0:K, 0:N]: A a K-major SW128 image with RA rows, B an
// MN-major image [K rows][N] whose 64-column blocks are lbo bytes apart
// (a [token][d] image read with the tokens as the contraction).
__device__ __forceinline__ void umma_tile_bmn(uint32_t tmem_d, uint32_t sa, int RA, uint32_t sb, uint32_t lbo, int K,
                                              uint32_t idesc, bool acc_first) {
  for (int k = 0; k < K / 16; ++k) {
    const int kb = k >> 2, ks = k & 3;
    umma_f16(tmem_d, umma_desc(sa + kb * RA * 128 + ks * 32), umma_desc_mn(sb + k * 2048, lbo), idesc,
             acc_first || k > 0);
  }
}

// A full MxN product over K (multiple of 16), operands as SW128 images with
// RA / RB rows: D = A[0:M, 0:K] * B[0:N, 0:K]^T.
__device__ __forceinline__ void umma_tile(uint32_t tmem_d, uint32_t sa, int RA, uint32_t sb, int RB, int K,
                                          uint32_t idesc, bool acc_first) {
  for (int k = 0; k < K / 16; ++k) {
    const int kb = k >> 2, ks = k & 3;
    umma_f16(tmem_d, umma_desc(sa + kb * RA * 128 + ks * 32), umma_desc(sb + kb * RB * 128 + ks * 32), idesc,
             acc_first || k > 0);
  }
}

// Arrive on `bar` once every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Warp-wide TMEM allocation of `ncols` (power of two >= 32); the base address
// is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// TMEM address of lane quarter q (lanes 32q..32q+31), column col.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int q, int col) {
  return base + ((uint32_t)(32 * q) << 16) + (uint32_t)col;
}


// 2-D tensor-map (TMA) tile load / store; coordinates in elements (x inner).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, const void *smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace gdn
