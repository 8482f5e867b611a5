// Warp-level tensor-core helpers (sm_80+ forms, used on sm_103a by the 16-head
// decode and the few-token cache projection): mma.sync m16n8k16 with bf16
// operands and fp32 accumulators, ldmatrix loads, and the address of a 16-byte
// chunk in a 128B-swizzled tile (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B: chunk j of row r at position j ^ (r mod 8)).
#pragma once

#include <stdint.h>

namespace mla {

// Warp-level MMA and shared-memory matrix loads (PTX ISA: mma.sync,
// ldmatrix).  Fragment layouts of m16n8k16 with g = lane / 4, t = lane % 4:
//   A (16 x 16, row-major): {a0a1, a2a3, a4a5, a6a7} = rows g, g+8, g, g+8 at
//       columns 2t..2t+1, 2t..2t+1, 2t+8..2t+9, 2t+8..2t+9
//   B (16 x 8, column-major): {b0b1, b2b3} = rows 2t..2t+1, 2t+8..2t+9 of column g
//   C (16 x 8 fp32): {c0, c1, c2, c3} = (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// byte offset of the 16-byte chunk `chunk` (8 dims) of token row r in a
// 128B-swizzled box: chunk position j ^ (r mod 8)
__device__ __forceinline__ uint32_t sw128(int r, int chunk) { return (uint32_t)r * 128u + ((uint32_t)(chunk ^ (r & 7)) << 4); }

}  // namespace mla
