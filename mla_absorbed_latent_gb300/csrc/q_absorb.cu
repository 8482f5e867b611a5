// Query-side key absorption: q_lat[b,h,:] = W_UK[h]^T q_nope[b,h,:].
//
// "DeepSeek MLA 吸收式缓存" §2.2: q^T (W_UK c_t) = (W_UK^T q)^T c_t, so the
// key up-projection moves from every cached token onto the one query token;
// "手搓 MLA" §四 writes it as einsum("thd,hdc->thc", q_nope, W_UK).
//
// Per head this is a small GEMM, M = B rows, N = 512, K = 128, run on the
// warp-level bf16 tensor-core MMA with fp32 accumulation; the result is
// rounded once to bf16 because it is the bf16 A operand of the score MMA.
// The output row is the 576-wide query of the latent attention: q_lat
// followed by a copy of q_pe.
#include "mla_common.cuh"

namespace mla {
namespace {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// grid (H, ceil(B/64)); 8 warps; warp w owns latent columns [64w, 64w+64).
__global__ void __launch_bounds__(256) q_absorb_kernel(const uint16_t* __restrict__ q_nope,
                                                        const uint16_t* __restrict__ q_pe,
                                                        const uint16_t* __restrict__ w_uk, int H, int B,
                                                        uint16_t* __restrict__ q_cat) {
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n_base = warp * 64;

  float acc[4][8][4];
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int ni = 0; ni < 8; ++ni)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mi][ni][r] = 0.f;

  const uint16_t* wk = w_uk + (size_t)h * DC * DN;
#pragma unroll 1
  for (int k0 = 0; k0 < DN; k0 += 16) {
    uint32_t bf[8][2];
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const uint16_t* row = wk + (size_t)(n_base + ni * 8 + g) * DN + k0 + 2 * t;
      bf[ni][0] = *reinterpret_cast<const uint32_t*>(row);
      bf[ni][1] = *reinterpret_cast<const uint32_t*>(row + 8);
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      const int r0 = b0 + mi * 16 + g, r1 = r0 + 8;
      uint32_t af[4] = {0u, 0u, 0u, 0u};
      if (r0 < B) {
        const uint16_t* a = q_nope + ((size_t)r0 * H + h) * DN + k0 + 2 * t;
        af[0] = *reinterpret_cast<const uint32_t*>(a);
        af[2] = *reinterpret_cast<const uint32_t*>(a + 8);
      }
      if (r1 < B) {
        const uint16_t* a = q_nope + ((size_t)r1 * H + h) * DN + k0 + 2 * t;
        af[1] = *reinterpret_cast<const uint32_t*>(a);
        af[3] = *reinterpret_cast<const uint32_t*>(a + 8);
      }
#pragma unroll
      for (int ni = 0; ni < 8; ++ni) mma_bf16_16816(acc[mi][ni], af, bf[ni]);
    }
  }

#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
    const int r0 = b0 + mi * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const int col = n_base + ni * 8 + 2 * t;
      if (r0 < B)
        *reinterpret_cast<uint32_t*>(q_cat + ((size_t)r0 * H + h) * DK + col) =
            pack_bf16x2(acc[mi][ni][0], acc[mi][ni][1]);
      if (r1 < B)
        *reinterpret_cast<uint32_t*>(q_cat + ((size_t)r1 * H + h) * DK + col) =
            pack_bf16x2(acc[mi][ni][2], acc[mi][ni][3]);
    }
  }

  // q_pe rows of this block: 64 rows x 8 vectors of 16 bytes
  for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {
    const int r = b0 + i / 8, v = i % 8;
    if (r < B)
      reinterpret_cast<uint4*>(q_cat + ((size_t)r * H + h) * DK + DC)[v] =
          reinterpret_cast<const uint4*>(q_pe + ((size_t)r * H + h) * DR)[v];
  }
}

}  // namespace

cudaError_t launch_q_absorb(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* q_cat,
                            cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  q_absorb_kernel<<<dim3(H, (B + 63) / 64), 256, 0, s>>>(
      static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe), static_cast<const uint16_t*>(W_UK),
      H, B, static_cast<uint16_t*>(q_cat));
  return cudaGetLastError();
}

}  // namespace mla
