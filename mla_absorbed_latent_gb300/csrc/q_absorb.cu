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

// grid (H, 4 column quarters, ceil(B/64)); 8 warps.  The CTA stages the 64
// query rows of head h (64 x 128 bf16) in shared memory once; warp w owns
// latent columns [128q + 16w, +16) and loads all of its W_UK fragments (16
// columns x K=128) before the first MMA, so the global loads overlap.
constexpr int QROWS = 64;
constexpr int QLD = DN + 8;  // padded bf16 row stride of the staged queries (conflict-free fragment reads)

__global__ void __launch_bounds__(256) q_absorb_kernel(const uint16_t* __restrict__ q_nope,
                                                        const uint16_t* __restrict__ q_pe,
                                                        const uint16_t* __restrict__ w_uk, int H, int B,
                                                        uint16_t* __restrict__ q_cat) {
  __shared__ __align__(16) uint16_t qs[QROWS * QLD];
  const int h = blockIdx.x, quarter = blockIdx.y;
  const int b0 = blockIdx.z * QROWS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n_base = quarter * 128 + warp * 16;

  // W_UK fragments of this warp's 16 columns, all of K = 128
  const uint16_t* wk = w_uk + (size_t)h * DC * DN;
  uint32_t bf[8][2][2];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      const uint16_t* row = wk + (size_t)(n_base + ni * 8 + g) * DN + kk * 16 + 2 * t;
      bf[kk][ni][0] = __ldg(reinterpret_cast<const unsigned int*>(row));
      bf[kk][ni][1] = __ldg(reinterpret_cast<const unsigned int*>(row + 8));
    }
  // the block's query rows (zeros past B)
  for (int i = threadIdx.x; i < QROWS * (DN / 8); i += blockDim.x) {
    const int r = i / (DN / 8), v = i % (DN / 8);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (b0 + r < B) x = __ldg(reinterpret_cast<const uint4*>(q_nope + ((size_t)(b0 + r) * H + h) * DN) + v);
    *reinterpret_cast<uint4*>(qs + r * QLD + v * 8) = x;
  }
  __syncthreads();

  float acc[4][2][4];
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mi][ni][r] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      const uint16_t* a0 = qs + (mi * 16 + g) * QLD + kk * 16 + 2 * t;
      const uint16_t* a1 = a0 + 8 * QLD;
      uint32_t af[4];
      af[0] = *reinterpret_cast<const uint32_t*>(a0);
      af[1] = *reinterpret_cast<const uint32_t*>(a1);
      af[2] = *reinterpret_cast<const uint32_t*>(a0 + 8);
      af[3] = *reinterpret_cast<const uint32_t*>(a1 + 8);
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) mma_bf16_16816(acc[mi][ni], af, bf[kk][ni]);
    }
  }

#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
    const int r0 = b0 + mi * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      const int col = n_base + ni * 8 + 2 * t;
      if (r0 < B)
        *reinterpret_cast<uint32_t*>(q_cat + ((size_t)r0 * H + h) * DK + col) =
            pack_bf16x2(acc[mi][ni][0], acc[mi][ni][1]);
      if (r1 < B)
        *reinterpret_cast<uint32_t*>(q_cat + ((size_t)r1 * H + h) * DK + col) =
            pack_bf16x2(acc[mi][ni][2], acc[mi][ni][3]);
    }
  }

  // q_pe rows of this block (first column quarter only): 64 rows x 8 vectors of 16 bytes
  if (quarter == 0) {
    for (int i = threadIdx.x; i < QROWS * 8; i += blockDim.x) {
      const int r = b0 + i / 8, v = i % 8;
      if (r < B)
        reinterpret_cast<uint4*>(q_cat + ((size_t)r * H + h) * DK + DC)[v] =
            reinterpret_cast<const uint4*>(q_pe + ((size_t)r * H + h) * DR)[v];
    }
  }
}

}  // namespace

cudaError_t launch_q_absorb(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* q_cat,
                            cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  q_absorb_kernel<<<dim3(H, 4, (B + QROWS - 1) / QROWS), 256, 0, s>>>(
      static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe), static_cast<const uint16_t*>(W_UK),
      H, B, static_cast<uint16_t*>(q_cat));
  return cudaGetLastError();
}

}  // namespace mla
