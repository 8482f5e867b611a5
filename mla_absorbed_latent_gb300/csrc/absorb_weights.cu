// Split of the latent up-projection wkv_b into the absorbed weights.
//
// "手搓 MLA:从 MHA 到 weight absorption" §三 splits the up-projected vector of
// every head into its no-RoPE key part and its value part; §四 then uses the
// key part on the query side (W_UK, absorbed into q) and the value part after
// the attention-weighted latent sum (W_UV).  Rows h*256 .. h*256+127 of wkv_b
// are head h's key projection, the next 128 its value projection.
//
// W_UK is stored transposed, [H][512][128] (d fastest), which is the K-major
// B operand of the per-head q-absorb GEMM; W_UV keeps [H][128][512] (c
// fastest), the K-major B operand of the up-projection.  Bit-exact copies.
#include "mla_common.cuh"

namespace mla {
namespace {

// W_UK[h][c][d] = wkv[h*256 + d][c]: 32x32 tile transpose through shared memory.
__global__ void __launch_bounds__(256) split_uk_kernel(const uint16_t* __restrict__ wkv,
                                                        uint16_t* __restrict__ wuk) {
  __shared__ uint16_t tile[32][33];
  const int h = blockIdx.z;
  const int c0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const uint16_t* src = wkv + (size_t)h * 256 * DC;
  for (int r = threadIdx.y; r < 32; r += 8)
    tile[r][threadIdx.x] = src[(size_t)(d0 + r) * DC + c0 + threadIdx.x];
  __syncthreads();
  uint16_t* dst = wuk + (size_t)h * DC * DN;
  for (int r = threadIdx.y; r < 32; r += 8)
    dst[(size_t)(c0 + r) * DN + d0 + threadIdx.x] = tile[threadIdx.x][r];
}

// W_UV[h][d][:] = wkv[h*256 + 128 + d][:], 16-byte vectors.
__global__ void split_uv_kernel(const uint4* __restrict__ wkv, uint4* __restrict__ wuv, int H) {
  const int per_row = DC * 2 / 16;  // 64 vectors per 512-wide bf16 row
  const size_t n = (size_t)H * DV * per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / per_row, col = i % per_row;
    const size_t h = row / DV, d = row % DV;
    wuv[i] = wkv[(h * 256 + DN + d) * per_row + col];
  }
}

}  // namespace

cudaError_t launch_absorb_weights(const void* wkv_b, int H, void* W_UK, void* W_UV, cudaStream_t s) {
  split_uk_kernel<<<dim3(DC / 32, DN / 32, H), dim3(32, 8), 0, s>>>(
      static_cast<const uint16_t*>(wkv_b), static_cast<uint16_t*>(W_UK));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  split_uv_kernel<<<256, 256, 0, s>>>(static_cast<const uint4*>(wkv_b), static_cast<uint4*>(W_UV), H);
  return cudaGetLastError();
}

}  // namespace mla
