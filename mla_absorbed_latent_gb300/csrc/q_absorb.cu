// Query-side key absorption: q_lat[b,h,:] = W_UK[h]^T q_nope[b,h,:].
//
// "DeepSeek MLA 吸收式缓存" §2.2: q^T (W_UK c_t) = (W_UK^T q)^T c_t, so the
// key up-projection moves from every cached token onto the one query token;
// "手搓 MLA" §四 writes it as einsum("thd,hdc->thc", q_nope, W_UK).
//
// Per head this is a small GEMM, M = B rows, N = 512, K = 128, run on the
// fifth-generation tensor core: two CTAs per head, each computing one half of
// the 512 latent columns (so each reads half of W_UK[h] and two CTAs fit on
// an SM); q_nope rows (A) and the W_UK[h] half (B) arrive as K-major
// 128B-swizzled TMA tiles; 8 tcgen05.mma (M=128 rows, N=256, K=16) accumulate
// the 128 x 256 fp32 result in tensor memory; the epilogue rounds it once to
// bf16, the A operand of the score MMA.  The output row is the 576-wide query
// of the latent attention: q_lat followed by a copy of q_pe.
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int QROWS = 128;                // batch rows per pass (MMA M)
constexpr uint32_t W_TILE = 256 * 128;    // 32 KB: 256 latent columns x 64 dims, 128B-swizzled
constexpr uint32_t Q_TILE = QROWS * 128;  // 16 KB: 128 rows x 64 dims, 128B-swizzled

struct __align__(1024) QaSmem {
  uint8_t w[2][W_TILE];  // tile dc: dims [64dc, 64dc+64) of this CTA's latent columns [256nh, 256nh+256)
  uint8_t q[2][Q_TILE];  // q_nope rows of the pass, dims [64dc, 64dc+64)
  uint64_t w_full, q_full, mma_done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(128, 1) q_absorb_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                           const __grid_constant__ CUtensorMap tm_q,
                                                           const __grid_constant__ CUtensorMap tm_qc,
                                                           const uint16_t* __restrict__ q_pe, int H, int B,
                                                           uint16_t* __restrict__ q_cat, int after_plan) {
  extern __shared__ uint8_t smem_raw[];
  QaSmem& S = *reinterpret_cast<QaSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int h = blockIdx.x, nh = blockIdx.y;  // head, half of the latent columns
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int passes = (B + QROWS - 1) / QROWS;

  if (tid == 0) {
    mbar_init(&S.w_full, 1);
    mbar_init(&S.q_full, 1);
    mbar_init(&S.mma_done, 1);
    fence_barrier_init();
  }
  // W_UK's tiles: inside a fused decode (after_plan) every write before the
  // plan kernel is complete once this grid runs, so they load at once; a
  // step-wise call may directly follow the kernel that wrote W_UK (a weight
  // split), so it loads them only after its wait
  auto load_w = [&]() {
    mbar_arrive_expect_tx(&S.w_full, 2 * W_TILE);
    for (int dc = 0; dc < 2; ++dc) tma_load_3d(S.w[dc], &tm_w, 64 * dc, 256 * nh, h, &S.w_full);
  };
  if (after_plan && tid == 0) load_w();
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // The queries, and the readers of q_cat in the step before, come from work
  // before the kernel ahead of this one.  When that kernel is the plan kernel
  // of the same decode (after_plan), which waits for its own predecessor before
  // it lets this grid start, they are complete already: this grid then runs
  // beside the plan kernel and waits for it only before it exits (so that its
  // completion still implies the plan's, which the later kernels rely on).
  if (!after_plan) {
    grid_dep_wait();
    if (tid == 0) load_w();
  }
  grid_dep_launch();
  const uint32_t tmem = S.tmem_base;
  const uint32_t idesc = idesc_bf16_f32(128, 256, false, false);

  for (int p = 0; p < passes; ++p) {
    const int b0 = p * QROWS;
    if (tid == 0) {
      // rows past B read as zeros (out-of-bounds fill)
      mbar_arrive_expect_tx(&S.q_full, 2 * Q_TILE);
      for (int dc = 0; dc < 2; ++dc) tma_load_3d(S.q[dc], &tm_q, 64 * dc, h, b0, &S.q_full);
      bool ok = mbar_wait(&S.q_full, (uint32_t)p & 1u);
      if (p == 0) ok = mbar_wait(&S.w_full, 0) && ok;
      if (ok) {
        fence_after_sync();
        for (int dc = 0; dc < 2; ++dc) {
          const uint64_t ad = smem_desc(smem_u32(S.q[dc]), 16, 1024, SWIZZLE_128B);
          const uint64_t bd = smem_desc(smem_u32(S.w[dc]), 16, 1024, SWIZZLE_128B);
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc,
                   (dc | kk) != 0 ? 1u : 0u);
        }
      }
      mma_commit(&S.mma_done);  // arrives even if nothing was issued
    }
    // q_pe rows of this pass, while the MMAs run (each CTA of the head half of them)
    for (int i = tid + nh * (QROWS * 4); i < (nh + 1) * (QROWS * 4); i += blockDim.x) {
      const int r = b0 + i / 8, v = i % 8;
      if (r < B)
        reinterpret_cast<uint4*>(q_cat + ((size_t)r * H + h) * DK + DC)[v] =
            __ldg(reinterpret_cast<const uint4*>(q_pe + ((size_t)r * H + h) * DR) + v);
    }
    (void)mbar_wait(&S.mma_done, (uint32_t)p & 1u);
    __syncwarp();
    fence_after_sync();
    // epilogue: warp w owns TMEM lanes (rows) 32w..32w+31.  Each 128-column
    // round goes TMEM -> bf16 in a 128B-swizzled staging tile (this warp's 8 KB
    // of the q tiles, free now that the MMAs have read them) -> two TMA stores
    // (rows past B are clipped by the tensor map)
    const int r0 = b0 + warp * 32;
    if (r0 < B) {
      uint8_t* stg = &S.q[0][0] + warp * 8192;
      for (int rd = 0; rd < 2; ++rd) {  // this CTA's 256 latent columns, 128 per round
        if (rd > 0 && lane == 0) bulk_wait_read_all();  // the last round's stores have read the tile
        __syncwarp();
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int c32 = 0; c32 < 2; ++c32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 128 * rd + 64 * half + 32 * c32, v);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int chunk = 4 * c32 + k;  // 16-byte unit of the 128-byte row
              *reinterpret_cast<uint4*>(stg + half * 4096 + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                             pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                             pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                             pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
            }
          }
        fence_proxy_async_smem();  // generic writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_qc, stg, 256 * nh + 128 * rd, h, r0);
          tma_store_3d(&tm_qc, stg + 4096, 256 * nh + 128 * rd + 64, h, r0);
          bulk_commit_group();
        }
      }
      if (lane == 0) bulk_wait_all();  // the staging tile is the next pass's q tile; stores complete before exit
    }
    fence_before_sync();
    __syncthreads();  // TMEM and the q tiles are rewritten by the next pass
    fence_after_sync();
  }
  if (passes == 0 && tid == 0) (void)mbar_wait(&S.w_full, 0);  // let the weight copies land before exit
  if (after_plan) grid_dep_wait();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_q_absorb(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* q_cat,
                            bool after_plan, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  CUtensorMap tm_w, tm_q;
  // W_UK: (128 dims, 512 latent columns, H heads), tiles of 64 x 256; q_nope: (128 dims, H, B), tiles of 64 x 1 x 128
  if (!encode_3d(&tm_w, W_UK, DN, DC, H, DN * 2, (uint64_t)DC * DN * 2, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_3d_box(&tm_q, q_nope, DN, H, B, DN * 2, (uint64_t)H * DN * 2, 64, 1, QROWS, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  CUtensorMap tm_qc;  // q_cat: (576 dims, H, B), stores of 64 dims x 1 head x 32 rows
  if (!encode_3d_box(&tm_qc, q_cat, DK, H, B, DK * 2, (uint64_t)H * DK * 2, 64, 1, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(QaSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(q_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(q_absorb_kernel, dim3(H, 2), dim3(128), smem, s, tm_w, tm_q, tm_qc, static_cast<const uint16_t*>(q_pe), H,
                    B, static_cast<uint16_t*>(q_cat), after_plan ? 1 : 0);
}

}  // namespace mla
