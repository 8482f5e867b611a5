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
#include "tc_ptx.cuh"

namespace mla {
namespace {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One CTA per head, 8 warps.  W_UK[h] (512 x 128 bf16, 128 KB) arrives by four
// 2-D TMA tiles of 256 rows x 64 dims (128B swizzle: conflict-free fragment
// reads) issued at entry, so it is read from HBM exactly once.  The batch is
// processed 64 rows at a time: the rows' q_nope are staged in padded rows, and
// warp w computes latent columns [64w, 64w+64) of all 64 rows.
constexpr int QROWS = 64;
constexpr int QLD = DN + 8;           // padded bf16 row stride (272 B) of the staged queries
constexpr uint32_t W_TILE = 256 * 128;  // 32 KB: 256 latent columns x 64 dims, 128B-swizzled

struct __align__(1024) QaSmem {
  uint8_t w[4][W_TILE];     // tile 2*dc + ch: dims [64dc, 64dc+64) of latent columns [256ch, 256ch+256)
  uint16_t q[QROWS * QLD];  // q_nope rows of the current pass
  uint64_t w_full;
};

__global__ void __launch_bounds__(256, 1) q_absorb_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                           const uint16_t* __restrict__ q_nope,
                                                           const uint16_t* __restrict__ q_pe, int H, int B,
                                                           uint16_t* __restrict__ q_cat) {
  extern __shared__ uint8_t smem_raw[];
  QaSmem& S = *reinterpret_cast<QaSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int h = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n_base = warp * 64;

  if (tid == 0) {
    mbar_init(&S.w_full, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&S.w_full, 4 * W_TILE);
    for (int dc = 0; dc < 2; ++dc)
      for (int ch = 0; ch < 2; ++ch) tc::tma_load_3d(S.w[2 * dc + ch], &tm_w, 64 * dc, 256 * ch, h, &S.w_full);
  }
  // fragment W_UK[h][c][k .. k+1] from the swizzled tiles (k even)
  auto wfrag = [&](int c, int k) -> uint32_t {
    const int kb = (k & 63) * 2, r = c & 255;
    return *reinterpret_cast<const uint32_t*>(S.w[2 * (k >> 6) + (c >> 8)] + r * 128 + ((((kb >> 4) ^ (r & 7))) << 4) +
                                              (kb & 15));
  };

  bool w_ready = false;
  for (int b0 = 0; b0 < B; b0 += QROWS) {
    for (int i = tid; i < QROWS * (DN / 8); i += blockDim.x) {
      const int r = i / (DN / 8), v = i % (DN / 8);
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (b0 + r < B) x = __ldg(reinterpret_cast<const uint4*>(q_nope + ((size_t)(b0 + r) * H + h) * DN) + v);
      *reinterpret_cast<uint4*>(S.q + r * QLD + v * 8) = x;
    }
    // q_pe rows of this pass: 64 rows x 8 vectors of 16 bytes
    for (int i = tid; i < QROWS * 8; i += blockDim.x) {
      const int r = b0 + i / 8, v = i % 8;
      if (r < B)
        reinterpret_cast<uint4*>(q_cat + ((size_t)r * H + h) * DK + DC)[v] =
            __ldg(reinterpret_cast<const uint4*>(q_pe + ((size_t)r * H + h) * DR) + v);
    }
    if (!w_ready) {
      (void)mbar_wait(&S.w_full, 0);  // bounded; the copies of a valid buffer always land
      w_ready = true;
    }
    __syncthreads();

    float acc[4][8][4];
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
      for (int ni = 0; ni < 8; ++ni)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mi][ni][r] = 0.f;
#pragma unroll 2
    for (int k0 = 0; k0 < DN; k0 += 16) {
      uint32_t bf[8][2];
#pragma unroll
      for (int ni = 0; ni < 8; ++ni) {
        const int c = n_base + ni * 8 + g;
        bf[ni][0] = wfrag(c, k0 + 2 * t);
        bf[ni][1] = wfrag(c, k0 + 8 + 2 * t);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const uint16_t* a0 = S.q + (mi * 16 + g) * QLD + k0 + 2 * t;
        const uint16_t* a1 = a0 + 8 * QLD;
        uint32_t af[4];
        af[0] = *reinterpret_cast<const uint32_t*>(a0);
        af[1] = *reinterpret_cast<const uint32_t*>(a1);
        af[2] = *reinterpret_cast<const uint32_t*>(a0 + 8);
        af[3] = *reinterpret_cast<const uint32_t*>(a1 + 8);
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
    __syncthreads();  // the staged rows are rewritten by the next pass
  }
  if (!w_ready) (void)mbar_wait(&S.w_full, 0);  // no pass ran: let the copies land before exit
}

}  // namespace

cudaError_t launch_q_absorb(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* q_cat,
                            cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  CUtensorMap tm_w;  // W_UK: (128 dims, 512 latent columns, H heads), tiles of 64 x 256, 128B swizzle
  if (!encode_3d(&tm_w, W_UK, DN, DC, H, DN * 2, (uint64_t)DC * DN * 2, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(QaSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(q_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  q_absorb_kernel<<<H, 256, smem, s>>>(tm_w, static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe),
                                       H, B, static_cast<uint16_t*>(q_cat));
  return cudaGetLastError();
}

}  // namespace mla
