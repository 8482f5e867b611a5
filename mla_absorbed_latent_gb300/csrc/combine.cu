// Merge of the split-KV partials and the value up-projection.
//
// Each split s of row b left O_s = (sum_{t in s} e^{x_t - m_s} c_t) / l_s and
// LSE_s = m_s + ln l_s per head.  The exact softmax over the whole row is
//   o_lat = sum_s e^{LSE_s - LSE} O_s,   LSE = ln sum_s e^{LSE_s}.
// Then "DeepSeek MLA 吸收式缓存" §2.3 (sum_t p_t W_UV c_t = W_UV sum_t p_t c_t)
// applies the value projection once per head: out[b,h,:] = W_UV[h] o_lat[b,h,:]
// ("手搓 MLA" §四, einsum("thc,hdc->thd", out_lat, W_UV)).
//
// One CTA per (head, 64 rows).  The merged o_lat tile stays in shared memory
// in fp32; the GEMM (M = rows, N = 128, K = 512) runs on the warp-level bf16
// tensor-core MMA with o_lat split into a bf16 high part and a bf16 residual,
// so the only rounding left is W_UV's own bf16 and the fp32 accumulation.
#include "mla_common.cuh"

namespace mla {
namespace {

constexpr int ROWS = 64;
constexpr int LDA = DC + 4;  // padded fp32 row stride of the o_lat tile

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// split two fp32 values into packed bf16 high parts and packed bf16 residuals
__device__ __forceinline__ void split2(float2 v, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(v.x - hf.x, v.y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ w_uv, int H, int B,
                                                       const int* __restrict__ plan,
                                                       const float* __restrict__ part_o,
                                                       const float* __restrict__ part_lse,
                                                       uint16_t* __restrict__ out, float* __restrict__ o_lat_out) {
  extern __shared__ __align__(16) float A[];  // [ROWS][LDA]
  const int h = blockIdx.x, b0 = blockIdx.y * ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;

  // ---- merge: warp w handles rows w, w+8, ...; lane owns 4 float4 of the row
  for (int r = warp; r < ROWS; r += 8) {
    const int b = b0 + r;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b < B && prefix[b + 1] > prefix[b]) {
      const int wf = worker_of_tile(prefix[b], T, W);
      const int wl = worker_of_tile(prefix[b + 1] - 1, T, W);
      float mx = -INFINITY;
      for (int w = wf; w <= wl; ++w) {
        if (worker_begin(w, T, W) == worker_begin(w + 1, T, W)) continue;
        mx = fmaxf(mx, part_lse[(size_t)(w + b) * H + h]);
      }
      float den = 0.f;
      for (int w = wf; w <= wl; ++w) {
        if (worker_begin(w, T, W) == worker_begin(w + 1, T, W)) continue;
        const float e = expf(part_lse[(size_t)(w + b) * H + h] - mx);
        den += e;
        const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)(w + b) * H + h) * DC);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = src[lane + 32 * i];
          acc[i].x = fmaf(e, v.x, acc[i].x);
          acc[i].y = fmaf(e, v.y, acc[i].y);
          acc[i].z = fmaf(e, v.z, acc[i].z);
          acc[i].w = fmaf(e, v.w, acc[i].w);
        }
      }
      const float inv = 1.f / den;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i].x *= inv; acc[i].y *= inv; acc[i].z *= inv; acc[i].w *= inv;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      reinterpret_cast<float4*>(A + r * LDA)[lane + 32 * i] = acc[i];
      if (o_lat_out != nullptr && b < B)
        reinterpret_cast<float4*>(o_lat_out + ((size_t)b * H + h) * DC)[lane + 32 * i] = acc[i];
    }
  }
  __syncthreads();

  // ---- up-projection: warp w owns output columns [16w, 16w+16)
  const int g = lane >> 2, t = lane & 3;
  float d[4][2][4];
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int k = 0; k < 4; ++k) d[mi][ni][k] = 0.f;
  const uint16_t* wv = w_uv + (size_t)h * DV * DC;
#pragma unroll 2
  for (int k0 = 0; k0 < DC; k0 += 16) {
    uint32_t bf[2][2];
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      const uint16_t* row = wv + (size_t)(warp * 16 + ni * 8 + g) * DC + k0 + 2 * t;
      bf[ni][0] = *reinterpret_cast<const uint32_t*>(row);
      bf[ni][1] = *reinterpret_cast<const uint32_t*>(row + 8);
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
      const float* a0 = A + (mi * 16 + g) * LDA + k0 + 2 * t;
      const float* a1 = a0 + 8 * LDA;
      uint32_t ah[4], al[4];
      split2(*reinterpret_cast<const float2*>(a0), ah[0], al[0]);
      split2(*reinterpret_cast<const float2*>(a1), ah[1], al[1]);
      split2(*reinterpret_cast<const float2*>(a0 + 8), ah[2], al[2]);
      split2(*reinterpret_cast<const float2*>(a1 + 8), ah[3], al[3]);
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        mma_bf16_16816(d[mi][ni], ah, bf[ni]);
        mma_bf16_16816(d[mi][ni], al, bf[ni]);
      }
    }
  }
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
    const int r0 = b0 + mi * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      const int col = warp * 16 + ni * 8 + 2 * t;
      if (r0 < B)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r0 * H + h) * DV + col) = pack_bf16x2(d[mi][ni][0], d[mi][ni][1]);
      if (r1 < B)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r1 * H + h) * DV + col) = pack_bf16x2(d[mi][ni][2], d[mi][ni][3]);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const void* W_UV, int H, int B, const int* plan, const float* part_o,
                           const float* part_lse, void* out, float* o_lat, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const size_t smem = (size_t)ROWS * LDA * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  combine_kernel<<<dim3(H, (B + ROWS - 1) / ROWS), 256, smem, s>>>(static_cast<const uint16_t*>(W_UV), H, B, plan,
                                                                   part_o, part_lse, static_cast<uint16_t*>(out),
                                                                   o_lat);
  return cudaGetLastError();
}

}  // namespace mla
