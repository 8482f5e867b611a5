// Merge of the split-KV partials and the value up-projection.
//
// Each split s of row b left O_s = (sum_{t in s} e^{x_t - m_s} c_t) / l_s and
// LSE_s = m_s + ln l_s per head.  The exact softmax over the whole row is
//   o_lat = sum_s e^{LSE_s - LSE} O_s,   LSE = ln sum_s e^{LSE_s}.
// Then "DeepSeek MLA 吸收式缓存" §2.3 (sum_t p_t W_UV c_t = W_UV sum_t p_t c_t)
// applies the value projection once per head: out[b,h,:] = W_UV[h] o_lat[b,h,:]
// ("手搓 MLA" §四, einsum("thc,hdc->thd", out_lat, W_UV)).
//
// One CTA per (head, 16 rows).  The merged o_lat tile stays in shared memory
// in fp32; the GEMM (M = rows, N = 128, K = 512) runs on the warp-level bf16
// tensor-core MMA with o_lat split into a bf16 high part and a bf16 residual,
// so the only rounding left is W_UV's own bf16 and the fp32 accumulation.
#include "mla_common.cuh"

namespace mla {
namespace {

constexpr int ROWS = 16;  // batch rows per CTA (grid = heads x row blocks)
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

  // W_UV fragments of this warp's output columns [16w, 16w+16) for the first
  // K block; issued before the merge so that their latency overlaps it
  const int g = lane >> 2, t = lane & 3;
  const uint16_t* wv = w_uv + (size_t)h * DV * DC;
  constexpr int KB = 8;  // k-steps of 16 fetched together
  uint32_t bf[KB][2][2];
  auto fetch_b = [&](int k0) {
#pragma unroll
    for (int kk = 0; kk < KB; ++kk)
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        const uint16_t* row = wv + (size_t)(warp * 16 + ni * 8 + g) * DC + k0 + kk * 16 + 2 * t;
        bf[kk][ni][0] = __ldg(reinterpret_cast<const unsigned int*>(row));
        bf[kk][ni][1] = __ldg(reinterpret_cast<const unsigned int*>(row + 8));
      }
  };
  fetch_b(0);

  // ---- merge: warp w handles rows 2w, 2w+1; lane owns 4 float4 of the row.
  // The row's split LSEs are read 32 at a time (one per lane), the weights
  // e^{LSE_s - max} formed once, then the partial rows summed two at a time.
  for (int r = warp * (ROWS / 8); r < (warp + 1) * (ROWS / 8); ++r) {
    const int b = b0 + r;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b < B && prefix[b + 1] > prefix[b]) {
      const int wf = worker_of_tile(prefix[b], T, W);
      const int wl = worker_of_tile(prefix[b + 1] - 1, T, W);
      auto lse_of = [&](int w) -> float {  // -inf for a worker without tiles
        if (w > wl || worker_begin(w, T, W) == worker_begin(w + 1, T, W)) return -INFINITY;
        return part_lse[(size_t)(w + b) * H + h];
      };
      float mx = -INFINITY;
      for (int w = wf; w <= wl; w += 32) mx = fmaxf(mx, lse_of(w + lane));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float den = 0.f;
      for (int w0 = wf; w0 <= wl; w0 += 32) {
        const float lw = lse_of(w0 + lane);
        const float e = lw == -INFINITY ? 0.f : expf(lw - mx);
        den += e;
        const int n = min(32, wl - w0 + 1);
        int k = 0;
        for (; k + 1 < n; k += 2) {
          const float e0 = __shfl_sync(0xffffffffu, e, k), e1 = __shfl_sync(0xffffffffu, e, k + 1);
          const float4* s0 = reinterpret_cast<const float4*>(part_o + ((size_t)(w0 + k + b) * H + h) * DC);
          const float4* s1 = reinterpret_cast<const float4*>(part_o + ((size_t)(w0 + k + 1 + b) * H + h) * DC);
          float4 v0[4], v1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v0[i] = e0 != 0.f ? s0[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
            v1[i] = e1 != 0.f ? s1[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[i].x = fmaf(e0, v0[i].x, fmaf(e1, v1[i].x, acc[i].x));
            acc[i].y = fmaf(e0, v0[i].y, fmaf(e1, v1[i].y, acc[i].y));
            acc[i].z = fmaf(e0, v0[i].z, fmaf(e1, v1[i].z, acc[i].z));
            acc[i].w = fmaf(e0, v0[i].w, fmaf(e1, v1[i].w, acc[i].w));
          }
        }
        if (k < n) {
          const float e0 = __shfl_sync(0xffffffffu, e, k);
          if (e0 != 0.f) {
            const float4* s0 = reinterpret_cast<const float4*>(part_o + ((size_t)(w0 + k + b) * H + h) * DC);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 v = s0[lane + 32 * i];
              acc[i].x = fmaf(e0, v.x, acc[i].x);
              acc[i].y = fmaf(e0, v.y, acc[i].y);
              acc[i].z = fmaf(e0, v.z, acc[i].z);
              acc[i].w = fmaf(e0, v.w, acc[i].w);
            }
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
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

  // ---- up-projection, M = 16 rows: warp w owns output columns [16w, 16w+16)
  float d[2][4];
#pragma unroll
  for (int ni = 0; ni < 2; ++ni)
#pragma unroll
    for (int k = 0; k < 4; ++k) d[ni][k] = 0.f;
#pragma unroll 1
  for (int k0 = 0; k0 < DC; k0 += 16 * KB) {
    uint32_t cur[KB][2][2];
#pragma unroll
    for (int kk = 0; kk < KB; ++kk)
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        cur[kk][ni][0] = bf[kk][ni][0];
        cur[kk][ni][1] = bf[kk][ni][1];
      }
    if (k0 + 16 * KB < DC) fetch_b(k0 + 16 * KB);
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      const float* a0 = A + g * LDA + k0 + kk * 16 + 2 * t;
      const float* a1 = a0 + 8 * LDA;
      uint32_t ah[4], al[4];
      split2(*reinterpret_cast<const float2*>(a0), ah[0], al[0]);
      split2(*reinterpret_cast<const float2*>(a1), ah[1], al[1]);
      split2(*reinterpret_cast<const float2*>(a0 + 8), ah[2], al[2]);
      split2(*reinterpret_cast<const float2*>(a1 + 8), ah[3], al[3]);
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        mma_bf16_16816(d[ni], ah, cur[kk][ni]);
        mma_bf16_16816(d[ni], al, cur[kk][ni]);
      }
    }
  }
  const int r0 = b0 + g, r1 = r0 + 8;
#pragma unroll
  for (int ni = 0; ni < 2; ++ni) {
    const int col = warp * 16 + ni * 8 + 2 * t;
    if (r0 < B)
      *reinterpret_cast<uint32_t*>(out + ((size_t)r0 * H + h) * DV + col) = pack_bf16x2(d[ni][0], d[ni][1]);
    if (r1 < B)
      *reinterpret_cast<uint32_t*>(out + ((size_t)r1 * H + h) * DV + col) = pack_bf16x2(d[ni][2], d[ni][3]);
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
