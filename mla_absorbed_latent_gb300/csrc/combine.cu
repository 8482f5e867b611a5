// Merge of the split-KV partials and the value up-projection.
//
// Each split s of row b left O_s = (sum_{t in s} e^{x_t - m_s} c_t) / l_s and
// LSE_s = m_s + ln l_s per head.  The exact softmax over the whole row is
//   o_lat = sum_s e^{LSE_s - LSE} O_s,   LSE = ln sum_s e^{LSE_s}.
// Then "DeepSeek MLA 吸收式缓存" §2.3 (sum_t p_t W_UV c_t = W_UV sum_t p_t c_t)
// applies the value projection once per head: out[b,h,:] = W_UV[h] o_lat[b,h,:]
// ("手搓 MLA" §四, einsum("thc,hdc->thd", out_lat, W_UV)).
//
// Two kernels: the merge (one warp per row and head, bandwidth-bound) writes
// each row's fp32 o_lat into the partial slot of the row's first split; the
// up-projection (one CTA per head) stages W_UV[h] once and runs the GEMM
// (M = rows, N = 128, K = 512) on the warp-level bf16 tensor-core MMA with
// o_lat split into a bf16 high part and a bf16 residual, so the only rounding
// left is W_UV's own bf16 and the fp32 accumulation.
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int ROWS = 16;     // batch rows projected per pass
constexpr int LDA = DC + 4;  // padded fp32 row stride of the o_lat tile (2,064 B)
constexpr uint32_t W_CHUNK = DV * 64 * 2;  // 16 KB: W_UV[h] rows x 64 latent dims, 128B-swizzled

struct __align__(1024) UpSmem {
  uint8_t w[8][W_CHUNK];      // W_UV[h] in 8 TMA tiles of 64 latent dims (K)
  float a[2][ROWS * LDA];     // merged o_lat rows, double-buffered across passes
  uint64_t w_full, a_full[2];
};

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

// slot of the merged o_lat of row b (the partial slot of the row's first segment)
__device__ __forceinline__ size_t merged_slot(const int* prefix, long long T, long long W, int b) {
  return (size_t)(worker_of_tile(prefix[b], T, W) + b);
}

// ---- merge: one warp per (row, head).  Lane k reads the LSE of the row's
// k-th split (32 at a time), the weights e^{LSE_s - max} are formed once, and
// every split row is loaded before any is summed (4 float4 per lane per
// split), so a warp keeps all of its row's partial bytes in flight.  The
// merged o_lat overwrites the row's first partial slot (only this warp reads
// the row's partials of this head, and it has read them all by then).
__global__ void __launch_bounds__(256) merge_kernel(int H, int B, const int* __restrict__ plan,
                                                     float* __restrict__ part_o, const float* __restrict__ part_lse,
                                                     float* __restrict__ o_lat_out) {
  grid_dep_wait();  // the partials of the attend step
  grid_dep_launch();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= B * H) return;
  const int b = gw / H, h = gw % H;
  const long long T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (prefix[b + 1] <= prefix[b]) {  // empty row: o_lat = 0 (the up-projection reads no slot for it)
    if (o_lat_out != nullptr)
#pragma unroll
      for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(o_lat_out + ((size_t)b * H + h) * DC)[lane + 32 * i] = acc[i];
    return;
  }
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
    for (int k = 0; k < n; k += 4) {
      float ek[4];
      float4 v[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ek[j] = __shfl_sync(0xffffffffu, e, min(k + j, 31));
        if (k + j >= n) ek[j] = 0.f;
        const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)(w0 + k + j + b) * H + h) * DC);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[j][i] = ek[j] != 0.f ? src[lane + 32 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i].x = fmaf(ek[j], v[j][i].x, acc[i].x);
          acc[i].y = fmaf(ek[j], v[j][i].y, acc[i].y);
          acc[i].z = fmaf(ek[j], v[j][i].z, acc[i].z);
          acc[i].w = fmaf(ek[j], v[j][i].w, acc[i].w);
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
  __syncwarp();  // every lane's partial reads precede the in-place write
  float4* dst = reinterpret_cast<float4*>(part_o + ((size_t)(wf + b) * H + h) * DC);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dst[lane + 32 * i] = acc[i];
    if (o_lat_out != nullptr) reinterpret_cast<float4*>(o_lat_out + ((size_t)b * H + h) * DC)[lane + 32 * i] = acc[i];
  }
}

// ---- up-projection: one CTA per head.  W_UV[h] (128 KB) arrives by eight 2-D
// TMA tiles (128B swizzle: conflict-free fragment reads) issued at entry; the
// merged rows arrive 16 at a time by one bulk copy per row, the next pass's
// rows in flight while the current pass computes.
__global__ void __launch_bounds__(256, 1) upproj_kernel(const __grid_constant__ CUtensorMap tm_w, int H, int B,
                                                         const int* __restrict__ plan,
                                                         const float* __restrict__ part_o,
                                                         uint16_t* __restrict__ out) {
  extern __shared__ uint8_t smem_raw[];
  UpSmem& S = *reinterpret_cast<UpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int h = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  const int passes = (B + ROWS - 1) / ROWS;

  if (tid == 0) {
    mbar_init(&S.w_full, 1);
    mbar_init(&S.a_full[0], ROWS);
    mbar_init(&S.a_full[1], ROWS);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    // W_UV is read before the wait: this kernel always follows the merge
    // kernel, which itself waited for all earlier work
    mbar_arrive_expect_tx(&S.w_full, 8 * W_CHUNK);
    for (int kc = 0; kc < 8; ++kc) tc::tma_load_3d(S.w[kc], &tm_w, 64 * kc, 0, h, &S.w_full);
  }
  grid_dep_wait();  // the merged rows
  grid_dep_launch();
  // pass p's rows into buffer p & 1: thread r < 16 copies row b0 + r (zeros
  // for empty rows and rows past B) and arrives once
  auto issue_rows = [&](int p) {
    if (tid < ROWS) {
      const int b = p * ROWS + tid;
      float* dst = S.a[p & 1] + tid * LDA;
      uint64_t* bar = &S.a_full[p & 1];
      if (b < B && prefix[b + 1] > prefix[b]) {
        mbar_arrive_expect_tx(bar, DC * 4);
        bulk_g2s(dst, part_o + (merged_slot(prefix, T, W, b) * H + h) * DC, DC * 4, bar);
      } else {
        for (int v = 0; v < DC / 4; ++v) reinterpret_cast<float4*>(dst)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        mbar_arrive(bar);
      }
    }
  };
  if (passes > 0) issue_rows(0);

  const int g = lane >> 2, t = lane & 3;
  bool w_ready = false;
  // fragment of W_UV[h][n][k .. k+1] in the swizzled tiles (k even)
  auto wfrag = [&](int n, int k) -> uint32_t {
    const int kb = (k & 63) * 2;
    return *reinterpret_cast<const uint32_t*>(S.w[k >> 6] + n * 128 + ((((kb >> 4) ^ (n & 7))) << 4) + (kb & 15));
  };
  for (int p = 0; p < passes; ++p) {
    if (p + 1 < passes) issue_rows(p + 1);  // its buffer was released by the barrier ending pass p-1
    (void)mbar_wait(&S.a_full[p & 1], (uint32_t)(p >> 1) & 1u);  // bounded
    if (!w_ready) {
      (void)mbar_wait(&S.w_full, 0);
      w_ready = true;
    }
    __syncthreads();  // zero rows written with plain stores are visible too
    const float* A = S.a[p & 1];
    float d[2][4];
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int k = 0; k < 4; ++k) d[ni][k] = 0.f;
#pragma unroll 4
    for (int k0 = 0; k0 < DC; k0 += 16) {
      const float* a0 = A + g * LDA + k0 + 2 * t;
      const float* a1 = a0 + 8 * LDA;
      uint32_t ah[4], al[4];
      split2(*reinterpret_cast<const float2*>(a0), ah[0], al[0]);
      split2(*reinterpret_cast<const float2*>(a1), ah[1], al[1]);
      split2(*reinterpret_cast<const float2*>(a0 + 8), ah[2], al[2]);
      split2(*reinterpret_cast<const float2*>(a1 + 8), ah[3], al[3]);
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        const int n = warp * 16 + ni * 8 + g;
        const uint32_t bf[2] = {wfrag(n, k0 + 2 * t), wfrag(n, k0 + 8 + 2 * t)};
        mma_bf16_16816(d[ni], ah, bf);
        mma_bf16_16816(d[ni], al, bf);
      }
    }
    const int r0 = p * ROWS + g, r1 = r0 + 8;
#pragma unroll
    for (int ni = 0; ni < 2; ++ni) {
      const int col = warp * 16 + ni * 8 + 2 * t;
      if (r0 < B)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r0 * H + h) * DV + col) = pack_bf16x2(d[ni][0], d[ni][1]);
      if (r1 < B)
        *reinterpret_cast<uint32_t*>(out + ((size_t)r1 * H + h) * DV + col) = pack_bf16x2(d[ni][2], d[ni][3]);
    }
    __syncthreads();  // buffer p & 1 is refilled by pass p + 2
  }
  if (!w_ready) (void)mbar_wait(&S.w_full, 0);  // no pass ran: let the copies land before exit
}

}  // namespace

cudaError_t launch_combine(const void* W_UV, int H, int B, const int* plan, const float* part_o,
                           const float* part_lse, void* out, float* o_lat, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  float* po = const_cast<float*>(part_o);  // the merge writes each row's o_lat into its first partial slot
  cudaError_t e = launch_pdl(merge_kernel, dim3((B * H + 7) / 8), dim3(256), 0, s, H, B, plan, po, part_lse, o_lat);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_w;  // W_UV: (512 latent, 128 rows, H heads), tiles of 64 x 128, 128B swizzle
  if (!encode_3d(&tm_w, W_UV, DC, DV, H, DC * 2, (uint64_t)DV * DC * 2, 64, DV, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(UpSmem) + 1024;
  e = cudaFuncSetAttribute(upproj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(upproj_kernel, dim3(H), dim3(256), smem, s, tm_w, H, B, plan, static_cast<const float*>(po),
                    static_cast<uint16_t*>(out));
}

}  // namespace mla
