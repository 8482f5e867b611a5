// The layer's output projection after the value up-projection:
//   y[r, :] = W_O . concat_h out[r, h, :]       (y = o @ Wo^T)
// "手搓 MLA" §三 and §四 end both the unabsorbed and the absorbed path with
// "@ Wo.T" on the heads' outputs side by side ([T, H*dv], head-major: the
// layout mla_decode writes); "DeepSeek MLA 吸收式缓存" §3.3 maps o_proj to wo.
// It sums over heads, so it cannot live inside the per-head merge; it runs as
// the next kernel of the chain, reading the merge's bf16 output directly, and
// its weight tiles load before it waits for that output.
//
// A GEMM on the fifth-generation tensor cores: one CTA per (128 output
// features, 64 rows, K split): D[128 features][64 rows] += W_O[:, k chunk] .
// o[:, k chunk]^T over 64-wide chunks of K = H*128 through a 4-stage ring of
// 128B-swizzled TMA tiles (the weight tile is A, the rows are B; both K-major).
// For a decode's few rows the weight stream binds (H*128 x hidden bf16) and K
// is split over several CTAs per tile so that every SM pulls it; the splits
// add into an fp32 workspace and the last one (a ticket per tile) writes y.
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int OP_M = 128, OP_N = 64, OP_ST = 4;
constexpr uint32_t OP_A = OP_M * 128, OP_B = OP_N * 128;  // bytes of one 64-wide K chunk of each operand

struct __align__(1024) OpSmem {
  uint8_t a[OP_ST][OP_A];
  uint8_t b[OP_ST][OP_B];
  uint64_t full[OP_ST], empty[OP_ST], done;
  uint32_t tmem_base;
  int abort_flag, last;
};

__device__ __noinline__ bool owait_slow(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 7) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort = 1;
        raise_error(err, MLA_ERR_TIMEOUT, 300 + where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool owait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return owait_slow(bar, parity, abort, err, where);
}

// blockIdx.x = feature tile * ksplit + split, blockIdx.y = row tile
__global__ void __launch_bounds__(128, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_o, int R,
                    int hidden, int chunks, int ksplit, uint16_t* __restrict__ y, float* __restrict__ acc,
                    int* __restrict__ tickets, int* err) {
  extern __shared__ uint8_t smem_raw[];
  OpSmem& S = *reinterpret_cast<OpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int ft = blockIdx.x / ksplit, split = blockIdx.x - ft * ksplit, rt = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c0 = (int)((long long)split * chunks / ksplit);
  const int nk = (int)((long long)(split + 1) * chunks / ksplit) - c0;
  const int f0 = ft * OP_M, r0 = rt * OP_N;

  if (tid == 0) {
    for (int s = 0; s < OP_ST; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.done, 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, OP_N);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort = &S.abort_flag;
  // every thread but the producer waits for the kernel before this one here
  // (the rows it wrote, the workspace cleared before this launch)
  if (!(warp == 0 && lane == 0)) grid_dep_wait();

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: the weight tiles of the first stages before the rows exist
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_o);
    const int pre = min(OP_ST, nk);
    for (int c = 0; c < pre; ++c) {
      mbar_arrive_expect_tx(&S.full[c], OP_A + OP_B);
      tma_load_3d(S.a[c], &tm_w, 64 * (c0 + c), f0, 0, &S.full[c]);
    }
    grid_dep_wait();  // the rows (the merge's output) come from the kernel before this one
    grid_dep_launch();
    for (int c = 0; c < pre; ++c) tma_load_3d(S.b[c], &tm_o, 64 * (c0 + c), r0, 0, &S.full[c]);
    int issued = pre;
    for (int c = pre; c < nk; ++c) {
      const int st = c % OP_ST;
      if (!owait(&S.empty[st], ((c / OP_ST) & 1) ^ 1, abort, err, 0)) break;
      mbar_arrive_expect_tx(&S.full[st], OP_A + OP_B);
      tma_load_3d(S.a[st], &tm_w, 64 * (c0 + c), f0, 0, &S.full[st]);
      tma_load_3d(S.b[st], &tm_o, 64 * (c0 + c), r0, 0, &S.full[st]);
      ++issued;
    }
    if (*abort)
      for (int k = max(0, issued - OP_ST); k < issued; ++k) (void)mbar_wait(&S.full[k % OP_ST], (k / OP_ST) & 1);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = idesc_bf16_f32(OP_M, OP_N, false, false);
    for (int c = 0; c < nk; ++c) {
      const int st = c % OP_ST;
      if (!owait(&S.full[st], (c / OP_ST) & 1, abort, err, 1)) break;
      fence_after_sync();
      const uint64_t ad = smem_desc(smem_u32(S.a[st]), 16, 1024, SWIZZLE_128B);
      const uint64_t bd = smem_desc(smem_u32(S.b[st]), 16, 1024, SWIZZLE_128B);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc, (c | kk) != 0 ? 1u : 0u);
      mma_commit(&S.empty[st]);
    }
    mma_commit(&S.done);
  }
  // ---- epilogue: thread j holds feature f0 + j of the tile's 64 rows
  const bool ok = owait(&S.done, 0, abort, err, 2);
  __syncwarp();
  fence_after_sync();
  const int f = f0 + tid;
  uint32_t v[OP_N];
  tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), v);
  tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32, v + 32);
  tmem_ld_wait();
  bool write = ok;
  if (ksplit > 1) {
    // add this split's partial into the tile's fp32 sums [feature][row], then
    // the last split of the tile writes y
    float* arow = acc + (size_t)f * (gridDim.y * OP_N) + r0;
    if (ok) {
#pragma unroll
      for (int q = 0; q < OP_N / 4; ++q)
        red_add_v4(arow + 4 * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) S.last = atomicAdd(tickets + ft * gridDim.y + rt, 1) == ksplit - 1 ? 1 : 0;
    __syncthreads();
    write = S.last != 0;
    if (write) {
      __threadfence();
      const float4* src = reinterpret_cast<const float4*>(arow);
#pragma unroll
      for (int q = 0; q < OP_N / 4; ++q) {
        const float4 x = __ldcg(src + q);
        v[4 * q] = __float_as_uint(x.x);
        v[4 * q + 1] = __float_as_uint(x.y);
        v[4 * q + 2] = __float_as_uint(x.z);
        v[4 * q + 3] = __float_as_uint(x.w);
      }
    }
  }
  if (write) {
    // y[r][f] bf16: for a fixed row the warp's 32 features are 64 contiguous bytes
#pragma unroll
    for (int k = 0; k < OP_N; ++k) {
      const int r = r0 + k;
      if (r < R) {
        const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[k]));
        y[(size_t)r * hidden + f] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, OP_N);
  }
}

}  // namespace

// K splits per (feature tile, row tile): as many CTAs as fit two per SM in
// one wave (rounding up would leave a short second wave), each at least 8
// chunks of K
int out_proj_splits(int R, int K, int hidden, int sms) {
  const long long tiles = (long long)(hidden / OP_M) * ((R + OP_N - 1) / OP_N);
  const int chunks = K / 64;
  const long long want = tiles > 0 ? (2LL * sms) / tiles : 1;
  long long k = want < chunks / 8 ? want : chunks / 8;
  return k > 1 ? (int)k : 1;
}

size_t out_proj_workspace_bytes(int R, int K, int hidden, int sms) {
  const int ks = out_proj_splits(R, K, hidden, sms);
  if (ks <= 1 || R <= 0) return 0;
  const size_t rpad = (size_t)((R + OP_N - 1) / OP_N) * OP_N;
  const size_t tiles = (size_t)(hidden / OP_M) * ((R + OP_N - 1) / OP_N);
  return align_up((size_t)hidden * rpad * 4, 256) + align_up(tiles * 4, 256);
}

cudaError_t launch_out_proj(const void* o, const void* W_O, int R, int K, int hidden, void* y, void* workspace,
                            int* err, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int ksplit = out_proj_splits(R, K, hidden, sms);
  CUtensorMap tm_w, tm_o;
  // W_O: (K, hidden) boxes of 64 x 128; rows: (K, R) boxes of 64 x 64 (rows past R read as zeros)
  if (!encode_3d(&tm_w, W_O, (uint64_t)K, (uint64_t)hidden, 1, (uint64_t)K * 2, (uint64_t)K * hidden * 2, 64, OP_M,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&tm_o, o, (uint64_t)K, (uint64_t)R, 1, (uint64_t)K * 2, (uint64_t)K * R * 2, 64, OP_N,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  float* acc = nullptr;
  int* tickets = nullptr;
  const int rtiles = (R + OP_N - 1) / OP_N;
  if (ksplit > 1) {
    const size_t acc_bytes = align_up((size_t)hidden * rtiles * OP_N * 4, 256);
    acc = static_cast<float*>(workspace);
    tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + acc_bytes);
    cudaError_t e = cudaMemsetAsync(workspace, 0, out_proj_workspace_bytes(R, K, hidden, sms), s);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = sizeof(OpSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(out_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(out_proj_kernel, dim3((hidden / OP_M) * ksplit, rtiles), dim3(128), smem, s, tm_w, tm_o, R, hidden,
                    K / 64, ksplit, static_cast<uint16_t*>(y), acc, tickets, err);
}

}  // namespace mla
