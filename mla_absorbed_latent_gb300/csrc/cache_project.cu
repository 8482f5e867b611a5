// Cache producer: the step before the append, fused with it.
//
// "手搓 MLA" §三 derives what the absorbed cache holds from each token's
// attention input x: c_kv = rmsnorm(x W_DKV^T, W_KVN) (512 wide) and
// k_pe = rope(x W_KR^T) (64 wide).  "DeepSeek MLA 吸收式缓存" §3.3 names the
// joint projection wkv_a (kv_a_proj_with_mqa: rows 0..511 are W_DKV, rows
// 512..575 W_KR) and the gain kv_norm.  Here the projection runs on the
// fifth-generation tensor cores and the epilogue finishes every token: the
// RMSNorm, the rotation, one bf16 rounding, then the page write of
// mla_cache_append (quantized per the pool's format, quant.cuh).
//
// Tiling.  A CTA pair (2-CTA cluster) owns a tile of 128 tokens; CTA r
// computes latent columns [256r, 256r+256) and RoPE-key columns
// [512+32r, 512+32r+32): M = 128 tokens, N = 256 + 32, K = hidden in 64-wide
// chunks through a 4-stage TMA ring (x tile 16 KB, weight tiles 32 + 4 KB, all
// 128B-swizzled, K-major).  The 288 fp32 accumulator columns fit in the CTA's
// tensor memory (the full 576 would not).  The RMSNorm needs both halves' sums
// of squares: the pair swaps its per-token sums (128 floats) through
// distributed shared memory.  A RoPE pair (2i, 2i+1) never straddles the two
// halves.
//
// Few tokens (decode appends one per row) would leave most SMs idle and read
// the 576 x hidden weight through two of them, so the hidden dimension is then
// split over `ksplit` CTA pairs per token tile: each stores its partial product
// (fp32) into its own slice of the caller's workspace, and project_finish_kernel
// (a CTA per token, chained by programmatic dependent launch) sums the slices in
// split order and runs the same epilogue: deterministic, and the epilogue of
// the few tokens spread over as many SMs.
//
// Thread roles (128 threads): lane 0 of warp 0 issues the TMA loads, lane 0 of
// warp 1 the MMAs; then all four warps run the epilogue, warp w on the tokens
// of TMEM lanes 32w..32w+31 (one token per thread).  Every mbarrier wait is
// bounded; a timeout is recorded as MLA_ERR_TIMEOUT.
#include <cmath>

#include "quant.cuh"
#include "tc_ptx.cuh"
#include "warp_mma.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int PJ_ROWS = 128;                  // tokens per tile (MMA M)
constexpr int PJ_STAGES = 4;
constexpr int PJ_THREADS = 128;
constexpr int PJ_HALF = DC / 2;               // latent columns per CTA
constexpr int PJ_ROPE = DR / 2;               // RoPE-key columns per CTA
constexpr uint32_t PJ_X_TILE = PJ_ROWS * 128;   // 16 KB: 128 tokens x 64 hidden
constexpr uint32_t PJ_WC_TILE = PJ_HALF * 128;  // 32 KB: 256 latent rows of wkv_a x 64 hidden
constexpr uint32_t PJ_WR_TILE = PJ_ROPE * 128;  // 4 KB: 32 RoPE-key rows x 64 hidden
constexpr uint32_t PJ_STAGE_BYTES = PJ_X_TILE + PJ_WC_TILE + PJ_WR_TILE;
constexpr uint32_t PJ_TMEM_COLS = 512;        // 288 used: latent half at 0, RoPE key at 256

// The RoPE rotation frequencies theta^(-2i/64), i = 0..31, as fixed-point phase
// increments: turn[i] = theta^(-2i/64) / (2 pi) in units of 2^-64 turn.
struct RopeFreq {
  uint64_t turn[DR / 2];
};

struct __align__(1024) PjSmem {
  uint8_t x[PJ_STAGES][PJ_X_TILE];
  uint8_t wc[PJ_STAGES][PJ_WC_TILE];
  uint8_t wr[PJ_STAGES][PJ_WR_TILE];
  float gamma[PJ_HALF];  // kv_norm gain of this CTA's latent columns
  float ss[PJ_ROWS];     // per-token sum of squares of this CTA's latent columns (read by the peer)
  uint64_t turn[PJ_ROPE / 2];  // phase increments of this CTA's 16 RoPE pairs (RopeFreq)
  uint64_t full[PJ_STAGES], empty[PJ_STAGES], mma_done;
  uint32_t tmem_base;
  int last;      // split mode: this pair runs the epilogue of its tile
  int issued;    // chunks whose loads the producer issued
  int consumed;  // chunks whose loads the MMA issuer saw land
};

__device__ __forceinline__ float bf16r(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// sin and cos of the angle pos * theta^(-2i/64), reduced to one turn as the
// phase accumulator of direct digital synthesis does: the wrapping 64-bit
// product pos * turn is the angle modulo one turn in units of 2^-64 turn
// (exact up to the rounding of turn, under pos * 2^-55 turn), its top 32 bits
// read as a signed number are the angle in [-pi, pi) in units of 2 pi / 2^32,
// and sincosf takes it from there.  No floating-point product of pos and the
// frequency is formed, so the reduction is as good at position 2^31 as at 0.
__device__ __forceinline__ void rope_sincos(long long pos, uint64_t turn, float* s, float* c) {
  const uint64_t ph = (uint64_t)pos * turn;
  const int32_t hi = (int32_t)(uint32_t)(ph >> 32);
  sincosf((float)hi * 1.46291807926715968e-09f, s, c);  // 2 pi / 2^32
}

__device__ __forceinline__ void store_bf16x32(uint8_t* dst, const float* y) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d[q] = make_uint4(pack_bf16x2(y[8 * q], y[8 * q + 1]), pack_bf16x2(y[8 * q + 2], y[8 * q + 3]),
                      pack_bf16x2(y[8 * q + 4], y[8 * q + 5]), pack_bf16x2(y[8 * q + 6], y[8 * q + 7]));
}

// Quantized page write of 32 finished (bf16-representable) values of one token
// (out of line: one copy of the quantizer code, called once per 32-value group).
// `col` is the position of y[0] in the 576-wide payload (a multiple of 32).
template <int FMT>
__device__ __noinline__ void write_quantized32(const float* y, int col, uint8_t* page, int slot) {
  if (col < DC) {
    const int g = col / 32;
    if (FMT == MLA_FMT_INT8) {
      int8_t code[32];
      const uint16_t sb = quant_i8<32>(y, code);
#pragma unroll
      for (int i = 0; i < 4; ++i) store_i8x8(page + I8_C_CODE + slot * DC + col + 8 * i, code + 8 * i);
      reinterpret_cast<uint16_t*>(page + I8_C_SCALE)[slot * 16 + g] = sb;
    } else {
      uint32_t w[4];
      uint16_t sb, zb;
      quant_i4_32(y, w, &sb, &zb);
      *reinterpret_cast<uint4*>(page + I4_C_CODE + slot * (DC / 2) + col / 2) = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint16_t*>(page + I4_C_SCALE)[slot * 16 + g] = sb;
      reinterpret_cast<uint16_t*>(page + I4_C_ZERO)[slot * 16 + g] = zb;
    }
    return;
  }
  // RoPE key: INT8 in groups of 8 dims in both quantized formats
  constexpr int pe_code_off = FMT == MLA_FMT_INT8 ? I8_PE_CODE : I4_PE_CODE;
  constexpr int pe_scale_off = FMT == MLA_FMT_INT8 ? I8_PE_SCALE : I4_PE_SCALE;
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    const int d = col - DC + 8 * q;  // first RoPE dim of the group
    int8_t code[8];
    const uint16_t sb = quant_i8<8>(y + 8 * q, code);
    store_i8x8(page + pe_code_off + slot * DR + d, code);
    reinterpret_cast<uint16_t*>(page + pe_scale_off)[slot * 8 + d / 8] = sb;
  }
}

// Writes 32 finished values of one token: to the optional bf16 payload row and,
// when `page` is not null, to the token's slot in the pool.
template <int FMT>
__device__ __forceinline__ void write_group32(const float* y, int col, uint8_t* page, int slot,
                                              uint8_t* latent_row) {
  if (latent_row != nullptr) store_bf16x32(latent_row + col * 2, y);
  if (page == nullptr) return;
  if (FMT == MLA_FMT_BF16)
    store_bf16x32(page + (size_t)slot * DK * 2 + col * 2, y);
  else
    write_quantized32<FMT>(y, col, page, slot);
}

template <int FMT>
__global__ void __launch_bounds__(PJ_THREADS, 1)
    project_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wc,
                   const __grid_constant__ CUtensorMap tm_wr, const uint16_t* __restrict__ kv_norm_w, float eps,
                   const RopeFreq freq, int num_pages, uint8_t* __restrict__ pages,
                   const int32_t* __restrict__ page_table, int max_pages, const int32_t* __restrict__ pos, int T,
                   int ntok, int chunks, int ksplit, uint16_t* __restrict__ latent_out, float* __restrict__ acc,
                   int* err) {
  extern __shared__ uint8_t smem_raw[];
  PjSmem& S = *reinterpret_cast<PjSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_launch();  // a split projection's finishing kernel may start its prologue (it waits for this grid)
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int mt = pair / ksplit, split = pair - mt * ksplit;
  const int tok0 = mt * PJ_ROWS;
  const int c_begin = (int)((long long)split * chunks / ksplit);
  const int nk = (int)((long long)(split + 1) * chunks / ksplit) - c_begin;

  if (tid == 0) {
    for (int s = 0; s < PJ_STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.mma_done, 1);
    S.issued = 0;
    S.consumed = 0;
    S.last = 0;
    fence_barrier_init();
  }
  for (int i = tid; i < PJ_HALF; i += PJ_THREADS)
    S.gamma[i] = __uint_as_float((uint32_t)kv_norm_w[PJ_HALF * rank + i] << 16);
  if (tid < PJ_ROPE / 2) S.turn[tid] = rank == 0 ? freq.turn[tid] : freq.turn[PJ_ROPE / 2 + tid];
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, PJ_TMEM_COLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0 && lane == 0) {
    // TMA producer
    const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % PJ_STAGES;
      if (i >= PJ_STAGES && !mbar_wait(&S.empty[s], (uint32_t)((i / PJ_STAGES) - 1) & 1u)) {
        raise_error(err, MLA_ERR_TIMEOUT, 20);
        break;
      }
      const int k = (c_begin + i) * 64;
      mbar_arrive_expect_tx(&S.full[s], PJ_STAGE_BYTES);
      tma_load_3d_hint(S.x[s], &tm_x, k, tok0, 0, &S.full[s], pol_x);  // token rows past ntok read as zeros
      tma_load_3d_hint(S.wc[s], &tm_wc, k, PJ_HALF * rank, 0, &S.full[s], pol_w);
      tma_load_3d_hint(S.wr[s], &tm_wr, k, DC + PJ_ROPE * rank, 0, &S.full[s], pol_w);
    }
    S.issued = i;
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: D_lat[128 x 256] (+)= X . Wc^T, D_rope[128 x 32] (+)= X . Wr^T
    const uint32_t id_c = idesc_bf16_f32(PJ_ROWS, PJ_HALF, false, false);
    const uint32_t id_r = idesc_bf16_f32(PJ_ROWS, PJ_ROPE, false, false);
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % PJ_STAGES;
      if (!mbar_wait(&S.full[s], (uint32_t)(i / PJ_STAGES) & 1u)) {
        raise_error(err, MLA_ERR_TIMEOUT, 21);
        break;
      }
      fence_after_sync();
      const uint64_t ad = smem_desc(smem_u32(S.x[s]), 16, 1024, SWIZZLE_128B);
      const uint64_t bc = smem_desc(smem_u32(S.wc[s]), 16, 1024, SWIZZLE_128B);
      const uint64_t br = smem_desc(smem_u32(S.wr[s]), 16, 1024, SWIZZLE_128B);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // K = 16 per MMA: 32 bytes further along the swizzled row
        const uint32_t accum = (i | kk) != 0 ? 1u : 0u;
        mma_ss(tmem, ad + (uint64_t)(kk * 2), bc + (uint64_t)(kk * 2), id_c, accum);
        mma_ss(tmem + PJ_HALF, ad + (uint64_t)(kk * 2), br + (uint64_t)(kk * 2), id_r, accum);
      }
      mma_commit(&S.empty[s]);  // the stage is free once these MMAs have read it
    }
    S.consumed = i;
    mma_commit(&S.mma_done);  // arrives once every MMA issued above has completed
  }
  __syncwarp();
  if (!mbar_wait(&S.mma_done, 0)) raise_error(err, MLA_ERR_TIMEOUT, 22);
  __syncwarp();
  fence_after_sync();
  __syncthreads();  // S.issued / S.consumed are final
  if (warp == 0 && lane == 0) {
    // loads issued but never seen landing (only after a timeout): let them land before exit
    for (int i = S.consumed; i < S.issued; ++i)
      if (!mbar_wait(&S.full[i % PJ_STAGES], (uint32_t)(i / PJ_STAGES) & 1u)) break;
  }

  const int row = warp * 32 + lane;
  const int tok = tok0 + row;
  const bool live = tok < ntok;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);

  bool run = true;
  if (ksplit > 1) {
    // this pair's partial product into its own slice of the workspace, live
    // token rows only; project_finish_kernel sums the slices in split order and
    // runs the epilogue, a CTA per token
    float* prow = acc + ((size_t)split * ntok + (live ? tok : 0)) * DK;
#pragma unroll 1
    for (int cc = 0; cc < 9; ++cc) {
      uint32_t v[32];
      tmem_ld32(trow + 32 * cc, v);  // warp-wide: every lane loads
      tmem_ld_wait();
      if (live) {
        const int col = cc < 8 ? PJ_HALF * rank + 32 * cc : DC + PJ_ROPE * rank;
        float4* dst = reinterpret_cast<float4*>(prow + col);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                               __uint_as_float(v[4 * q + 3]));
      }
    }
    run = false;
  }

  if (run) {
    // the token's slot in the pool (and the position its key is rotated by)
    uint8_t* page = nullptr;
    int slot = 0;
    long long p = 0;
    if (live) {
      const int b = tok / T, t = tok - b * T;
      const int p0 = pos[b];
      p = (long long)p0 + t;
      if (p0 < 0 || p >= (long long)max_pages * PAGE) {
        raise_error(err, MLA_ERR_BOUNDS, b);
      } else {
        const int phys = page_table[(size_t)b * max_pages + (int)(p / PAGE)];
        if (phys < 0 || phys >= num_pages) {
          raise_error(err, MLA_ERR_BOUNDS, phys);
        } else {
          constexpr size_t pb = FMT == MLA_FMT_BF16   ? PAGE_BYTES_BF16
                                : FMT == MLA_FMT_INT8 ? PAGE_BYTES_INT8
                                                      : PAGE_BYTES_INT4;
          page = pages + (size_t)phys * pb;
          slot = (int)(p % PAGE);
        }
      }
    }
    uint8_t* lrow = (live && latent_out != nullptr) ? reinterpret_cast<uint8_t*>(latent_out + (size_t)tok * DK)
                                                    : nullptr;

    // RMSNorm: sum of squares over this CTA's 256 columns, plus the peer's
    float ss = 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t v[32];
      tmem_ld32(trow + 32 * cc, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a = __uint_as_float(v[j]);
        ss = fmaf(a, a, ss);
      }
    }
    S.ss[row] = ss;
    cluster_sync();
    const float tot = ss + ld_cluster_f32(mapa(smem_u32(&S.ss[row]), (uint32_t)rank ^ 1u));
    const float rinv = rsqrtf(tot * (1.0f / DC) + eps);

#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t v[32];
      tmem_ld32(trow + 32 * cc, v);
      tmem_ld_wait();
      if (live) {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = bf16r(__uint_as_float(v[j]) * rinv * S.gamma[32 * cc + j]);
        write_group32<FMT>(y, PJ_HALF * rank + 32 * cc, page, slot, lrow);
      }
    }
    {
      // cos and sin of this token's 16 rotation angles, one at a time (a rolled
      // loop keeps one copy of that code), into the first x stage of the ring,
      // free now that every MMA has completed: [pair][token] float2
      float2* rot = reinterpret_cast<float2*>(S.x[0]);
#pragma unroll 1
      for (int i = 0; i < PJ_ROPE / 2; ++i) {
        float sn, cs;
        rope_sincos(p, S.turn[i], &sn, &cs);
        rot[i * PJ_ROWS + row] = make_float2(cs, sn);
      }
      uint32_t v[32];
      tmem_ld32(trow + PJ_HALF, v);
      tmem_ld_wait();
      if (live) {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float2 r = rot[(j / 2) * PJ_ROWS + row];
          const float a = __uint_as_float(v[j]), b = __uint_as_float(v[j + 1]);
          y[j] = bf16r(a * r.x - b * r.y);
          y[j + 1] = bf16r(a * r.y + b * r.x);
        }
        write_group32<FMT>(y, DC + PJ_ROPE * rank, page, slot, lrow);
      }
    }
  }

  fence_before_sync();
  cluster_sync();  // the peer has read S.ss; nothing touches TMEM any more
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, PJ_TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// At most 64 tokens (a decode-time append): the projection on the warp-level
// tensor-core instruction, without clusters or tensor memory.  One CTA per (64
// output columns, slice of the hidden dimension): its weight block [64
// columns][slice] and the tokens' block [64 tokens][slice] arrive by TMA
// (128B-swizzled 64 x 64 tiles, all at once), warp w multiplies tokens
// 16 (w % 4) .. + 15 by columns 32 (w / 4) .. + 31 with mma.sync m16n8k16, and
// the CTA stores its fp32 partial [tokens][64 columns] into its workspace
// slice; project_finish_kernel sums the slices and runs the epilogue.
// ---------------------------------------------------------------------------
constexpr int PS_TOK = 64;           // tokens (the MMA's M: 4 tiles of 16)
constexpr int PS_COLS = 64;          // output columns per CTA
constexpr int PS_NG = DK / PS_COLS;  // 9 column groups (the last: the RoPE key)
constexpr int PS_MAXCH = 8;          // 64-wide hidden chunks per CTA
constexpr uint32_t PS_TILE = 64 * 128;  // 8 KB: 64 rows of 64 bf16

struct __align__(1024) PsSmem {
  uint8_t w[PS_MAXCH][PS_TILE];
  uint8_t x[PS_MAXCH][PS_TILE];
  uint64_t full[PS_MAXCH];  // chunk i's weight and token tiles have landed
};

__global__ void __launch_bounds__(256) project_small_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                            const __grid_constant__ CUtensorMap tm_w, int ntok,
                                                            int chunks, int ksplit, float* __restrict__ acc,
                                                            int* err) {
  extern __shared__ uint8_t smem_raw[];
  PsSmem& S = *reinterpret_cast<PsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  grid_dep_launch();  // the finishing kernel may start its prologue (it waits for this grid)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cg = blockIdx.x, split = blockIdx.y;
  const int c_begin = (int)((long long)split * chunks / ksplit);
  const int nk = (int)((long long)(split + 1) * chunks / ksplit) - c_begin;  // 1..PS_MAXCH (host's choice)
  if (tid == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
    for (int i = 0; i < PS_MAXCH; ++i) mbar_init(&S.full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint64_t pol_w = policy_evict_first();  // the weight is read once per call
    for (int i = 0; i < nk; ++i) {
      const int k = (c_begin + i) * 64;
      mbar_arrive_expect_tx(&S.full[i], 2u * PS_TILE);
      tma_load_3d_hint(S.w[i], &tm_w, k, PS_COLS * cg, 0, &S.full[i], pol_w);
      tma_load_3d(S.x[i], &tm_x, k, 0, 0, &S.full[i]);  // token rows past ntok read as zeros
    }
  }
  const int mt = warp & 3, nh = warp >> 2;  // token tile, column half
  float d[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll 1
  for (int i = 0; i < nk; ++i) {
    if (!mbar_wait(&S.full[i], 0)) {  // bounded
      if (lane == 0) raise_error(err, MLA_ERR_TIMEOUT, 30);
      for (int j = i + 1; j < nk; ++j) mbar_wait(&S.full[j], 0);  // the later copies, again bounded
      return;
    }
    const uint32_t xb = smem_u32(S.x[i]), wb = smem_u32(S.w[i]);
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
      // A: tokens 16 mt + (lane % 16), dims 32 kp + 16 h + 8 (lane / 16) of k-step h;
      // B: columns 32 nh + 8 j + (lane % 8), dims 32 kp + 8 (lane / 8) (two k-steps)
      uint32_t a[2][4], b[4][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) ldsm_x4(a[h], xb + sw128(16 * mt + (lane & 15), 4 * kp + 2 * h + (lane >> 4)));
#pragma unroll
      for (int j = 0; j < 4; ++j) ldsm_x4(b[j], wb + sw128(32 * nh + 8 * j + (lane & 7), 4 * kp + (lane >> 3)));
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_bf16_16816(d[j], a[h], b[j][2 * h], b[j][2 * h + 1]);
    }
  }
  // the partial: token rows 16 mt + g, + 8; columns 64 cg + 32 nh + 8 j + 2 t, + 1
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int tok = 16 * mt + g + 8 * r;
    if (tok < ntok) {
      float* row = acc + ((size_t)split * ntok + tok) * DK + PS_COLS * cg + 32 * nh + 2 * t;
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<float2*>(row + 8 * j) = make_float2(d[j][2 * r], d[j][2 * r + 1]);
    }
  }
}

// The epilogue of a split projection (few tokens): one CTA per token, one
// thread per payload column.  The column's value is the sum of the ksplit pairs'
// partials in split order (so the result does not depend on which pair finished
// first); then, as in project_kernel: RMSNorm over the 512 latent columns with
// the gain, the rotation of the RoPE key's pairs (2i, 2i+1), one bf16 rounding,
// the page write (quantized per the pool's format) and the optional payload row.
constexpr int PF_THREADS = DK;  // 576

template <int FMT>
__global__ void __launch_bounds__(PF_THREADS) project_finish_kernel(
    const float* __restrict__ acc, int ksplit, int ntok, const uint16_t* __restrict__ kv_norm_w, float eps,
    const RopeFreq freq, int num_pages, uint8_t* __restrict__ pages, const int32_t* __restrict__ page_table,
    int max_pages, const int32_t* __restrict__ pos, int T, uint16_t* __restrict__ latent_out, int* err) {
  __shared__ __align__(16) float y[DK];
  __shared__ float red[PF_THREADS / 32];
  const int tok = blockIdx.x, c = threadIdx.x, lane = c & 31, warp = c >> 5;
  const float g = c < DC ? __uint_as_float((uint32_t)kv_norm_w[c] << 16) : 0.f;
  // the token's slot in the pool (and the position its key is rotated by):
  // inputs of the call, read before the wait (the kernel before this one in
  // the stream writes only the partials)
  const int b = tok / T, t = tok - b * T;
  const int p0 = pos[b];
  const long long p = (long long)p0 + t;
  uint8_t* page = nullptr;
  int slot = 0;
  if (p0 < 0 || p >= (long long)max_pages * PAGE) {
    if (c == 0) raise_error(err, MLA_ERR_BOUNDS, b);
  } else {
    const int phys = page_table[(size_t)b * max_pages + (int)(p / PAGE)];
    if (phys < 0 || phys >= num_pages) {
      if (c == 0) raise_error(err, MLA_ERR_BOUNDS, phys);
    } else {
      constexpr size_t pb = FMT == MLA_FMT_BF16 ? PAGE_BYTES_BF16 : FMT == MLA_FMT_INT8 ? PAGE_BYTES_INT8 : PAGE_BYTES_INT4;
      page = pages + (size_t)phys * pb;
      slot = (int)(p % PAGE);
    }
  }
  grid_dep_wait();  // the partials of every split
  // the projection of column c: the splits' partials, summed in split order
  const float* a = acc + (size_t)tok * DK + c;
  const size_t sstride = (size_t)ntok * DK;
  float v = 0.f;
  int s = 0;
  for (; s + 16 <= ksplit; s += 16) {  // sixteen loads in flight
    float q[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) q[k] = a[(s + k) * sstride];
#pragma unroll
    for (int k = 0; k < 16; ++k) v += q[k];
  }
  if (s + 8 <= ksplit) {
    float q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = a[(s + k) * sstride];
#pragma unroll
    for (int k = 0; k < 8; ++k) v += q[k];
    s += 8;
  }
  for (; s < ksplit; ++s) v += a[s * sstride];
  // RMSNorm: the sum of squares of the 512 latent columns (warps 0..15)
  float ss = c < DC ? v * v : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (c < DC) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < DC / 32; ++w) tot += red[w];
    const float rinv = rsqrtf(tot * (1.0f / DC) + eps);
    y[c] = bf16r(v * rinv * g);
  } else {
    // RoPE key: pair (2i, 2i+1) is the lane pair (even, odd) of warps 16, 17
    const int rc = c - DC, i = rc >> 1;
    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
    float sn, cs;
    rope_sincos(p, freq.turn[i], &sn, &cs);
    const float x0 = (rc & 1) ? other : v, x1 = (rc & 1) ? v : other;  // y[2i], y[2i+1] before the rotation
    y[c] = bf16r((rc & 1) ? x0 * sn + x1 * cs : x0 * cs - x1 * sn);
  }
  __syncthreads();
  if (latent_out != nullptr && c < DK / 8)
    reinterpret_cast<uint4*>(latent_out + (size_t)tok * DK)[c] =
        make_uint4(pack_bf16x2(y[8 * c], y[8 * c + 1]), pack_bf16x2(y[8 * c + 2], y[8 * c + 3]),
                   pack_bf16x2(y[8 * c + 4], y[8 * c + 5]), pack_bf16x2(y[8 * c + 6], y[8 * c + 7]));
  if (page != nullptr) {
    if (FMT == MLA_FMT_BF16) {
      if (c < DK / 8)
        reinterpret_cast<uint4*>(page + (size_t)slot * DK * 2)[c] =
            make_uint4(pack_bf16x2(y[8 * c], y[8 * c + 1]), pack_bf16x2(y[8 * c + 2], y[8 * c + 3]),
                       pack_bf16x2(y[8 * c + 4], y[8 * c + 5]), pack_bf16x2(y[8 * c + 6], y[8 * c + 7]));
    } else if (c < DK / 32) {
      write_quantized32<FMT>(y + 32 * c, 32 * c, page, slot);
    }
  }
}

}  // namespace

// turn[i] = theta^(-2i/64) / (2 pi) modulo one turn, times 2^64, rounded:
// formed in double (scaling by 2^64 is exact), wrapping to 0 at a whole turn
RopeFreq rope_freq(float rope_theta) {
  RopeFreq fr;
  for (int i = 0; i < DR / 2; ++i) {
    const double u = std::pow((double)rope_theta, -2.0 * i / DR) / 6.283185307179586;
    const double v = std::nearbyint(std::ldexp(u - std::floor(u), 64));
    fr.turn[i] = v >= 18446744073709551616.0 ? 0 : (uint64_t)v;
  }
  return fr;
}

int project_splits(long long ntok, int hidden, int sms, int requested) {
  const int chunks = hidden / 64;
  const long long mtiles = (ntok + PJ_ROWS - 1) / PJ_ROWS;
  if (chunks <= 0 || mtiles <= 0) return 1;
  if (requested > 0) return requested < chunks ? requested : chunks;
  if (2 * mtiles >= sms) return 1;
  const int want = (int)(sms / (2 * mtiles));
  const int cap = chunks / 2 > 1 ? chunks / 2 : 1;  // at least two 64-wide chunks of hidden per pair
  const int k = want < cap ? want : cap;
  return k > 1 ? k : 1;
}

int project_small_splits(int hidden, int sms) {
  const int chunks = hidden / 64;
  int k = sms / PS_NG;  // about one CTA per SM
  const int need = (chunks + PS_MAXCH - 1) / PS_MAXCH;  // at most PS_MAXCH chunks per CTA
  if (k < need) k = need;
  if (k > chunks) k = chunks;
  return k > 1 ? k : 1;
}

size_t project_small_workspace_bytes(long long ntok, int ksplit) {
  return ntok <= 0 ? 0 : align_up((size_t)ksplit * ntok * DK * 4, 256);
}

size_t project_workspace_bytes(long long ntok, int ksplit) {
  if (ksplit <= 1 || ntok <= 0) return 0;
  return align_up((size_t)ksplit * ntok * DK * 4, 256);  // one fp32 partial payload per (pair, token)
}

cudaError_t launch_cache_project(const void* x, int hidden, const void* wkv_a, const void* kv_norm_w, float eps,
                                 float rope_theta, int fmt, int num_pages, void* pages, const int32_t* page_table,
                                 int max_pages, const int32_t* pos, int B, int T, void* latent_out, int ksplit,
                                 bool small, void* workspace, int* err, cudaStream_t s) {
  const long long ntok = (long long)B * T;
  if (ntok == 0) return cudaSuccess;
  void (*finish)(const float*, int, int, const uint16_t*, float, RopeFreq, int, uint8_t*, const int32_t*, int,
                 const int32_t*, int, uint16_t*, int*) =
      fmt == MLA_FMT_BF16 ? project_finish_kernel<MLA_FMT_BF16>
      : fmt == MLA_FMT_INT8 ? project_finish_kernel<MLA_FMT_INT8>
                            : project_finish_kernel<MLA_FMT_INT4>;
  if (small) {
    if (ntok > PS_TOK || hidden % 64 != 0 || (hidden / 64 + ksplit - 1) / ksplit > PS_MAXCH) return cudaErrorInvalidValue;
    CUtensorMap tm_x, tm_w;
    // x: (hidden, tokens) bf16, wkv_a: (hidden, 576), innermost first; boxes of 64 x 64, 128B swizzle
    if (!encode_3d(&tm_x, x, (uint64_t)hidden, (uint64_t)ntok, 1, (uint64_t)hidden * 2, (uint64_t)ntok * hidden * 2,
                   64, PS_TOK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&tm_w, wkv_a, (uint64_t)hidden, DK, 1, (uint64_t)hidden * 2, (uint64_t)DK * hidden * 2, 64,
                   PS_COLS, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const RopeFreq fr = rope_freq(rope_theta);
    float* acc = static_cast<float*>(workspace);
    const size_t smem = sizeof(PsSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(project_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    project_small_kernel<<<dim3(PS_NG, ksplit), 256, smem, s>>>(tm_x, tm_w, (int)ntok, hidden / 64, ksplit, acc, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(finish, dim3((unsigned)ntok), dim3(PF_THREADS), 0, s, static_cast<const float*>(acc), ksplit,
                      (int)ntok, static_cast<const uint16_t*>(kv_norm_w), eps, fr, num_pages,
                      static_cast<uint8_t*>(pages), page_table, max_pages, pos, T,
                      static_cast<uint16_t*>(latent_out), err);
  }
  const long long mtiles = (ntok + PJ_ROWS - 1) / PJ_ROWS;
  const int chunks = hidden / 64;
  CUtensorMap tm_x, tm_wc, tm_wr;
  // x: (hidden, tokens) bf16, boxes of 64 x 128; wkv_a: (hidden, 576), boxes of 64 x 256 and 64 x 32
  if (!encode_3d(&tm_x, x, (uint64_t)hidden, (uint64_t)ntok, 1, (uint64_t)hidden * 2, (uint64_t)ntok * hidden * 2, 64,
                 PJ_ROWS, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_3d(&tm_wc, wkv_a, (uint64_t)hidden, DK, 1, (uint64_t)hidden * 2, (uint64_t)DK * hidden * 2, 64, PJ_HALF,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_3d(&tm_wr, wkv_a, (uint64_t)hidden, DK, 1, (uint64_t)hidden * 2, (uint64_t)DK * hidden * 2, 64, PJ_ROPE,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const RopeFreq fr = rope_freq(rope_theta);
  float* acc = ksplit > 1 ? static_cast<float*>(workspace) : nullptr;
  const size_t smem = sizeof(PjSmem) + 1024;
  void (*kernel)(CUtensorMap, CUtensorMap, CUtensorMap, const uint16_t*, float, RopeFreq, int, uint8_t*,
                 const int32_t*, int, const int32_t*, int, int, int, int, uint16_t*, float*, int*) =
      fmt == MLA_FMT_BF16 ? project_kernel<MLA_FMT_BF16>
      : fmt == MLA_FMT_INT8 ? project_kernel<MLA_FMT_INT8>
                            : project_kernel<MLA_FMT_INT4>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * mtiles * ksplit));
  cfg.blockDim = dim3(PJ_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, tm_x, tm_wc, tm_wr, static_cast<const uint16_t*>(kv_norm_w), eps, fr, num_pages,
                         static_cast<uint8_t*>(pages), page_table, max_pages, pos, T, (int)ntok, chunks, ksplit,
                         static_cast<uint16_t*>(latent_out), acc, err);
  if (e != cudaSuccess || ksplit <= 1) return e;
  return launch_pdl(finish, dim3((unsigned)ntok), dim3(PF_THREADS), 0, s, static_cast<const float*>(acc), ksplit,
                    (int)ntok, static_cast<const uint16_t*>(kv_norm_w), eps, fr, num_pages,
                    static_cast<uint8_t*>(pages), page_table, max_pages, pos, T, static_cast<uint16_t*>(latent_out),
                    err);
}

}  // namespace mla
