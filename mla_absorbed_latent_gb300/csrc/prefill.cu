// Unabsorbed ("compute-friendly") causal prefill.
//
// "手搓 MLA" §三 computes MLA without absorption: every cached latent is
// up-projected once into per-head keys and values (k_nope, v = split(kv_up):
// k_nope = W_UK c, v = W_UV c), the RoPE key is appended (k = [k_nope; k_pe],
// 192 wide, "DeepSeek MLA 吸收式缓存" §2.1/§2.4) and standard attention runs
// over the expanded tensors.  Its closing notes place this form at prefill
// and the absorbed one at decode: per (query, key) pair it costs 2 H (192 +
// 128) FLOPs instead of the absorbed 2 H (576 + 512), for a one-time
// expansion of 2 H 256 512 FLOPs per cached token.  The result is the same
// attention ("DeepSeek MLA 吸收式缓存" §2.2/§2.3 prove the two equal); query t
// of row b (the row's last T tokens are its queries) sees keys 0 .. n - T + t.
//
// Two kernels on the fifth-generation tensor cores:
//  expand_kernel   one CTA per (128-token tile, head, row):
//                  D[128 tokens][256] = C[128][512] . W_h^T, where C is the
//                  tile's cached latents (two pages, by TMA) and W_h the head's
//                  256 rows of wkv_b (k_nope rows then v rows); the tile's rows
//                  go to the workspace as bf16 [row][slot][head][256] (zeros
//                  past the row's length).
//  prefill_kernel  one CTA per (128-query tile, head, row): flash attention
//                  with Q = [q_nope; q_pe] (K = 192) resident in shared memory,
//                  64-key tiles of K = [k_nope (workspace); k_pe (cache page)]
//                  and V (workspace) in a 3-stage ring, S (128 x 64 fp32) in a
//                  double TMEM buffer, O (128 x 128 fp32) in TMEM.  Each softmax
//                  thread owns one query row: it moves its reference maximum
//                  only when a tile's maximum exceeds it by more than 2^8
//                  (then O and l are rescaled first), so p <= 2^8 always.
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int ROWS = 128;   // tokens per expansion tile / queries per attention tile (MMA M)
constexpr int KT = 64;      // keys per attention tile (one cache page)
constexpr int EXP_N = 256;  // expansion outputs per head: k_nope (128) then v (128)
constexpr uint32_t CH = 64 * 2;  // bytes of one 64-element row chunk (128B swizzle span)
constexpr long long PF_WAIT_NS = 2000000000ll;

// bounded wait of the prefill kernels (false after ~2 s or once another thread gave up)
__device__ __noinline__ bool pwait_slow(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 7) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > (uint64_t)PF_WAIT_NS) {
        *abort = 1;
        raise_error(err, MLA_ERR_TIMEOUT, 200 + where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return pwait_slow(bar, parity, abort, err, where);
}

// page id of logical page j of row b (outside the pool: page 0, reported)
__device__ __forceinline__ int page_of(const int32_t* page_table, int max_pages, int num_pages, int b, int j,
                                       int* err) {
  int p = j < max_pages ? page_table[(size_t)b * max_pages + j] : 0;
  if (p < 0 || p >= num_pages) {
    raise_error(err, MLA_ERR_BOUNDS, p);
    p = 0;
  }
  return p;
}

// clamped length of row b
__device__ __forceinline__ int row_len(const int32_t* seqlens, int b, int max_pages) {
  long long n = seqlens[b];
  const long long cap = (long long)max_pages * PAGE;
  if (n < 0) n = 0;
  if (n > cap) n = cap;
  return (int)n;
}

// ---------------------------------------------------------------------------
// expansion
// ---------------------------------------------------------------------------
struct __align__(1024) ExpSmem {
  uint8_t a[2][ROWS * CH];   // latent chunk kc: [128 tokens][64 dims] 128B-swizzled (two 64-token boxes)
  uint8_t w[2][EXP_N * CH];  // weight chunk kc: [256 outputs][64 dims] 128B-swizzled
  uint64_t full[2], empty[2], done;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(128, 1)
    expand_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_w,
                  const int32_t* __restrict__ page_table, int max_pages, int num_pages,
                  const int32_t* __restrict__ seqlens, int H, int T, uint16_t* __restrict__ kv, int* err) {
  extern __shared__ uint8_t smem_raw[];
  ExpSmem& S = *reinterpret_cast<ExpSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = row_len(seqlens, b, max_pages);
  const int t0 = tile * ROWS;
  if (t0 >= n) return;  // nothing of this row here (uniform over the CTA)
  const size_t S_CAP = (size_t)max_pages * PAGE;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.done, 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort = &S.abort_flag;
  constexpr int NK = DC / 64;  // 8 chunks of the latent width
  if (tid == 0) {
    // the tile's two pages (the second only if the row reaches it; else its rows are zeros)
    const int p0 = page_of(page_table, max_pages, num_pages, b, 2 * tile, err);
    const int p1 = t0 + PAGE < n ? page_of(page_table, max_pages, num_pages, b, 2 * tile + 1, err) : p0;
    const uint32_t idesc = idesc_bf16_f32(ROWS, EXP_N, false, false);
    int issued = 0;
    bool ok = true;
    // chunk kc: load, then the MMAs of chunk kc - 1 (two stages)
    for (int kc = 0; kc <= NK && ok; ++kc) {
      if (kc < NK) {
        const int st = kc & 1;
        ok = pwait(&S.empty[st], ((kc >> 1) & 1) ^ 1, abort, err, 0);
        if (!ok) break;
        mbar_arrive_expect_tx(&S.full[st], ROWS * CH + EXP_N * CH);
        tma_load_3d(S.a[st], &tm_c, 64 * kc, 0, p0, &S.full[st]);
        tma_load_3d(S.a[st] + 64 * CH, &tm_c, 64 * kc, 0, p1, &S.full[st]);
        tma_load_3d(S.w[st], &tm_w, 64 * kc, EXP_N * h, 0, &S.full[st]);
        ++issued;
      }
      if (kc >= 1) {
        const int c = kc - 1, st = c & 1;
        ok = pwait(&S.full[st], (c >> 1) & 1, abort, err, 1);
        if (!ok) break;
        fence_after_sync();
        const uint64_t ad = smem_desc(smem_u32(S.a[st]), 16, 1024, SWIZZLE_128B);
        const uint64_t bd = smem_desc(smem_u32(S.w[st]), 16, 1024, SWIZZLE_128B);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc, (c | kk) != 0 ? 1u : 0u);
        mma_commit(&S.empty[st]);
      }
    }
    mma_commit(&S.done);  // arrives when every MMA issued above has completed
    if (!ok)              // copies in flight land before the CTA exits
      for (int k = max(0, issued - 2); k < issued; ++k) (void)mbar_wait(&S.full[k & 1], (k >> 1) & 1);
  }
  // epilogue: thread r owns token t0 + r: 256 columns -> bf16 -> kv[b][t0+r][h][:]
  const bool ok = pwait(&S.done, 0, abort, err, 2);
  __syncwarp();
  fence_after_sync();
  const int r = warp * 32 + lane, t = t0 + r;
  uint4* dst = reinterpret_cast<uint4*>(kv + (((size_t)b * S_CAP + t) * H + h) * EXP_N);
#pragma unroll 1
  for (int c32 = 0; c32 < EXP_N / 32; ++c32) {
    uint32_t v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32 * c32, v);
    tmem_ld_wait();
    if (ok && t < n) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[4 * c32 + k] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
    } else if (t < (int)S_CAP && t < ((n + PAGE - 1) / PAGE) * PAGE) {
      // the row's last page past its length: zeros, so that p = 0 never meets garbage
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[4 * c32 + k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// causal flash attention over the expanded keys and values
// ---------------------------------------------------------------------------
constexpr int PF_ST = 3;                         // key/value ring stages
constexpr uint32_t Q_BYTES = 3 * ROWS * CH;      // [128][192]: 3 chunks of [128][64], 128B-swizzled
constexpr uint32_t K_BYTES = 3 * KT * CH;        // [64][192]: 3 chunks of [64][64]
constexpr uint32_t V_BYTES = 2 * KT * CH;        // [64][128]: 2 chunks of [64 keys][64 dims] (MN-major B)
constexpr uint32_t P_BYTES = ROWS * CH;          // [128][64] bf16, 128B-swizzled (K-major A)
constexpr uint32_t TM_S = 0, TM_O = 128;         // TMEM columns: S double buffer [0,128), O [128,256)
constexpr float PF_RESCALE = 8.f;                // move the reference when a tile's max exceeds it by > 2^8

struct __align__(1024) PfSmem {
  uint8_t q[Q_BYTES];
  uint8_t kv[PF_ST][K_BYTES + V_BYTES];
  uint8_t p[2][P_BYTES];
  uint64_t q_full, kv_full[PF_ST], kv_empty[PF_ST], s_full[2], s_free[2], p_full[2], pv_done[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PfSmem) + 1024 <= 232448, "prefill shared memory exceeds 227 KB");

struct PfArgs {
  const int32_t* page_table;
  const int32_t* seqlens;
  uint16_t* out;  // [B][T][H][128]
  int* err;
  int H, T, max_pages, num_pages;
  float scale_log2;
};

__global__ void __launch_bounds__(256, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                   const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_pe,
                   const PfArgs a) {
  extern __shared__ uint8_t smem_raw[];
  PfSmem& S = *reinterpret_cast<PfSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, T = a.T;
  const int n = row_len(a.seqlens, b, a.max_pages);
  const int t0 = qt * ROWS;
  if (t0 >= T) return;
  if (qt == 0 && h == 0 && tid == 0 && (n < T || n != a.seqlens[b])) raise_error(a.err, MLA_ERR_BOUNDS, b);
  // keys up to the view of the tile's last query: n - T + (last query index)
  const int qlast = min(t0 + ROWS, T) - 1;
  const int view = n - T + qlast + 1;  // keys 0 .. view-1 (may be < 1 for rows shorter than T)
  const int J = view > 0 ? (view + KT - 1) / KT : 0;

  if (tid == 0) {
    mbar_init(&S.q_full, 1);
    for (int s = 0; s < PF_ST; ++s) {
      mbar_init(&S.kv_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.s_free[s], 4);  // the 4 softmax warps
      mbar_init(&S.p_full[s], 4);
      mbar_init(&S.pv_done[s], 1);
    }
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort = &S.abort_flag;
  const size_t S_CAP = (size_t)a.max_pages * PAGE;

  if (warp == 0 && lane == 0 && J > 0) {
    // ---------------------------------------------------------- TMA producer
    const long long qrow = (long long)b * T + t0;  // flat (row, token) index of the tile's first query
    mbar_arrive_expect_tx(&S.q_full, Q_BYTES);
    tma_load_3d(S.q, &tm_qn, 0, h, (int)qrow, &S.q_full);
    tma_load_3d(S.q + ROWS * CH, &tm_qn, 64, h, (int)qrow, &S.q_full);
    tma_load_3d(S.q + 2 * ROWS * CH, &tm_qp, 0, h, (int)qrow, &S.q_full);
    int issued = 0;
    for (int j = 0; j < J; ++j) {
      const int st = j % PF_ST;
      if (!pwait(&S.kv_empty[st], ((j / PF_ST) & 1) ^ 1, abort, a.err, 10)) break;
      const int pg = page_of(a.page_table, a.max_pages, a.num_pages, b, j, a.err);
      uint8_t* dst = S.kv[st];
      const int krow = (int)((size_t)b * S_CAP + (size_t)j * KT);  // flat (row, slot) of the tile's first key
      mbar_arrive_expect_tx(&S.kv_full[st], K_BYTES + V_BYTES);
      tma_load_3d(dst, &tm_kv, 0, h, krow, &S.kv_full[st]);                  // k_nope dims 0..63
      tma_load_3d(dst + KT * CH, &tm_kv, 64, h, krow, &S.kv_full[st]);       // k_nope dims 64..127
      tma_load_3d(dst + 2 * KT * CH, &tm_pe, DC, 0, pg, &S.kv_full[st]);     // k_pe (the cache page)
      tma_load_3d(dst + K_BYTES, &tm_kv, 128, h, krow, &S.kv_full[st]);      // v dims 0..63
      tma_load_3d(dst + K_BYTES + KT * CH, &tm_kv, 192, h, krow, &S.kv_full[st]);  // v dims 64..127
      ++issued;
    }
    if (*abort) {
      (void)mbar_wait(&S.q_full, 0);
      for (int k = max(0, issued - PF_ST); k < issued; ++k) (void)mbar_wait(&S.kv_full[k % PF_ST], (k / PF_ST) & 1);
    }
  } else if (warp == 1 && lane == 0 && J > 0) {
    // ---------------------------------------------------------- MMA issuer:
    // S_0, S_1, then per tile j: P_j . V_j once P_j is written, S_{j+2}
    const uint32_t id_s = idesc_bf16_f32(ROWS, KT, false, false);
    const uint32_t id_pv = idesc_bf16_f32(ROWS, 128, false, true);
    bool ok = pwait(&S.q_full, 0, abort, a.err, 11);
    auto issue_s = [&](int j) -> bool {
      const int st = j % PF_ST, sb = j & 1;
      if (!pwait(&S.kv_full[st], (j / PF_ST) & 1, abort, a.err, 12)) return false;
      if (!pwait(&S.s_free[sb], ((j >> 1) & 1) ^ 1, abort, a.err, 13)) return false;
      fence_after_sync();
      const uint32_t qa = smem_u32(S.q), ka = smem_u32(S.kv[st]);
#pragma unroll
      for (int c = 0; c < 3; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + TM_S + KT * sb, smem_desc(qa + c * ROWS * CH + kk * 32, 16, 1024, SWIZZLE_128B),
                 smem_desc(ka + c * KT * CH + kk * 32, 16, 1024, SWIZZLE_128B), id_s, (c | kk) != 0 ? 1u : 0u);
      mma_commit(&S.s_full[sb]);
      return true;
    };
    for (int j = 0; j < min(2, J) && ok; ++j) ok = issue_s(j);
    for (int j = 0; j < J && ok; ++j) {
      const int st = j % PF_ST, pb = j & 1;
      if (!pwait(&S.p_full[pb], (j >> 1) & 1, abort, a.err, 14)) break;
      fence_after_sync();
      const uint32_t pa = smem_u32(S.p[pb]), va = smem_u32(S.kv[st] + K_BYTES);
#pragma unroll
      for (int kk = 0; kk < KT / 16; ++kk)
        mma_ss(tmem + TM_O, smem_desc(pa + kk * 32, 16, 1024, SWIZZLE_128B),
               smem_desc(va + kk * 16 * CH, KT * CH, 1024, SWIZZLE_128B), id_pv, (j | kk) != 0 ? 1u : 0u);
      mma_commit(&S.pv_done[pb]);
      mma_commit(&S.kv_empty[st]);
      if (j + 2 < J && !issue_s(j + 2)) break;
    }
    mma_commit(&S.q_full);  // (a spent barrier) once every MMA issued above has completed
    (void)mbar_wait(&S.q_full, 1);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- softmax warps:
    // thread r (TMEM lane r) owns query t0 + r
    const int q4 = warp & 3, r = q4 * 32 + lane, t = t0 + r;
    const uint32_t t_row = tmem + ((uint32_t)(q4 * 32) << 16);
    // keys this query sees: 0 .. lim-1 (padding rows past T see none)
    const int lim = t < T ? n - T + t + 1 : 0;
    const float c = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int sb = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!pwait(&S.s_full[sb], ph, abort, a.err, 15)) { ok = false; break; }
      __syncwarp();
      fence_after_sync();
      uint32_t v[KT];
      tmem_ld32(t_row + TM_S + KT * sb, v);
      tmem_ld32(t_row + TM_S + KT * sb + 32, v + 32);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.s_free[sb]);
      float s[KT];
      const int kl = lim - KT * j;  // visible keys of this tile
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        s[k] = k < kl ? __uint_as_float(v[k]) * c : -INFINITY;
        mt = fmaxf(mt, s[k]);
      }
      // the reference: the first tile's maximum, then moved only by > 2^8
      float alpha = 1.f;
      if (mt > m_ref + PF_RESCALE || m_ref == -INFINITY) {
        const float m_new = fmaxf(mt, m_ref);
        if (m_new != m_ref) {
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_new);
          m_ref = m_new;
        }
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds tiles < j in the old reference: rescale after P_{j-1} . V_{j-1}
        if (!pwait(&S.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, a.err, 16)) { ok = false; break; }
        __syncwarp();
        fence_after_sync();
#pragma unroll 1
        for (int c32 = 0; c32 < 4; ++c32) {
          uint32_t o[32];
          tmem_ld32(t_row + TM_O + 32 * c32, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(t_row + TM_O + 32 * c32, o);
        }
        tmem_st_wait();
        fence_before_sync();
      }
      l *= alpha;
      const float mr = fmaxf(m_ref, -3.0e38f);  // -inf only when every s is -inf (p = 0)
      uint32_t pk[KT / 2];
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < KT / 2; ++k) {
        const float p0 = ex2(s[2 * k] - mr), p1 = ex2(s[2 * k + 1] - mr);
        sum += p0 + p1;
        pk[k] = pack_bf16x2(p0, p1);
      }
      l += sum;
      // P tile sb is free once P_{j-2} . V_{j-2} has completed
      if (j >= 2 && !pwait(&S.pv_done[sb], ph ^ 1u, abort, a.err, 17)) { ok = false; break; }
      __syncwarp();
      uint8_t* prow = S.p[sb] + r * CH;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_smem();  // generic writes -> the tensor core's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[sb]);
    }
    // ---- O / l of this query
    if (ok && J > 0 && pwait(&S.pv_done[(J - 1) & 1], ((J - 1) >> 1) & 1, abort, a.err, 18)) {
      __syncwarp();
      fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.out + (((size_t)b * T + t) * H + h) * DV);
#pragma unroll 1
      for (int c32 = 0; c32 < 4; ++c32) {
        uint32_t o[32];
        tmem_ld32(t_row + TM_O + 32 * c32, o);
        tmem_ld_wait();
        if (t < T) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[4 * c32 + k] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                                          pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                                          pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                                          pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
        }
      }
    } else if (J == 0 && t < T) {
      // the row holds none of the keys this query would see (shorter than T; reported by the host check)
      uint4* dst = reinterpret_cast<uint4*>(a.out + (((size_t)b * T + t) * H + h) * DV);
      for (int k = 0; k < DV / 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

size_t prefill_workspace_bytes(int B, int H, int max_pages) {
  return align_up((size_t)B * max_pages * PAGE * H * EXP_N * 2, 1024);
}

cudaError_t launch_prefill(const void* q_nope, const void* q_pe, const void* wkv_b, int H, int T, int num_pages,
                           const void* pages, const int32_t* page_table, int max_pages, const int32_t* seqlens, int B,
                           float scale, void* workspace, void* out, int* err, cudaStream_t s) {
  if (B == 0 || T == 0) return cudaSuccess;
  const uint64_t row = (uint64_t)DK * 2;  // bytes per cache slot
  const uint64_t S_CAP = (uint64_t)max_pages * PAGE;
  CUtensorMap tm_c, tm_w, tm_qn, tm_qp, tm_kv, tm_pe;
  // latents of a page: (576 dims, 64 slots, pages), boxes of 64 dims x 64 slots, 128B swizzle
  bool ok = encode_3d(&tm_c, pages, DK, PAGE, (uint64_t)num_pages, row, PAGE_BYTES_BF16, 64, PAGE,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  // wkv_b: (512 latent, H*256 rows, 1), boxes of 64 x 256
  ok = ok && encode_3d(&tm_w, wkv_b, DC, (uint64_t)H * EXP_N, 1, DC * 2, (uint64_t)H * EXP_N * DC * 2, 64, EXP_N,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  // queries: (dims, H, B*T), boxes of 64 dims x 1 head x 128 tokens
  ok = ok && encode_3d_box(&tm_qn, q_nope, DN, H, (uint64_t)B * T, DN * 2, (uint64_t)H * DN * 2, 64, 1, ROWS,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_3d_box(&tm_qp, q_pe, DR, H, (uint64_t)B * T, DR * 2, (uint64_t)H * DR * 2, 64, 1, ROWS,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  // expanded keys/values: (256, H, B*S_CAP), boxes of 64 x 1 head x 64 keys
  ok = ok && encode_3d_box(&tm_kv, workspace, EXP_N, H, (uint64_t)B * S_CAP, EXP_N * 2, (uint64_t)H * EXP_N * 2, 64, 1,
                           KT, CU_TENSOR_MAP_SWIZZLE_128B);
  // the RoPE keys of a page: the same view as tm_c (x = 512)
  tm_pe = tm_c;
  if (!ok) return cudaErrorInvalidValue;
  const size_t es = sizeof(ExpSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)es);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((S_CAP + ROWS - 1) / ROWS);
  // plain stream order for both kernels: the expansion reads the cache the
  // work before it may write, and the attention reads the expansion
  expand_kernel<<<dim3(tiles, H, B), 128, es, s>>>(tm_c, tm_w, page_table, max_pages, num_pages, seqlens, H, T,
                                                   static_cast<uint16_t*>(workspace), err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  PfArgs args;
  args.page_table = page_table;
  args.seqlens = seqlens;
  args.out = static_cast<uint16_t*>(out);
  args.err = err;
  args.H = H;
  args.T = T;
  args.max_pages = max_pages;
  args.num_pages = num_pages;
  args.scale_log2 = scale * 1.4426950408889634f;
  const size_t ps = sizeof(PfSmem) + 1024;
  e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ps);
  if (e != cudaSuccess) return e;
  prefill_kernel<<<dim3((T + ROWS - 1) / ROWS, H, B), 256, ps, s>>>(tm_qn, tm_qp, tm_kv, tm_pe, args);
  return cudaGetLastError();
}

}  // namespace mla
