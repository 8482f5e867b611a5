// Split-KV absorbed decode on the fifth-generation tensor cores (128 heads,
// the DeepSeek-V3 shape), bf16 latent cache.
//
// What it computes (per worker range of 64-token pages, see decode_plan.cu),
// following "DeepSeek MLA 吸收式缓存" §2.2–§2.4 and §6.1 (MQA over the latent:
// key width 576, value width 512):
//   S[h,t] = q_lat[h] . c_t + q_pe[h] . k_pe_t          (M = 128 heads, N = 64 tokens, K = 576)
//   online softmax over t (log2 domain, scale folded in)
//   O[h,:] += P[h,t] c_t                                (M = 128, N = 512, K = 64)
//   emitted per segment as O / l and LSE = (m + log2 l) ln 2.
//
// Why a CTA pair.  O is 128 x 512 fp32 = 256 KB, all of one SM's tensor memory,
// leaving nothing for S.  The pair splits the latent width: CTA r owns latent
// dims [256r, 256r+256) and RoPE dims [32r, 32r+32).  Each CTA
//  * TMA-loads only its half of every page tile (HBM bytes are not duplicated),
//  * computes a partial S over its 288 dims into TMEM,
//  * sends that partial (fp32) to the peer through distributed shared memory
//    and adds the peer's; fp32 addition commutes, so both CTAs hold identical
//    scores and take identical softmax decisions,
//  * accumulates its O half (128 x 256 fp32) in TMEM with P (bf16, in TMEM)
//    as the A operand and its V half (shared memory, latent-major) as B.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2..5 softmax (thread = head row = TMEM lane).  Every wait is
// bounded; a timeout records MLA_ERR_TIMEOUT, stops all roles, lets in-flight
// copies and MMAs land, frees TMEM and returns.
//
// Tensor memory map (512 columns): O half [0,256), S double buffer [256,384),
// P double buffer (bf16 pairs) [384,448).
// Shared memory: Q half (4 x [128][64] 128B-swizzled + [128][32] 64B-swizzled),
// 3 stages of page-tile halves (4 x [64][64] + [64][32]), the peer's partial
// scores [128][68] fp32, barriers.
#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int TC_THREADS = 192;
constexpr int STAGES = 3;
constexpr int TILE = 64;
constexpr int HALF_C = 256;
constexpr int PE_HALF = 32;
constexpr uint32_t Q_CHUNK = 128 * 64 * 2;                   // 16,384
constexpr uint32_t Q_PE_OFF = 4 * Q_CHUNK;                   // 65,536
constexpr uint32_t Q_BYTES = 128 * (HALF_C + PE_HALF) * 2;   // 73,728
constexpr uint32_t KV_CHUNK = TILE * 64 * 2;                 // 8,192
constexpr uint32_t KV_PE_OFF = 4 * KV_CHUNK;                 // 32,768
constexpr uint32_t KV_BYTES = TILE * (HALF_C + PE_HALF) * 2; // 36,864
constexpr int XLD = 68;                                      // padded row of the exchange buffer
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0, TM_S = 256, TM_P = 384;
constexpr float RESCALE_LOG2 = 8.f;  // move the running max only when it grows by > 2^8

struct __align__(1024) SmemTC {
  uint8_t q[Q_BYTES];
  uint8_t kv[STAGES][KV_BYTES];
  float xbuf[128 * XLD];
  uint64_t kv_full[STAGES], kv_empty[STAGES];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_free, mma_done;
  uint64_t x_full, x_empty;
  uint32_t tmem_base;
  volatile int abort_flag;
};

static_assert(sizeof(SmemTC) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(offsetof(SmemTC, kv) % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzled tiles need 1 KB alignment");

struct TcArgs {
  const int* plan;
  const int32_t* page_table;
  float* part_o;
  float* part_lse;
  int* err;
  int B, max_pages, num_pages;
  float scale_log2;
};

// Bounded wait shared by all roles: gives up after WAIT_LIMIT_NS (records
// MLA_ERR_TIMEOUT and raises the CTA's abort flag) or as soon as another role
// has aborted.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(SmemTC& S, uint64_t* bar, uint32_t parity, int* err, int where) {
  auto probe = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (probe()) return true;
    if (S.abort_flag) return false;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
      S.abort_flag = 1;
      raise_error(err, MLA_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// largest row b with prefix[b] <= x (rows with no tiles are skipped)
__device__ __forceinline__ int row_of_tile(const int* prefix, int B, int x) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }
__device__ __forceinline__ uint32_t f2u(float v) { return __float_as_uint(v); }

__global__ void __launch_bounds__(TC_THREADS, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_q_c, const __grid_constant__ CUtensorMap tm_q_pe,
                     const __grid_constant__ CUtensorMap tm_kv_c, const __grid_constant__ CUtensorMap tm_kv_pe,
                     const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  SmemTC& S = *reinterpret_cast<SmemTC*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int worker = blockIdx.x >> 1;
  const int T = a.plan[0], W = a.plan[1], B = a.B;
  const int* prefix = a.plan + PLAN_HDR;
  const int* seq_c = a.plan + PLAN_HDR + B + 1;
  const int x0 = (int)worker_begin(worker, T, W), x1 = (int)worker_begin(worker + 1, T, W);
  const bool has_work = x0 < x1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.kv_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
    }
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.s_free[s], 4);
      mbar_init(&S.p_full[s], 4);
      mbar_init(&S.pv_done[s], 1);
    }
    mbar_init(&S.o_free, 4);
    mbar_init(&S.mma_done, 1);
    mbar_init(&S.x_full, 128);
    mbar_init(&S.x_empty, 128);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer arrives on our barriers and writes our exchange buffer
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;

  if (has_work && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&tm_q_c);
    prefetch_tmap(&tm_q_pe);
    prefetch_tmap(&tm_kv_c);
    prefetch_tmap(&tm_kv_pe);
    const uint64_t pol = policy_evict_first();
    int last_use[STAGES];
    for (int s = 0; s < STAGES; ++s) last_use[s] = -1;
    int q_loads = 0;
    int b = row_of_tile(prefix, B, x0);
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      while (b < B - 1 && x >= prefix[b + 1]) ++b;
      if (x == x0 || x == prefix[b]) {  // new segment: this row's query half
        if (!wait_bar<false>(S, &S.q_empty, (q_loads & 1) ^ 1, a.err, 1)) break;
        mbar_arrive_expect_tx(&S.q_full, Q_BYTES);
        for (int ci = 0; ci < 4; ++ci)
          tma_load_3d(S.q + ci * Q_CHUNK, &tm_q_c, HALF_C * rank + 64 * ci, 0, b, &S.q_full);
        tma_load_3d(S.q + Q_PE_OFF, &tm_q_pe, DC + PE_HALF * rank, 0, b, &S.q_full);
        ++q_loads;
      }
      const int st = i % STAGES, u = i / STAGES;
      if (!wait_bar<false>(S, &S.kv_empty[st], (u & 1) ^ 1, a.err, 2)) break;
      int page = a.page_table[(size_t)b * a.max_pages + (x - prefix[b])];
      if (page < 0 || page >= a.num_pages) {
        raise_error(a.err, MLA_ERR_BOUNDS, page);
        page = 0;
      }
      mbar_arrive_expect_tx(&S.kv_full[st], KV_BYTES);
      for (int ci = 0; ci < 4; ++ci)
        tma_load_3d_hint(S.kv[st] + ci * KV_CHUNK, &tm_kv_c, HALF_C * rank + 64 * ci, 0, page, &S.kv_full[st], pol);
      tma_load_3d_hint(S.kv[st] + KV_PE_OFF, &tm_kv_pe, DC + PE_HALF * rank, 0, page, &S.kv_full[st], pol);
      last_use[st] = u;
    }
    if (S.abort_flag) {  // let copies in flight land before the CTA can exit
      for (int s = 0; s < STAGES; ++s)
        if (last_use[s] >= 0) (void)mbar_wait(&S.kv_full[s], last_use[s] & 1);
      if (q_loads > 0) (void)mbar_wait(&S.q_full, (q_loads - 1) & 1);
    }
  } else if (has_work && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_bf16_f32(128, TILE, false, false);
    const uint32_t idesc_pv = idesc_bf16_f32(128, HALF_C, false, true);
    const uint32_t q_addr = smem_u32(S.q);
    int q_seen = 0, pv_segments = 0;
    int prev_i = -1, prev_st = 0;
    bool prev_first = false, ok = true;

    auto issue_pv = [&](int j, int st, bool first) -> bool {
      const int sb = j & 1;
      if (!wait_bar<false>(S, &S.p_full[sb], (j >> 1) & 1, a.err, 6)) return false;
      if (first) {
        if (pv_segments > 0 && !wait_bar<false>(S, &S.o_free, (pv_segments - 1) & 1, a.err, 7)) return false;
        ++pv_segments;
      }
      fence_after_sync();
      const uint32_t kv_addr = smem_u32(S.kv[st]);
#pragma unroll
      for (int kk = 0; kk < TILE / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_P + 32 * sb + 8 * kk,
               smem_desc(kv_addr + kk * 16 * 128, KV_CHUNK, 1024, SWIZZLE_128B), idesc_pv,
               (first && kk == 0) ? 0u : 1u);
      mma_commit(&S.pv_done[sb]);
      mma_commit(&S.kv_empty[st]);
      return true;
    };

    int b = row_of_tile(prefix, B, x0);
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      while (b < B - 1 && x >= prefix[b + 1]) ++b;
      const bool first = (x == x0) || (x == prefix[b]);
      const bool last = (x + 1 == x1) || (x + 1 == prefix[b + 1]);
      if (first) {
        if (!wait_bar<false>(S, &S.q_full, q_seen & 1, a.err, 3)) { ok = false; break; }
        ++q_seen;
      }
      const int st = i % STAGES, u = i / STAGES, sb = i & 1;
      if (!wait_bar<false>(S, &S.kv_full[st], u & 1, a.err, 4)) { ok = false; break; }
      if (!wait_bar<false>(S, &S.s_free[sb], ((i >> 1) & 1) ^ 1, a.err, 5)) { ok = false; break; }
      fence_after_sync();
      const uint32_t kv_addr = smem_u32(S.kv[st]);
      const uint32_t d = tmem + TM_S + TILE * sb;
#pragma unroll
      for (int ci = 0; ci < 4; ++ci)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(d, smem_desc(q_addr + ci * Q_CHUNK + kk * 32, 16, 1024, SWIZZLE_128B),
                 smem_desc(kv_addr + ci * KV_CHUNK + kk * 32, 16, 1024, SWIZZLE_128B), idesc_s,
                 (ci | kk) != 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_ss(d, smem_desc(q_addr + Q_PE_OFF + kk * 32, 16, 512, SWIZZLE_64B),
               smem_desc(kv_addr + KV_PE_OFF + kk * 32, 16, 512, SWIZZLE_64B), idesc_s, 1u);
      mma_commit(&S.s_full[sb]);
      if (last) mma_commit(&S.q_empty);
      if (prev_i >= 0 && !issue_pv(prev_i, prev_st, prev_first)) { ok = false; break; }
      prev_i = i;
      prev_st = st;
      prev_first = first;
    }
    if (ok && prev_i >= 0) (void)issue_pv(prev_i, prev_st, prev_first);
    mma_commit(&S.mma_done);
    (void)mbar_wait(&S.mma_done, 0);  // every issued MMA has finished
  } else if (has_work && warp >= 2) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;  // head = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t t_s = tmem + lane_off + TM_S, t_p = tmem + lane_off + TM_P, t_o = tmem + lane_off + TM_O;
    const uint32_t peer_row = mapa(smem_u32(&S.xbuf[row * XLD]), peer);
    const uint32_t peer_full = mapa(smem_u32(&S.x_full), peer);
    const uint32_t peer_empty = mapa(smem_u32(&S.x_empty), peer);
    const float* my_row = &S.xbuf[row * XLD];
    float m_ref = -INFINITY, l = 0.f;
    int b = row_of_tile(prefix, B, x0);
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      while (b < B - 1 && x >= prefix[b + 1]) ++b;
      const bool first = (x == x0) || (x == prefix[b]);
      const bool last = (x + 1 == x1) || (x + 1 == prefix[b + 1]);
      const int nvalid = min(TILE, seq_c[b] - TILE * (x - prefix[b]));
      const int st = i % STAGES, sb = i & 1;

      // (a) a tile past the end of its sequence: zero the unused value rows so
      //     that P = 0 never meets stale (possibly non-finite) cache contents
      if (nvalid < TILE) {
        const bool ok = wait_bar<false>(S, &S.kv_full[st], (i / STAGES) & 1, a.err, 8);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int units = (TILE - nvalid) * 4 * 8;  // 16-byte units in 4 chunks of 128-byte rows
        for (int idx = threadIdx.x - 64; idx < units; idx += 128) {
          const int r = nvalid + idx / 32, ci = (idx % 32) / 8, v = idx % 8;
          *reinterpret_cast<uint4*>(S.kv[st] + ci * KV_CHUNK + r * 128 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }

      // (b) this CTA's partial scores
      bool ok = wait_bar<false>(S, &S.s_full[sb], (i >> 1) & 1, a.err, 9);
      if (!__all_sync(0xffffffffu, ok)) break;
      fence_after_sync();
      uint32_t r[TILE];
      tmem_ld32(t_s + TILE * sb, r);
      tmem_ld32(t_s + TILE * sb + 32, r + 32);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.s_free[sb]);

      // (c) swap partial scores with the peer CTA
      ok = wait_bar<true>(S, &S.x_empty, (i & 1) ^ 1, a.err, 10);
      if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
      for (int k = 0; k < TILE / 4; ++k)
        st_cluster_v4(peer_row + 16 * k, u2f(r[4 * k]), u2f(r[4 * k + 1]), u2f(r[4 * k + 2]), u2f(r[4 * k + 3]));
      mbar_arrive_remote(peer_full);
      ok = wait_bar<true>(S, &S.x_full, i & 1, a.err, 11);
      if (!__all_sync(0xffffffffu, ok)) break;
      float s[TILE];
#pragma unroll
      for (int k = 0; k < TILE / 4; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(my_row + 4 * k);
        s[4 * k + 0] = u2f(r[4 * k + 0]) + v.x;
        s[4 * k + 1] = u2f(r[4 * k + 1]) + v.y;
        s[4 * k + 2] = u2f(r[4 * k + 2]) + v.z;
        s[4 * k + 3] = u2f(r[4 * k + 3]) + v.w;
      }
      mbar_arrive_remote(peer_empty);

      // (d) online softmax in the log2 domain with a lazily moved reference max
      float mt = -INFINITY;
#pragma unroll
      for (int t = 0; t < TILE; ++t) {
        s[t] = t < nvalid ? s[t] * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[t]);
      }
      if (first) {
        m_ref = mt;
        l = 0.f;
      }
      const bool need = !first && mt > m_ref + RESCALE_LOG2;
      if (__any_sync(0xffffffffu, need)) {
        // O may only be touched once every PV issued so far has completed
        ok = wait_bar<false>(S, &S.pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, a.err, 12);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_after_sync();
        const float alpha = need ? ex2(m_ref - mt) : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < HALF_C / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(t_o + 32 * ch, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = f2u(u2f(o[k]) * alpha);
          tmem_st32(t_o + 32 * ch, o);
        }
        tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mt;
        }
      }
      float sum = 0.f;
      uint32_t pk[TILE / 2];
#pragma unroll
      for (int c = 0; c < TILE / 2; ++c) {
        const float p0 = ex2(s[2 * c] - m_ref), p1 = ex2(s[2 * c + 1] - m_ref);
        sum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += sum;

      // (e) P into TMEM once PV(i-2) has finished with that buffer
      ok = wait_bar<false>(S, &S.pv_done[sb], ((i >> 1) & 1) ^ 1, a.err, 13);
      if (!__all_sync(0xffffffffu, ok)) break;
      fence_after_sync();
      tmem_st32(t_p + 32 * sb, pk);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[sb]);

      // (f) end of the row's segment: O / l and the natural-log LSE
      if (last) {
        ok = wait_bar<false>(S, &S.pv_done[sb], (i >> 1) & 1, a.err, 14);
        if (!__all_sync(0xffffffffu, ok)) break;
        fence_after_sync();
        const float inv = 1.f / l;
        const int seg = worker + b;
        float* dst = a.part_o + ((size_t)seg * 128 + row) * DC + HALF_C * rank;
#pragma unroll 1
        for (int ch = 0; ch < HALF_C / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(t_o + 32 * ch, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            reinterpret_cast<float4*>(dst + 32 * ch)[k] =
                make_float4(u2f(o[4 * k]) * inv, u2f(o[4 * k + 1]) * inv, u2f(o[4 * k + 2]) * inv,
                            u2f(o[4 * k + 3]) * inv);
        }
        if (rank == 0) a.part_lse[(size_t)seg * 128 + row] = (m_ref + log2f(l)) * 0.69314718055994531f;
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.o_free);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer no longer touches our shared memory
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 tensor map: dims (d0 fastest), byte strides of dims 1 and 2, box (b0, b1, 1)
bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemBytes = sizeof(SmemTC) + 1024;

std::mutex g_tc_mu;
int g_tc_workers[64] = {};

}  // namespace

// persistent workers (CTA pairs) that fit on the device at once
int attend_tc_workers(int num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (g_tc_workers[dev] == 0) {
    int clusters = 0;
    if (cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (num_sms / 2));
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&clusters, attend_tc_kernel, &cfg) != cudaSuccess) clusters = 0;
    }
    (void)cudaGetLastError();
    g_tc_workers[dev] = clusters > 0 ? std::min(clusters, num_sms / 2) : num_sms / 2;
  }
  return g_tc_workers[dev];
}

cudaError_t launch_attend_tc(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                             const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                             int workers, float* part_o, float* part_lse, int* err, cudaStream_t s) {
  if (H != 128 || fmt != MLA_FMT_BF16 || workers < 1) return cudaErrorNotSupported;
  CUtensorMap tq_c, tq_pe, tkv_c, tkv_pe;
  const uint64_t row = (uint64_t)DK * 2;  // 1,152 bytes per query row / token slot
  if (!encode_3d(&tq_c, q_cat, DK, 128, B, row, row * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&tq_pe, q_cat, DK, 128, B, row, row * 128, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !encode_3d(&tkv_c, pages, DK, PAGE, num_pages, row, PAGE_BYTES_BF16, 64, TILE, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&tkv_pe, pages, DK, PAGE, num_pages, row, PAGE_BYTES_BF16, 32, TILE, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  TcArgs args;
  args.plan = plan;
  args.page_table = page_table;
  args.part_o = part_o;
  args.part_lse = part_lse;
  args.err = err;
  args.B = B;
  args.max_pages = max_pages;
  args.num_pages = num_pages;
  args.scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * workers);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_tc_kernel, tq_c, tq_pe, tkv_c, tkv_pe, args);
}

}  // namespace mla
