// Split-KV absorbed decode on the fifth-generation tensor cores (128 heads,
// the DeepSeek-V3 shape), bf16 latent cache.
//
// What it computes (per worker range of 64-token pages, see decode_plan.cu),
// following "DeepSeek MLA 吸收式缓存" §2.2–§2.4 and §6.1 (MQA over the latent:
// key width 576, value width 512):
//   S[h,t] = q_lat[h] . c_t + q_pe[h] . k_pe_t          (M = 128 heads, K = 576)
//   online softmax over t (log2 domain, scale folded in)
//   O[h,:] += P[h,t] c_t                                (M = 128, N = 512)
//   emitted per segment as O / l and LSE = (m + log2 l) ln 2.
//
// Why a CTA pair.  O is 128 x 512 fp32 = 256 KB, all of one SM's tensor memory.
// The pair splits the latent width: CTA r owns latent dims [256r, 256r+256)
// and RoPE dims [32r, 32r+32).  Each CTA
//  * TMA-loads only its half of every 64-token page (HBM bytes are not
//    duplicated), 4 pages in flight;
//  * keeps its half of the 128-head query (288 bf16 per head) in TMEM as the
//    A operand of the score MMA;
//  * per 32-token half page, computes a partial S (M=128, N=32, K=288) into
//    TMEM and sends it to the peer's shared memory; adds the peer's partial.
//    fp32 addition commutes, so both CTAs hold identical scores and take
//    identical softmax decisions;
//  * accumulates its O half (128 x 256 fp32) in TMEM with P (bf16, TMEM) as the
//    A operand and its V half (shared memory, latent-major) as B.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2..9 softmax.  Softmax warps w and w+4 share TMEM lanes
// 32*(w%4)..+31 (one head per lane) and split each half page's 32 columns
// 16/16; the partners combine row maxima and sums through shared memory.
// The softmax loop is software-pipelined: it sends half page h while it
// finishes half page h-1, so the exchange latency hides behind work.  Each
// thread sends its 16 partial scores with asynchronous remote stores that
// complete on the peer's transaction-counted barrier.
// Every wait is bounded; a timeout records MLA_ERR_TIMEOUT, stops all roles,
// lets in-flight copies and MMAs land, frees TMEM and returns.
//
// Tensor memory (512 columns): O [0,256), q_lat half [256,384), q_pe half
// [384,400), S double buffer [400,464), P double buffer (bf16 pairs) [464,496).
#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int TC_THREADS = 320;
constexpr int NSOFT = 256;                                    // softmax threads (warps 2..9)
constexpr int STAGES = 4;
constexpr int TILE = 64;                                      // tokens per page / TMA stage
constexpr int HT = 32;                                        // tokens per half page (MMA N, softmax unit)
constexpr int HALF_C = 256;
constexpr int PE_HALF = 32;
constexpr uint32_t KV_CHUNK = TILE * 64 * 2;                  // 8,192: [64 tokens][64 dims] 128B-swizzled
constexpr uint32_t KV_PE_OFF = 4 * KV_CHUNK;                  // 32,768: [64 tokens][32 dims] 64B-swizzled
constexpr uint32_t KV_BYTES = TILE * (HALF_C + PE_HALF) * 2;  // 36,864
constexpr uint32_t XBYTES = 128 * HT * 4;                     // 16,384: one partial score half tile
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_QPE = 384, TM_S = 400, TM_P = 464;
constexpr float RESCALE_LOG2 = 8.f;  // move the running max only when it grows by > 2^8
constexpr long long WAIT_LIMIT_CYCLES = 4000000000ll;  // ~2 s at the maximum SM clock

struct __align__(1024) SmemTC {
  uint8_t kv[STAGES][KV_BYTES];
  float xin[2][128 * HT];   // the peer's partial scores, row-major, 16-byte chunks swizzled by row
  float red_m[2][2][128];   // partner row maxima [buffer][column half][row]
  float red_l[2][128];      // partner row sums at a segment end
  uint64_t kv_full[STAGES], kv_empty[STAGES];
  uint64_t q_ready;
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_free, mma_done;
  uint64_t x_full[2], x_empty[2];
  uint32_t tmem_base;
  volatile int abort_flag;
};
static_assert(sizeof(SmemTC) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(KV_BYTES % 1024 == 0, "swizzled tiles need 1 KB alignment");

struct TcArgs {
  const uint16_t* q_cat;  // [B][128][576] bf16
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
  // the SM cycle counter is cheap to read; the abort flag and the time limit
  // are checked every 8 probes (each probe may itself suspend the thread)
  const long long t0 = clock64();
  for (uint32_t k = 1;; ++k) {
    if (probe()) return true;
    if ((k & 7) == 0) {
      if (S.abort_flag) return false;
      if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
        S.abort_flag = 1;
        raise_error(err, MLA_ERR_TIMEOUT, where);
        return false;
      }
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

// row of the tile cursor: tiles [start, end) belong to row b of length n
struct RowCursor {
  int b, start, end, n;
  __device__ __forceinline__ void init(const int* prefix, const int* seq_c, int B, int x) {
    b = row_of_tile(prefix, B, x);
    start = prefix[b];
    end = prefix[b + 1];
    n = seq_c[b];
  }
  // loads only when the tile moves to a later row
  __device__ __forceinline__ void advance(const int* prefix, const int* seq_c, int x) {
    while (x >= end) {
      ++b;
      start = end;
      end = prefix[b + 1];
      n = seq_c[b];
    }
  }
};

// what the softmax warps need to know about one half page
struct HalfInfo {
  int b;        // row
  int nvalid;   // valid tokens of the whole page (1..64)
  int j;        // half index in the page (0, 1)
  bool seg_first, seg_last;  // first / last half page of the row's segment
};

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }
__device__ __forceinline__ uint32_t f2u(float v) { return __float_as_uint(v); }

// byte offset of 16-byte chunk c (0..7) of row r in a [128][32] fp32 exchange buffer
__device__ __forceinline__ uint32_t xchunk(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__(TC_THREADS, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_kv_c, const __grid_constant__ CUtensorMap tm_kv_pe,
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
  const int ntiles = x1 - x0;
  const int nhalf = 2 * ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.kv_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
    }
    mbar_init(&S.q_ready, 8);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.s_free[s], 8);
      mbar_init(&S.p_full[s], 8);
      mbar_init(&S.pv_done[s], 1);
      mbar_init(&S.x_full[s], 1);   // local expect_tx arrival + the peer's bulk bytes
      mbar_init(&S.x_empty[s], 8);  // one arrival per peer softmax warp
    }
    mbar_init(&S.o_free, 8);
    mbar_init(&S.mma_done, 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer arrives on our barriers and writes our exchange buffers
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;

  if (ntiles > 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp walks the tiles; lane l holds the page id of tile
    // jbase + l of the current row (one gather per 32 tiles), lane 0 waits and
    // issues the copies.
    if (lane == 0) {
      prefetch_tmap(&tm_kv_c);
      prefetch_tmap(&tm_kv_pe);
    }
    const uint64_t pol = policy_evict_first();
    int last_use[STAGES];
    for (int s = 0; s < STAGES; ++s) last_use[s] = -1;
    RowCursor rc;
    rc.init(prefix, seq_c, B, x0);
    int page_row = -1, jbase = 0, page_reg = 0;
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      rc.advance(prefix, seq_c, x);
      const int j = x - rc.start;
      if (rc.b != page_row || j - jbase >= 32) {
        page_row = rc.b;
        jbase = j;
        page_reg = (j + lane < rc.end - rc.start) ? a.page_table[(size_t)rc.b * a.max_pages + j + lane] : 0;
      }
      int page = __shfl_sync(0xffffffffu, page_reg, j - jbase);
      int ok = 1;
      if (lane == 0) {
        const int st = i % STAGES, u = i / STAGES;
        ok = wait_bar<false>(S, &S.kv_empty[st], (u & 1) ^ 1, a.err, 2);
        if (ok) {
          if (page < 0 || page >= a.num_pages) {
            raise_error(a.err, MLA_ERR_BOUNDS, page);
            page = 0;
          }
          mbar_arrive_expect_tx(&S.kv_full[st], KV_BYTES);
          for (int ci = 0; ci < 4; ++ci)
            tma_load_3d_hint(S.kv[st] + ci * KV_CHUNK, &tm_kv_c, HALF_C * rank + 64 * ci, 0, page, &S.kv_full[st],
                             pol);
          tma_load_3d_hint(S.kv[st] + KV_PE_OFF, &tm_kv_pe, DC + PE_HALF * rank, 0, page, &S.kv_full[st], pol);
          last_use[st] = u;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
    if (lane == 0 && S.abort_flag) {  // let copies in flight land before the CTA can exit
      for (int s = 0; s < STAGES; ++s)
        if (last_use[s] >= 0) (void)mbar_wait(&S.kv_full[s], last_use[s] & 1);
    }
  } else if (ntiles > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // order: S(h), then PV(h-2); S(h) needs the softmax to have read S(h-2),
    // PV(h-2) needs P(h-2).
    const uint32_t idesc_s = idesc_bf16_f32(128, HT, false, false);
    const uint32_t idesc_pv = idesc_bf16_f32(128, HALF_C, false, true);
    int q_seen = 0, pv_segments = 0;
    bool ok = true;
    RowCursor rc;          // cursor of the S side
    RowCursor rc_pv;       // cursor of the PV side (two half pages behind)
    rc.init(prefix, seq_c, B, x0);
    rc_pv = rc;

    auto issue_pv = [&](int g) -> bool {  // PV of half page g
      const int i = g >> 1, jj = g & 1, pb = g & 1, st = i % STAGES;
      if (!wait_bar<false>(S, &S.p_full[pb], (g >> 1) & 1, a.err, 6)) return false;
      bool seg_first = false;
      if (jj == 0) {
        const int xr = x0 + i;
        rc_pv.advance(prefix, seq_c, xr);
        seg_first = (xr == x0) || (xr == rc_pv.start);
      }
      // the first half page of a segment overwrites O: wait for the previous
      // segment's epilogue to have read it
      if (seg_first) {
        if (pv_segments > 0 && !wait_bar<false>(S, &S.o_free, (pv_segments - 1) & 1, a.err, 7)) return false;
        ++pv_segments;
      }
      fence_after_sync();
      const uint32_t kv_addr = smem_u32(S.kv[st]);
#pragma unroll
      for (int kk = 0; kk < HT / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_P + 16 * pb + 8 * kk,
               smem_desc(kv_addr + (HT * jj + 16 * kk) * 128, KV_CHUNK, 1024, SWIZZLE_128B), idesc_pv,
               (seg_first && kk == 0) ? 0u : 1u);
      mma_commit(&S.pv_done[pb]);
      if (jj == 1) mma_commit(&S.kv_empty[st]);
      return true;
    };

    for (int h = 0; h < nhalf; ++h) {
      const int i = h >> 1, jj = h & 1, st = i % STAGES, sb = h & 1;
      if (jj == 0) {
        const int x = x0 + i;
        rc.advance(prefix, seq_c, x);
        if (x == x0 || x == rc.start) {  // the query of this segment must be in TMEM
          if (!wait_bar<false>(S, &S.q_ready, q_seen & 1, a.err, 3)) { ok = false; break; }
          ++q_seen;
        }
        if (!wait_bar<false>(S, &S.kv_full[st], (i / STAGES) & 1, a.err, 4)) { ok = false; break; }
      }
      if (!wait_bar<false>(S, &S.s_free[sb], ((h >> 1) & 1) ^ 1, a.err, 5)) { ok = false; break; }
      fence_after_sync();
      const uint32_t kv_addr = smem_u32(S.kv[st]);
      const uint32_t d = tmem + TM_S + HT * sb;
#pragma unroll
      for (int ci = 0; ci < 4; ++ci)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(d, tmem + TM_Q + ci * 32 + kk * 8,
                 smem_desc(kv_addr + ci * KV_CHUNK + jj * (HT * 128) + kk * 32, 16, 1024, SWIZZLE_128B), idesc_s,
                 (ci | kk) != 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_ts(d, tmem + TM_QPE + kk * 8,
               smem_desc(kv_addr + KV_PE_OFF + jj * (HT * 64) + kk * 32, 16, 512, SWIZZLE_64B), idesc_s, 1u);
      mma_commit(&S.s_full[sb]);
      if (h >= 2 && !issue_pv(h - 2)) { ok = false; break; }
    }
    if (ok && nhalf >= 2) ok = issue_pv(nhalf - 2);
    if (ok) (void)issue_pv(nhalf - 1);
    mma_commit(&S.mma_done);
    (void)mbar_wait(&S.mma_done, 0);  // every issued MMA has finished
  } else if (ntiles > 0 && warp >= 2) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;               // TMEM lane quadrant
    const int ch = (warp - 2) >> 2;        // column half of each half page: 0 or 1
    const int row = q4 * 32 + lane;        // head = TMEM lane
    const int stid = threadIdx.x - 64;     // 0..255
    const uint32_t t_row = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t pair_bar = 1 + q4;      // named barrier shared with the partner warp
    const float c = a.scale_log2;          // > 0
    uint32_t peer_xin[2], peer_xfull[2], peer_xempty[2];  // cluster addresses in the peer CTA
    for (int k = 0; k < 2; ++k) {
      peer_xin[k] = mapa(smem_u32(S.xin[k]), peer);
      peer_xfull[k] = mapa(smem_u32(&S.x_full[k]), peer);
      peer_xempty[k] = mapa(smem_u32(&S.x_empty[k]), peer);
    }
    float m_ref = -INFINITY, l = 0.f;
    RowCursor rc;
    rc.init(prefix, seq_c, B, x0);
    uint32_t own_a[16], own_b[16];
    HalfInfo info_a, info_b;

    // A wait that fails does not leave the stage: it marks the thread failed and
    // the stage runs on (every later wait returns at once), so that the pair
    // barrier is still reached by both partner warps; the partners leave the
    // loop together, at the reduction barrier of stage B.
    bool failed = false;

    // A(h): read this CTA's partial scores of half page h and send them to the peer
    auto stage_a = [&](int h, uint32_t* own, HalfInfo& inf) {
      const int i = h >> 1, jj = h & 1, sb = h & 1, st = i % STAGES;
      const int x = x0 + i;
      if (jj == 0) rc.advance(prefix, seq_c, x);
      inf.b = rc.b;
      inf.nvalid = min(TILE, rc.n - TILE * (x - rc.start));
      inf.j = jj;
      inf.seg_first = jj == 0 && (x == x0 || x == rc.start);
      inf.seg_last = jj == 1 && (x + 1 == x1 || x + 1 == rc.end);
      if (inf.seg_first) {
        // this row's query half into TMEM; every S of the previous segment has
        // completed (this thread waited for each of them)
        const uint16_t* qrow = a.q_cat + ((size_t)rc.b * 128 + row) * DK;
        const uint4* qc = reinterpret_cast<const uint4*>(qrow + HALF_C * rank + 128 * ch);
        uint32_t v[64];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint4 u = qc[k];
          v[4 * k] = u.x; v[4 * k + 1] = u.y; v[4 * k + 2] = u.z; v[4 * k + 3] = u.w;
        }
        uint32_t pe[16];
        const uint4* qp = reinterpret_cast<const uint4*>(qrow + DC + PE_HALF * rank);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 u = qp[k];
          pe[4 * k] = u.x; pe[4 * k + 1] = u.y; pe[4 * k + 2] = u.z; pe[4 * k + 3] = u.w;
        }
        tmem_st32(t_row + TM_Q + 64 * ch, v);
        tmem_st32(t_row + TM_Q + 64 * ch + 32, v + 32);
        if (ch == 0) tmem_st16(t_row + TM_QPE, pe);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.q_ready);
      }
      if (stid == 0) mbar_arrive_expect_tx(&S.x_full[sb], XBYTES);  // the peer's partial for this half page
      if (!wait_bar<false>(S, &S.s_full[sb], (h >> 1) & 1, a.err, 9)) failed = true;
      __syncwarp();
      fence_after_sync();
      tmem_ld16(t_row + TM_S + HT * sb + 16 * ch, own);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.s_free[sb]);
      if (jj == 0 && inf.nvalid < TILE) {
        // page past the end of its sequence: zero the unused value rows so that
        // P = 0 never meets stale (possibly non-finite) cache contents
        const int units = (TILE - inf.nvalid) * 4 * 8;  // 16-byte units in 4 chunks of 128-byte rows
        for (int idx = stid; idx < units; idx += NSOFT) {
          const int r = inf.nvalid + idx / 32, ci = (idx % 32) / 8, v = idx % 8;
          *reinterpret_cast<uint4*>(S.kv[st] + ci * KV_CHUNK + r * 128 + v * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      // the peer has consumed what we sent into this buffer two half pages ago
      if (lane == 0 && !wait_bar<true>(S, &S.x_empty[sb], ((h >> 1) & 1) ^ 1, a.err, 10)) failed = true;
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_async_v4(peer_xin[sb] + xchunk(row, 4 * ch + k), own[4 * k], own[4 * k + 1], own[4 * k + 2],
                    own[4 * k + 3], peer_xfull[sb]);
    };

    // B(h): add the peer's partial, online softmax, P into TMEM, epilogue at a
    // segment end; returns false (on both partner warps alike) once either failed
    auto stage_b = [&](int h, const uint32_t* own, const HalfInfo& inf) -> bool {
      const int sb = h & 1;
      if (!wait_bar<false>(S, &S.x_full[sb], (h >> 1) & 1, a.err, 11)) failed = true;
      __syncwarp();
      const uint8_t* xi = reinterpret_cast<const uint8_t*>(S.xin[sb]);
      float s[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(xi + xchunk(row, 4 * ch + k));
        s[4 * k + 0] = u2f(own[4 * k + 0]) + v.x;
        s[4 * k + 1] = u2f(own[4 * k + 1]) + v.y;
        s[4 * k + 2] = u2f(own[4 * k + 2]) + v.z;
        s[4 * k + 3] = u2f(own[4 * k + 3]) + v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_relaxed(peer_xempty[sb]);  // our buffer may be refilled
      const int t0 = HT * inf.j + 16 * ch;  // token index of s[0] in the page
      if (inf.nvalid < TILE) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (t0 + k >= inf.nvalid) s[k] = -INFINITY;
      }
      float mraw = s[0];
#pragma unroll
      for (int k = 1; k < 16; ++k) mraw = fmaxf(mraw, s[k]);
      S.red_m[sb][ch][row] = mraw * c;
      const bool pair_ok = named_barrier_and(pair_bar, 64, !failed);
      const float mt = fmaxf(S.red_m[sb][0][row], S.red_m[sb][1][row]);
      if (inf.seg_first) {
        m_ref = mt;
        l = 0.f;
      }
      const bool need = !inf.seg_first && mt > m_ref + RESCALE_LOG2;
      if (__any_sync(0xffffffffu, need)) {
        // O may only be touched once every PV issued so far has completed
        if (!wait_bar<false>(S, &S.pv_done[(h - 1) & 1], ((h - 1) >> 1) & 1, a.err, 12)) failed = true;
        __syncwarp();
        fence_after_sync();
        const float alpha = need ? ex2(m_ref - mt) : 1.f;
#pragma unroll 1
        for (int k32 = 0; k32 < 4; ++k32) {
          uint32_t o[32];
          const uint32_t col = t_row + TM_O + 128 * ch + 32 * k32;
          tmem_ld32(col, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = f2u(u2f(o[k]) * alpha);
          tmem_st32(col, o);
        }
        tmem_st_wait();
        if (need) {
          l *= alpha;
          m_ref = mt;
        }
      }
      // p = 2^(s*c - m_ref), two at a time in half precision (the exponent is
      // <= RESCALE_LOG2, so p <= 256; P is rounded to bf16 for the MMA anyway)
      uint32_t pk[8];
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __half2 xh = __floats2half2_rn(fmaf(s[2 * k], c, -m_ref), fmaf(s[2 * k + 1], c, -m_ref));
        const uint32_t yh = ex2_h2(*reinterpret_cast<const uint32_t*>(&xh));
        const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&yh));
        sum += p.x + p.y;
        pk[k] = pack_bf16x2(p.x, p.y);
      }
      l += sum;
      // P buffer sb is free once PV(h-2) has completed
      if (!wait_bar<false>(S, &S.pv_done[sb], ((h >> 1) & 1) ^ 1, a.err, 13)) failed = true;
      __syncwarp();
      fence_after_sync();
      tmem_st8(t_row + TM_P + 16 * sb + 8 * ch, pk);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[sb]);
      if (inf.seg_last) {
        if (!wait_bar<false>(S, &S.pv_done[sb], (h >> 1) & 1, a.err, 14)) failed = true;
        __syncwarp();
        fence_after_sync();
        S.red_l[ch][row] = l;
        named_barrier(pair_bar, 64);
        const float L = S.red_l[0][row] + S.red_l[1][row];
        const float inv = 1.f / L;
        const int seg = worker + inf.b;
        float* dst = a.part_o + ((size_t)seg * 128 + row) * DC + HALF_C * rank + 128 * ch;
#pragma unroll 1
        for (int k32 = 0; k32 < 4; ++k32) {
          uint32_t o[32];
          tmem_ld32(t_row + TM_O + 128 * ch + 32 * k32, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            reinterpret_cast<float4*>(dst + 32 * k32)[k] =
                make_float4(u2f(o[4 * k]) * inv, u2f(o[4 * k + 1]) * inv, u2f(o[4 * k + 2]) * inv,
                            u2f(o[4 * k + 3]) * inv);
        }
        if (rank == 0 && ch == 0) a.part_lse[(size_t)seg * 128 + row] = (m_ref + log2f(L)) * 0.69314718055994531f;
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.o_free);
      }
      return pair_ok;
    };

    // software pipeline: A(h) then B(h-1); even and odd halves swap the buffers
    for (int h = 0; h <= nhalf; h += 2) {
      if (h < nhalf) stage_a(h, own_a, info_a);
      if (h >= 1 && !stage_b(h - 1, own_b, info_b)) break;
      if (h + 1 > nhalf) break;
      if (h + 1 < nhalf) stage_a(h + 1, own_b, info_b);
      if (!stage_b(h, own_a, info_a)) break;
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

cudaLaunchConfig_t launch_config(int workers, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * workers);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

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
      cudaLaunchAttribute attr[1];
      cudaLaunchConfig_t cfg = launch_config(num_sms / 2, nullptr, attr);
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
  if (!(scale > 0.f)) return cudaErrorInvalidValue;  // the row max is taken before scaling
  CUtensorMap tkv_c, tkv_pe;
  const uint64_t row = (uint64_t)DK * 2;  // 1,152 bytes per token slot
  if (!encode_3d(&tkv_c, pages, DK, PAGE, num_pages, row, PAGE_BYTES_BF16, 64, TILE, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&tkv_pe, pages, DK, PAGE, num_pages, row, PAGE_BYTES_BF16, 32, TILE, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  TcArgs args;
  args.q_cat = static_cast<const uint16_t*>(q_cat);
  args.plan = plan;
  args.page_table = page_table;
  args.part_o = part_o;
  args.part_lse = part_lse;
  args.err = err;
  args.B = B;
  args.max_pages = max_pages;
  args.num_pages = num_pages;
  args.scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(workers, s, attr);
  return cudaLaunchKernelEx(&cfg, attend_tc_kernel, tkv_c, tkv_pe, args);
}

}  // namespace mla
