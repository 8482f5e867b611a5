// Split-KV absorbed decode for 16 heads (the V2-Lite layer) on the warp-level
// tensor-core instruction mma.sync m16n8k16 (bf16 operands, fp32 accumulate).
//
// What it computes is the decode of "DeepSeek MLA 吸收式缓存" §2.2–§2.4 in its
// MQA form (§6.1: key width 576, value width 512), per split of a row's tokens:
//   s_t = scale (q_lat . c_t + q_pe . k_pe_t),  online softmax over t,
//   O   = sum_t p_t c_t,  emitted as O / l (bf16) and LSE = m + ln l per head.
//
// Why this instruction.  With 16 heads the decode does 2 x 16 x (576 + 512) =
// 34,816 FLOP per 1,152-byte cached token, 30 FLOP/B: at the HBM rate that is
// ~200 TFLOP/s, more than twice what the fp32 FMA pipes deliver, so a CUDA-core
// kernel cannot stream the cache at HBM speed.  The fifth-generation MMA has
// 128 rows, of which 16 heads fill one eighth.  mma.sync's M = 16 is exactly
// the head count: the query is the A operand (16 heads x 16 dims), a token
// block of the cache is B, with no padding rows (its ~600 TFLOP/s on this part
// leave the kernel HBM-bound).
//
// Layout.  One CTA per (worker, group of 16 heads), one CTA per SM.  A worker
// walks its contiguous range of 64-token pages (see decode_plan.cu) in halves
// of 32 tokens; each half page arrives by TMA as nine [32 tokens][64 dims]
// boxes with the 128-byte swizzle into a 4-stage ring, L2 evict-first.  Four
// warp roles work on different half pages at once, synchronised by mbarriers
// only (every wait bounded), each one half page behind the one before:
//   producer (1 warp)   computes each half page's descriptor (row, valid
//                       tokens, segment start / end) and refills a stage as
//                       soon as the roles that read it are done with it;
//   scores   (9 warps)  warp c owns key dims [64c, 64c+64) (box c): its 16-head
//                       x 64-dim query slice sits in registers as A fragments
//                       for the whole segment, and it multiplies it with all
//                       32 tokens of its box (4 token tiles x 4 k-steps, B by
//                       ldmatrix); the nine partial score tiles go to a
//                       double-buffered exchange tile;
//   softmax  (4 warps)  8 threads per head, 4 tokens each: add the nine
//                       partials, mask, and run the online softmax in fp32 with
//                       a rescale at every new maximum (the pages' online
//                       softmax); P in bf16 and the rescale factor to a
//                       double-buffered tile;
//   P.V      (8 warps)  warp w accumulates O for latent dims [64w, 64w+64) (16
//                       heads x 64 fp32 in registers): 8 dim tiles x 2 token
//                       k-steps, P as A (ldmatrix), the box as B (ldmatrix.trans).
// Every byte of a stage is read from shared memory once for the scores and the
// latent part once more for P.V.
#include "tc_ptx.cuh"
#include "warp_mma.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int MH = 16;                     // heads per CTA (the MMA's M)
constexpr int MT = 32;                     // tokens per half page
constexpr int NBOX = DK / 64;              // 9 boxes of 64 key dims
constexpr int NSC = NBOX;                  // score warps
constexpr int NSM = 4;                     // softmax warps
constexpr int NPV = DC / 64;               // P.V warps (8)
constexpr int SM_WARP0 = NSC;              // first softmax warp
constexpr int PV_WARP0 = NSC + NSM;        // first P.V warp
constexpr int PROD_WARP = NSC + NSM + NPV; // the TMA producer warp
constexpr int MTHREADS = 32 * (PROD_WARP + 1);  // 704
constexpr uint32_t BOX_BYTES = MT * 128;   // 4 KB: 32 rows of 64 bf16
constexpr uint32_t HALF_PAGE = NBOX * BOX_BYTES;  // 36,864
constexpr int RED_LD = MT;                 // fp32 row pitch of a partial score tile (columns swizzled: red_col)
constexpr int P_LD = MT + 8;               // bf16 row pitch of the P tile (80 B: conflict-free ldmatrix)
constexpr int NST = 4;                     // stages of the half-page ring

struct __align__(1024) SmemMMA {
  uint8_t kv[NST][NBOX][BOX_BYTES];        // 147,456 B, 128B-swizzled boxes
  float red[2][NBOX][MH][RED_LD];          // partial scores, double-buffered (36 KB)
  uint16_t p[2][MH][P_LD];                 // P (bf16), the A operand of P.V
  float alpha[2][MH];                      // rescale factor of a half page
  float lfin[2][MH];                       // l of each head at a segment's end
  uint64_t full[NST], empty[NST];          // stage landed / read by the scores and the P.V
  uint64_t red_full[2], red_empty[2];      // partial scores written / read
  uint64_t p_full[2], p_empty[2];          // P, alpha (and l) written / read
  int4 info[NST];                          // per stage: row, valid tokens, flags (HP_*), -
  int abort_flag;
};
static_assert(sizeof(SmemMMA) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
// flags of a half page's descriptor
constexpr int HP_FIRST = 1, HP_LAST_OF_SEG = 2, HP_LAST = 4;

// column of token column col (even) of head row h in a partial score tile:
// pairs of columns XOR-swizzled by the row, so that the writers' float2 stores
// (8 rows x 4 column pairs per instruction) spread over the banks
__device__ __forceinline__ int red_col(int h, int col) { return col ^ ((h & 7) << 2); }
// a probe that, while the phase is incomplete, suspends the thread for up to
// `ns` nanoseconds (it resumes as soon as the phase completes), so waiting
// warps do not keep the shared-memory pipe busy with probes that the copies'
// issue would queue behind
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t PROBE_SLEEP_NS = 20000;

// bounded wait: false after the time limit (recorded, and every role told
// through the abort flag) or once another warp gave up; the polling loop out
// of line
__device__ __noinline__ bool mwait_slow(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait_sleep(bar, parity, PROBE_SLEEP_NS)) return true;
    if ((k & 7) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort = 1;
        raise_error(err, MLA_ERR_TIMEOUT, 400 + where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mwait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return mwait_slow(bar, parity, abort, err, where);
}
// the same, by every lane of a warp, with one outcome for the whole warp (a lane
// that saw the phase complete and one that saw the abort flag agree on giving up)
__device__ __forceinline__ bool mwait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  return __all_sync(0xffffffffu, mwait(bar, parity, abort, err, where));
}

__global__ void __launch_bounds__(MTHREADS, 1)
    attend_mma_kernel(const __grid_constant__ CUtensorMap tm_kv, const uint16_t* __restrict__ q_cat, int H,
                      int num_pages, const int32_t* __restrict__ page_table, int max_pages, int B, float scale_log2,
                      const int* __restrict__ plan, int seg_cap, uint16_t* __restrict__ part_o,
                      float* __restrict__ part_lse, int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmemMMA& S = *reinterpret_cast<SmemMMA*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  grid_dep_wait();  // the plan, the query and the cache may come from the kernels before this one
  grid_dep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int worker = blockIdx.x, hg = blockIdx.y;
  const int T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  const int* seq_c = plan + plan_off_seq(B);
  if (worker >= W) return;  // a plan may use fewer workers than this launch has CTAs
  const int x0 = (int)worker_begin(worker, T, W), x1 = (int)worker_begin(worker + 1, T, W);
  if (x0 >= x1) return;

  if (tid == 0) {
    prefetch_tmap(&tm_kv);
    for (int k = 0; k < NST; ++k) {
      mbar_init(&S.full[k], 1);
      mbar_init(&S.empty[k], NSC + NPV);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&S.red_full[k], NSC);
      mbar_init(&S.red_empty[k], NSM);
      mbar_init(&S.p_full[k], NSM);
      mbar_init(&S.p_empty[k], NPV);
    }
    S.abort_flag = 0;
    fence_barrier_init();
  }
  int lo = 0, hi = B;  // first row whose tiles contain x0: prefix[lo] <= x0 < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x0) lo = mid; else hi = mid;
  }
  __syncthreads();  // the only block-wide barrier: barriers initialised
  volatile int* abort = &S.abort_flag;

  if (warp == PROD_WARP) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the range (lane-uniform values); lane 0 issues.  The
    // row's bounds stay in registers and the page ids of 32 tiles at a time are
    // fetched by the 32 lanes at once, so a half page costs no dependent global
    // load on the way to its copy.
    const uint64_t policy = policy_evict_first();
    int b = lo, pb0 = prefix[lo], pb1 = prefix[lo + 1], nb = seq_c[lo];
    int pt_base = -1, pt_val = 0;  // lane l: page id of tile pt_base + l of row b
    int i = 0, prev_b = -1;
    bool ok = true;
    for (int x = x0; x < x1 && ok; ++x) {
      while (x >= pb1) {  // the next row with tiles
        ++b;
        pb0 = pb1;
        pb1 = prefix[b + 1];
        nb = seq_c[b];
        pt_base = -1;
      }
      const int j = x - pb0;
      if (pt_base < 0 || j >= pt_base + 32) {
        pt_base = j;
        pt_val = j + lane < max_pages ? page_table[(size_t)b * max_pages + j + lane] : 0;
      }
      int phys = __shfl_sync(0xffffffffu, pt_val, j - pt_base);
      if (phys < 0 || phys >= num_pages) {
        if (lane == 0) raise_error(err, MLA_ERR_BOUNDS, phys);
        phys = 0;
      }
      const int valid = min(PAGE, nb - PAGE * j);  // >= 1
      const bool tile_last_of_seg = x + 1 == x1 || x + 1 >= pb1;
      for (int half = 0; half < (valid > MT ? 2 : 1); ++half, ++i) {
        const int st = i % NST;
        const bool last_half = half == 1 || valid <= MT;
        const int nvalid = half == 0 ? min(MT, valid) : valid - MT;
        const int flags = (b != prev_b ? HP_FIRST : 0) | (last_half && tile_last_of_seg ? HP_LAST_OF_SEG : 0) |
                          (last_half && x + 1 == x1 ? HP_LAST : 0);
        prev_b = b;
        // the stage's last half page (i - NST) has been read by every role
        if (i >= NST && !mwait_warp(&S.empty[st], ((i / NST) - 1) & 1, abort, err, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          S.info[st] = make_int4(b, nvalid, flags, 0);  // published by the arrive below
          mbar_arrive_expect_tx(&S.full[st], HALF_PAGE);
#pragma unroll 1
          for (int c9 = 0; c9 < NBOX; ++c9)
            tma_load_3d_hint(S.kv[st][c9], &tm_kv, 64 * c9, MT * half, phys, &S.full[st], policy);
        }
      }
    }
    if (!ok && lane == 0) {
      // let the copies still in flight land before the CTA can exit (bounded)
      for (int k = max(0, i - NST); k < i; ++k) (void)mbar_wait(&S.full[k % NST], (k / NST) & 1);
    }
    return;
  }

  if (warp < NSC) {
    // ------------------------------------------------------------ score warps
    const int box = warp;
    uint32_t qa[4][4];
    for (int i = 0;; ++i) {
      const int st = i % NST, rb = i & 1;
      if (!mwait_warp(&S.full[st], (i / NST) & 1, abort, err, 1)) break;
      const int4 hp = S.info[st];
      const int nvalid = hp.y;
      if (hp.z & HP_FIRST) {
        // new row: this warp's query slice into A fragments
        const uint32_t* q = reinterpret_cast<const uint32_t*>(q_cat + ((size_t)hp.x * H + hg * MH) * DK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int d = 64 * box + 16 * kk + 2 * t;  // even: a bf16 pair
          qa[kk][0] = q[(g * DK + d) >> 1];
          qa[kk][1] = q[((g + 8) * DK + d) >> 1];
          qa[kk][2] = q[(g * DK + d + 8) >> 1];
          qa[kk][3] = q[((g + 8) * DK + d + 8) >> 1];
        }
      }
      // the exchange tile rb was read by the softmax of half page i - 2
      if (i >= 2 && !mwait_warp(&S.red_empty[rb], ((i >> 1) - 1) & 1, abort, err, 2)) break;
      const uint32_t bb = smem_u32(S.kv[st][box]);
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      // B fragments of the four token tiles (tokens 8n..8n+7) for all 64 dims
      // (b[n][kp]: dims 32kp + 8m, m = 0..3, i.e. two k-steps), loaded first;
      // then the 16 MMAs k-step by k-step across the four independent
      // accumulators
      uint32_t b[4][2][4];
#pragma unroll
      for (int kp = 0; kp < 2; ++kp)
#pragma unroll
        for (int n = 0; n < 4; ++n) ldsm_x4(b[n][kp], bb + sw128(8 * n + (lane & 7), 4 * kp + (lane >> 3)));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int n = 0; n < 4; ++n)
          mma_bf16_16816(acc[n], qa[kk], b[n][kk >> 1][2 * (kk & 1)], b[n][kk >> 1][2 * (kk & 1) + 1]);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        *reinterpret_cast<float2*>(&S.red[rb][box][g][red_col(g, 8 * n + 2 * t)]) = make_float2(acc[n][0], acc[n][1]);
        *reinterpret_cast<float2*>(&S.red[rb][box][g + 8][red_col(g + 8, 8 * n + 2 * t)]) =
            make_float2(acc[n][2], acc[n][3]);
      }
      if (nvalid < MT && box < NPV) {
        // value rows of this box past the sequence end to zero (p = 0 there, but
        // 0 x NaN is NaN); this warp's score reads of them are done
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int k = nvalid * 8 + lane; k < MT * 8; k += 32)
          *reinterpret_cast<uint4*>(S.kv[st][box] + (size_t)k * 16) = z;
        fence_proxy_async_smem();  // the next TMA copy into this stage comes after these writes
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.red_full[rb]);
        mbar_arrive(&S.empty[st]);
      }
      if (hp.z & HP_LAST) break;
    }
    return;
  }

  if (warp < PV_WARP0) {
    // ------------------------------------------------------------ softmax warps
    // head sh, tokens 4 sj .. 4 sj + 3 (8 threads per head, 4 heads per warp)
    const int sid = tid - 32 * SM_WARP0;
    const int sh = sid >> 3, sj = sid & 7;
    float m_run = -INFINITY, l_run = 0.f;
    for (int i = 0;; ++i) {
      const int st = i % NST, rb = i & 1;
      // (the score warps read this half page's descriptor after its stage landed)
      if (!mwait_warp(&S.red_full[rb], (i >> 1) & 1, abort, err, 3)) break;
      const int4 hp = S.info[st];
      const int nvalid = hp.y;
      if (hp.z & HP_FIRST) {
        m_run = -INFINITY;
        l_run = 0.f;
      }
      float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c9 = 0; c9 < NBOX; ++c9) {
        const float4 v = *reinterpret_cast<const float4*>(&S.red[rb][c9][sh][red_col(sh, 4 * sj)]);
        sc.x += v.x;
        sc.y += v.y;
        sc.z += v.z;
        sc.w += v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.red_empty[rb]);
      // tokens past the sequence end: their rows hold whatever the page slot held,
      // so the score is replaced, not combined
      const int k0 = 4 * sj;
      sc.x = k0 < nvalid ? sc.x * scale_log2 : -INFINITY;
      sc.y = k0 + 1 < nvalid ? sc.y * scale_log2 : -INFINITY;
      sc.z = k0 + 2 < nvalid ? sc.z * scale_log2 : -INFINITY;
      sc.w = k0 + 3 < nvalid ? sc.w * scale_log2 : -INFINITY;
      float mt = fmaxf(fmaxf(sc.x, sc.y), fmaxf(sc.z, sc.w));
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m_run, mt);  // finite: every half page holds a token
      const float alpha = ex2(m_run - m_new);  // 0 at a segment's first half page
      const float p0 = ex2(sc.x - m_new), p1 = ex2(sc.y - m_new), p2 = ex2(sc.z - m_new), p3 = ex2(sc.w - m_new);
      float sum = (p0 + p1) + (p2 + p3);
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      // the P tile rb (and its alpha, l) was read by the P.V of half page i - 2
      if (i >= 2 && !mwait_warp(&S.p_empty[rb], ((i >> 1) - 1) & 1, abort, err, 4)) break;
      *reinterpret_cast<uint2*>(&S.p[rb][sh][k0]) = make_uint2(pack_bf16x2(p0, p1), pack_bf16x2(p2, p3));
      if (sj == 0) {
        S.alpha[rb][sh] = alpha;
        if (hp.z & HP_LAST_OF_SEG) {
          S.lfin[rb][sh] = l_run;
          part_lse[(size_t)(worker + hp.x) * H + hg * MH + sh] = (m_run + log2f(l_run)) * 0.69314718055994531f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[rb]);
      if (hp.z & HP_LAST) break;
    }
    return;
  }

  // -------------------------------------------------------------- P.V warps
  const int w = warp - PV_WARP0;  // latent dims [64w, 64w+64)
  float o[8][4];                  // O of heads g, g+8 over dims 64w + 8j + 2t, +1
  for (int i = 0;; ++i) {
    const int st = i % NST, rb = i & 1;
    // P, alpha (and l) of all 16 heads; the stage (with the tail rows the score
    // warps zeroed before the exchange tile filled)
    if (!mwait_warp(&S.p_full[rb], (i >> 1) & 1, abort, err, 5)) break;
    if (!mwait_warp(&S.full[st], (i / NST) & 1, abort, err, 6)) break;
    const int4 hp = S.info[st];
    if (hp.z & HP_FIRST) {
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    }
    // ---- O = alpha O + P . V over this warp's 64 latent dims -----------------
    const float ag = S.alpha[rb][g], ag8 = S.alpha[rb][g + 8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= ag;
      o[j][1] *= ag;
      o[j][2] *= ag8;
      o[j][3] *= ag8;
    }
    const uint32_t vb = smem_u32(S.kv[st][w]);
    const uint32_t pb = smem_u32(&S.p[rb][0][0]);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t pa[4], b[4][4];
      ldsm_x4(pa, pb + (uint32_t)((lane & 15) * P_LD + 16 * kk + 8 * (lane >> 4)) * 2u);
      // matrices: tokens 16kk + 8(m & 1) + 0..7 at dims 16jp + 8(m >> 1) + 0..7
      const int m = lane >> 3, r = 16 * kk + 8 * (m & 1) + (lane & 7);
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) ldsm_x4_trans(b[jp], vb + sw128(r, 2 * jp + (m >> 1)));
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        mma_bf16_16816(o[2 * jp], pa, b[jp][0], b[jp][1]);
        mma_bf16_16816(o[2 * jp + 1], pa, b[jp][2], b[jp][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[st]);  // this warp's reads of the stage are done
    if (hp.z & HP_LAST_OF_SEG) {
      const float ig = 1.f / S.lfin[rb][g], ig8 = 1.f / S.lfin[rb][g + 8];
      // heads hg * MH + g and + 8 (head-major partials: segment seg of head h at h * seg_cap + seg)
      const size_t seg = (size_t)(worker + hp.x), hstride = (size_t)seg_cap * DC;
      uint16_t* dst = part_o + ((size_t)(hg * MH + g) * seg_cap + seg) * DC + 64 * w + 2 * t;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        *reinterpret_cast<uint32_t*>(dst + 8 * j) = pack_bf16x2(o[j][0] * ig, o[j][1] * ig);
        *reinterpret_cast<uint32_t*>(dst + 8 * hstride + 8 * j) = pack_bf16x2(o[j][2] * ig8, o[j][3] * ig8);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.p_empty[rb]);  // P, alpha and l of rb read
    if (hp.z & HP_LAST) break;
  }
}

}  // namespace

int attend_mma_workers(int num_sms) { return num_sms; }

cudaError_t launch_attend_mma(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                              const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                              int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s) {
  if (fmt != MLA_FMT_BF16 || H % MH != 0) return cudaErrorNotSupported;
  CUtensorMap tm;
  // pages as [num_pages][64 tokens][576 dims] bf16; a box is 32 tokens x 64 dims
  if (!encode_3d(&tm, pages, DK, PAGE, (uint64_t)num_pages, DK * 2, PAGE_BYTES_BF16, 64, MT,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(SmemMMA) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attend_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attend_mma_kernel, dim3(workers, H / MH), dim3(MTHREADS), smem, s, tm,
                    static_cast<const uint16_t*>(q_cat), H, num_pages, page_table, max_pages, B,
                    scale * 1.4426950408889634f, plan, seg_cap, part_o, part_lse, err);
}

}  // namespace mla
