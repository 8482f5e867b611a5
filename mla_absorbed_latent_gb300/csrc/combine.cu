// Merge of the split-KV partials and the value up-projection, in one kernel.
//
// Each split s of row b left O_s = (sum_{t in s} e^{x_t - m_s} c_t) / l_s and
// LSE_s = m_s + ln l_s per head.  The exact softmax over the whole row is
//   o_lat = sum_s e^{LSE_s - LSE} O_s,   LSE = ln sum_s e^{LSE_s}.
// Then "DeepSeek MLA 吸收式缓存" §2.3 (sum_t p_t W_UV c_t = W_UV sum_t p_t c_t)
// applies the value projection once per head: out[b,h,:] = W_UV[h] o_lat[b,h,:]
// ("手搓 MLA" §四, einsum("thc,hdc->thd", out_lat, W_UV)).
//
// One CTA per (head h, group of RB rows).  The segments of a group's rows are
// consecutive slots of the partial buffer (slot w + b for worker w, row b), and
// the partials are head-major (a head's segments are consecutive 1 KB rows), so
// for every 64-wide latent chunk TMA boxes of 64 segments bring that chunk of
// the group's segments ([segments][64] bf16) into a ring slot, as many boxes as
// the group needs.  The merge warps (a thread per row and 8-dim unit) sum their
// row's segments with the softmax weights, round o_lat once into a bf16 high
// part and a bf16 residual, and write both as K-major 128B-swizzled operand
// tiles; an MMA warp issues the fifth-generation tensor-core MMAs
//   D[128 out dims][RB rows] += W_UV[h][:, chunk] . hi^T + W_UV[h][:, chunk] . lo^T
// (M = 128, N = RB, K = 64 per chunk), so the only roundings left are W_UV's
// own bf16, the residual's (relative 2^-16) and the fp32 accumulation.
// W_UV[h] streams through a ring of 128B-swizzled TMA tiles whose first loads
// are issued before the kernel waits for the attention step; the two rings
// have a loader warp each.
#include "tc_ptx.cuh"
#include "warp_mma.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int KC = 64;                    // latent dims per chunk
constexpr int NCHUNK = DC / KC;           // 8

constexpr int SBOX = 64;                  // segments per TMA box: a tile holds as many boxes as its segments need
                                          // (an issued box costs ~100-200 SM cycles: few, large boxes)
constexpr uint32_t W_TILE = DV * KC * 2;  // 16 KB: W_UV[h] rows x 64 latent dims, 128B-swizzled


template <int RB>
struct CombLayout {
  // ring depths of the W_UV tiles, the partial tiles and the operand tiles.
  // An operand tile of chunk k is rewritten only after the MMAs of chunk
  // k - BST (issued once every merge warp wrote chunk k - BST) complete, a
  // round trip of about 2.5 us; with 64 rows (one CTA per SM) four operand
  // tiles keep the merge warps that many chunks ahead of the tensor core
  static constexpr int WST = RB >= 64 ? 3 : 2, PST = RB >= 64 ? 4 : 3, BST = RB >= 64 ? 4 : 2;
  // segments per partial tile: every warp waits for every tile of a chunk and
  // a ring slot is free only when all have read it, so the tile holds all of
  // a typical group's segments (64 rows: B + W = 140 at 64 rows and 152 SMs)
  static constexpr int SEGB = RB >= 64 ? 192 : 128;
  static constexpr uint32_t P_TILE = SEGB * KC * 2;  // [SEGB segments][64 dims] bf16
  static constexpr int NW = RB / 4;          // merge warps: 4 rows x 8 units each
  static constexpr int THREADS = 32 * (NW + 3);  // + the W_UV loader / TMEM owner, partial loader and MMA warps
  static constexpr uint32_t TCOLS = RB < 32 ? 32 : RB;  // TMEM columns (allocations are >= 32)
  static constexpr uint32_t B_TILE = RB * 128;   // [RB rows][64 dims] bf16, 128B-swizzled
  static constexpr uint32_t OFF_W = 0;
  static constexpr uint32_t OFF_P = OFF_W + WST * W_TILE;
  static constexpr uint32_t OFF_B = OFF_P + PST * P_TILE;  // [BST][hi, lo]
  static constexpr uint32_t OFF_BAR = OFF_B + BST * 2 * B_TILE;
  // barriers: w_full, w_empty, p_full, p_empty, b_full, b_free, d_full
  static constexpr uint32_t NBAR = 2 * WST + 2 * PST + 2 * BST + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
  static constexpr uint32_t OFF_WGT = OFF_MISC + 16;         // float [RB + max workers]: weight per segment
  static size_t bytes(int max_workers) { return OFF_WGT + (size_t)(RB + max_workers) * 4 + 1024; }
};

// bounded wait for the combine kernel: false after the time limit or once
// another thread of the CTA gave up (the polling loop out of line)
__device__ __noinline__ bool cwait_slow(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 7) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort = 1;
        raise_error(err, MLA_ERR_TIMEOUT, 100 + where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool cwait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return cwait_slow(bar, parity, abort, err, where);
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Exact recompute of a flagged row.  The attend kernel flags a row whose
// weights it could not form exactly in its running reference (a score far
// above it, or exchanged half scores too large for fp16); here each (row,
// head) of such a row is recomputed from the cache with the online softmax of
// the pages, which rescales at every new maximum, in fp32: one token per
// thread for the scores of a chunk, then every thread its latent dims of
// sum_t p_t c_t; o_lat = that / l; out = W_UV[h] o_lat.  Rare path: plain
// loads, no staging.
// ---------------------------------------------------------------------------
__device__ __forceinline__ size_t fmt_page_bytes(int fmt) {
  return fmt == MLA_FMT_BF16 ? PAGE_BYTES_BF16 : fmt == MLA_FMT_INT8 ? PAGE_BYTES_INT8 : PAGE_BYTES_INT4;
}
__device__ __forceinline__ float bf16_at(const uint8_t* p) {
  return __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16);
}
// physical page of logical page j of row b (an id outside the pool reads page 0 and is reported)
__device__ const uint8_t* fix_page(const FixCtx& fx, int b, int j, int* err) {
  int pid = fx.page_table[(size_t)b * fx.max_pages + j];
  if (pid < 0 || pid >= fx.num_pages) {
    raise_error(err, MLA_ERR_BOUNDS, pid);
    pid = 0;
  }
  return fx.pages + (size_t)pid * fmt_page_bytes(fx.fmt);
}
// elements 8u .. 8u+7 (u < 72) of the 576-wide key of slot `slot`, in fp32;
// quantized codes as x = code * s (+ z), the block quantizers of "DeepSeek-V2-Lite
// MLA 吸收式 KV 缓存优化" §3.2
__device__ void fix_key_unit(int fmt, const uint8_t* pg, int slot, int u, float* f) {
  if (fmt == MLA_FMT_BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(pg + (size_t)slot * DK * 2 + u * 16);
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
    return;
  }
  const bool i8 = fmt == MLA_FMT_INT8;
  if (u >= DC / 8) {  // RoPE key: INT8 codes, one bf16 scale per 8 dims (both quantized formats)
    const int g = u - DC / 8;
    const int8_t* c = reinterpret_cast<const int8_t*>(pg + (i8 ? I8_PE_CODE : I4_PE_CODE) + slot * DR + 8 * g);
    const float sc = bf16_at(pg + (i8 ? I8_PE_SCALE : I4_PE_SCALE) + (slot * (DR / 8) + g) * 2);
    for (int k = 0; k < 8; ++k) f[k] = (float)c[k] * sc;
    return;
  }
  const int grp = u / 4;  // 32-channel group
  if (i8) {
    const int8_t* c = reinterpret_cast<const int8_t*>(pg + I8_C_CODE + slot * DC + 8 * u);
    const float sc = bf16_at(pg + I8_C_SCALE + (slot * (DC / 32) + grp) * 2);
    for (int k = 0; k < 8; ++k) f[k] = (float)c[k] * sc;
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(pg + I4_C_CODE + slot * (DC / 2) + 4 * u);
    const float sc = bf16_at(pg + I4_C_SCALE + (slot * (DC / 32) + grp) * 2);
    const float z = bf16_at(pg + I4_C_ZERO + (slot * (DC / 32) + grp) * 2);
    for (int k = 0; k < 8; ++k) f[k] = fmaf((float)((w >> (4 * k)) & 0xFu), sc, z);
  }
}
// latent element d (< 512) of slot `slot`, in fp32
__device__ __forceinline__ float fix_latent(int fmt, const uint8_t* pg, int slot, int d) {
  if (fmt == MLA_FMT_BF16) return bf16_at(pg + ((size_t)slot * DK + d) * 2);
  const int grp = d / 32;
  if (fmt == MLA_FMT_INT8)
    return (float)*reinterpret_cast<const int8_t*>(pg + I8_C_CODE + slot * DC + d) *
           bf16_at(pg + I8_C_SCALE + (slot * (DC / 32) + grp) * 2);
  const uint32_t code = (pg[I4_C_CODE + slot * (DC / 2) + d / 2] >> (4 * (d & 1))) & 0xFu;
  return fmaf((float)code, bf16_at(pg + I4_C_SCALE + (slot * (DC / 32) + grp) * 2),
              bf16_at(pg + I4_C_ZERO + (slot * (DC / 32) + grp) * 2));
}
template <int NT>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) r += red[w];
  __syncthreads();
  return r;
}
// One (row, head) over the first n > 0 tokens of page-table row pb, exactly:
// qrow is its 576-wide query, w_uv its head's W_UV [128][512]; writes out[128]
// (bf16) and, when given, o_lat[512].  Every thread of the CTA calls it (NT
// threads); scratch: 1,120 + NT floats of shared memory.
template <int NT>
__device__ __noinline__ void exact_head(const FixCtx fx, int pb, int n, const uint16_t* qrow, const uint16_t* w_uv,
                                        uint16_t* out, float* o_lat, float* scratch, int* err) {
  constexpr int DPT = (DC + NT - 1) / NT;  // latent dims per thread
  const int tid = threadIdx.x;
  float* q = scratch;          // [576]
  float* pw = q + DK;          // [NT] weights of the chunk's tokens
  float* red = pw + NT;        // [32]
  float* ol = red + 32;        // [512]
  for (int i = tid; i < DK; i += NT) q[i] = __uint_as_float((uint32_t)qrow[i] << 16);
  __syncthreads();
  float acc[DPT];
#pragma unroll
  for (int k = 0; k < DPT; ++k) acc[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int t0 = 0; t0 < n; t0 += NT) {
    const int t = t0 + tid;
    float sc = -INFINITY;
    if (t < n) {
      const uint8_t* pg = fix_page(fx, pb, t / PAGE, err);
      float dot = 0.f;
      for (int u = 0; u < DK / 8; ++u) {
        float f[8];
        fix_key_unit(fx.fmt, pg, t % PAGE, u, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) dot = fmaf(q[8 * u + k], f[k], dot);
      }
      sc = dot * fx.scale_log2;
    }
    const float m_new = fmaxf(m, block_max<NT>(sc, red));  // finite: token t0 < n is valid
    const float alpha = exp2f(m - m_new);                    // 0 at the first chunk
    const float p = t < n ? exp2f(sc - m_new) : 0.f;
    pw[tid] = p;
    l = l * alpha + block_sum<NT>(p, red);  // its barriers also publish pw
    const int cnt = min(NT, n - t0);
#pragma unroll
    for (int k = 0; k < DPT; ++k) {
      const int d = tid + k * NT;
      if (d < DC) {
        float a = acc[k] * alpha;
        const uint8_t* pg = nullptr;
        for (int j = 0; j < cnt; ++j) {
          const int tj = t0 + j;
          if (j == 0 || tj % PAGE == 0) pg = fix_page(fx, pb, tj / PAGE, err);
          a = fmaf(pw[j], fix_latent(fx.fmt, pg, tj % PAGE, d), a);
        }
        acc[k] = a;
      }
    }
    m = m_new;
    __syncthreads();  // pw is rewritten by the next chunk
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < DPT; ++k) {
    const int d = tid + k * NT;
    if (d < DC) {
      ol[d] = acc[k] * inv;
      if (o_lat != nullptr) o_lat[d] = acc[k] * inv;
    }
  }
  __syncthreads();
  for (int j = tid; j < DV; j += NT) {
    const uint4* w = reinterpret_cast<const uint4*>(w_uv + (size_t)j * DC);
    float o = 0.f;
    for (int c8 = 0; c8 < DC / 8; ++c8) {
      const uint4 v = w[c8];
      const float* x = ol + 8 * c8;
      o = fmaf(bf16lo(v.x), x[0], o); o = fmaf(bf16hi(v.x), x[1], o);
      o = fmaf(bf16lo(v.y), x[2], o); o = fmaf(bf16hi(v.y), x[3], o);
      o = fmaf(bf16lo(v.z), x[4], o); o = fmaf(bf16hi(v.z), x[5], o);
      o = fmaf(bf16lo(v.w), x[6], o); o = fmaf(bf16hi(v.w), x[7], o);
    }
    const __nv_bfloat16 ob = __float2bfloat16_rn(o);
    out[j] = *reinterpret_cast<const uint16_t*>(&ob);
  }
  __syncthreads();  // scratch reuse by the next row
}

template <int RB>
__global__ void __launch_bounds__(CombLayout<RB>::THREADS, 1)
    combine_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
                   const uint16_t* __restrict__ W_UV, int H, int B, QSpec qs,
                   const int* __restrict__ plan, const float* __restrict__ part_lse, uint16_t* __restrict__ out,
                   float* __restrict__ o_lat, int* err) {
  using L = CombLayout<RB>;
  constexpr int NW = L::NW;
  constexpr int WST = L::WST, PST = L::PST, BST = L::BST, SEGB = L::SEGB;
  constexpr uint32_t P_TILE = L::P_TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* w_full = bars;
  uint64_t* w_empty = w_full + WST;
  uint64_t* p_full = w_empty + WST;
  uint64_t* p_empty = p_full + PST;
  uint64_t* b_full = p_empty + PST;
  uint64_t* b_free = b_full + BST;
  uint64_t* d_full = b_free + BST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 12);
  float* wgt = reinterpret_cast<float*>(sm + L::OFF_WGT);

  const int h = blockIdx.x, b0 = blockIdx.y * RB;  // h: head of the partials (a virtual head)
  const int hr = h % qs.Hr;                        // its real head: the W_UV it applies
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warp NW: TMEM owner and W_UV loader; warp NW + 1: partial loader; warp
  // NW + 2: MMA issuer.  Each has a warp of its own: a lane blocked in
  // mbarrier.try_wait stalls its whole warp, and a merge warp that also issued
  // a chunk's MMAs (about 0.45 us of issue) would fall behind the others and
  // hold back the release of the partial ring, which waits for every warp
  const bool loader = warp >= NW, w_loader = warp == NW;
  // output row ((row, token) * heads + head) of plan row bv for this head; -1
  // for padding (one query token per row and pass: bv * heads + head, no division)
  const bool single = qs.NG == 1 && qs.T == 1 && qs.G == 1;
  auto out_row = [&](int bv) -> long long {
    if (single) return (long long)bv * qs.Hr + hr;
    const int t = qs.token(bv, h);
    return t < qs.T ? ((long long)(bv / qs.NG) * qs.T + t) * qs.Hr + hr : -1;
  };

  if (tid == 0) {
    for (int s = 0; s < WST; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 1);
    }
    for (int s = 0; s < PST; ++s) {
      mbar_init(&p_full[s], 1);
      mbar_init(&p_empty[s], NW);
    }
    for (int s = 0; s < BST; ++s) {
      mbar_init(&b_full[s], NW);
      mbar_init(&b_free[s], 1);
    }
    mbar_init(d_full, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (w_loader) {
    tmem_alloc(tmem_slot, L::TCOLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (w_loader && lane == 0) {
    // W_UV is a weight: its first tiles load while the attention step finishes
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_p);
    prefetch_l2_bulk(W_UV + (size_t)hr * DV * DC, DV * DC * 2);  // W_UV[hr] into L2 for the later tiles
    for (int kc = 0; kc < WST; ++kc) {
      mbar_arrive_expect_tx(&w_full[kc], W_TILE);
      tma_load_3d(sm + L::OFF_W + kc * W_TILE, &tm_w, KC * kc, 0, hr, &w_full[kc]);
    }
  }
  // ---- the slots [s_lo, s_hi) that hold every segment of the group's rows:
  // segment w + b of row b, rows and workers both increasing along the tiles.
  // The plan is read before the wait: every kernel of the decode chain waits
  // for its predecessor before it lets the next one start, so the plan kernel
  // has completed (and its writes are visible) once this grid runs at all;
  // the attention step writes only the partials, their log-sum-exps and the
  // exact-recompute flags, read after the wait.
  const long long T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  const int b_end = min(b0 + RB, B);
  const int t0 = prefix[b0], t1 = prefix[b_end];
  const int s_lo = t1 > t0 ? worker_of_tile(t0, T, W) + b0 : 0;
  const int s_hi = t1 > t0 ? worker_of_tile(t1 - 1, T, W) + b_end : 0;
  const int nsub = (s_hi - s_lo + SEGB - 1) / SEGB;  // partial tiles per chunk (0 when every row is empty)
  // this merge thread's row: its segments [rs.x, rs.y] (segment w + b of row
  // b; empty when x > y)
  const int r = tid >> 3, u = tid & 7;  // row of the group, 8-dim unit of the chunk
  const int b = b0 + r;
  int2 rs = make_int2(1, 0);
  if (!loader && b < B) {
    const int p0 = prefix[b], p1 = prefix[b + 1];
    if (p1 > p0) rs = make_int2(worker_of_tile(p0, T, W) + b, worker_of_tile(p1 - 1, T, W) + b);
  }
  grid_dep_wait();  // the partials and their log-sum-exps
  grid_dep_launch();

  if (loader) {
    // ------------------------------------------------------------ TMA loaders:
    // lane 0 of warp NW refills the W_UV ring, lane 0 of warp NW + 1 streams
    // the partial tiles
    if (w_loader && lane == 0) {
      int wi = WST;  // W tiles issued so far
      for (int kc = WST; kc < NCHUNK; ++kc, ++wi) {  // stage kc % WST was read by chunk kc - WST's MMAs
        const int st = kc % WST;
        if (!cwait(&w_empty[st], ((kc / WST) & 1) ^ 1, abort, err, 0)) break;
        mbar_arrive_expect_tx(&w_full[st], W_TILE);
        tma_load_3d(sm + L::OFF_W + st * W_TILE, &tm_w, KC * kc, 0, hr, &w_full[st]);
      }
      if (*abort)  // let copies in flight land before the CTA exits
        for (int k = max(0, wi - WST); k < wi; ++k) (void)mbar_wait(&w_full[k % WST], (k / WST) & 1);
    } else if (warp == NW + 2 && lane == 0) {
      // ---------------------------------------------------------- MMA issue
      //   D[128 out dims][RB rows] += W_UV[h][:, chunk] . hi^T + W_UV[h][:, chunk] . lo^T
      // (the 8 MMAs of a chunk take about 0.45 us to issue)
      const uint32_t idesc = idesc_bf16_f32(128, RB, false, false);
      bool final_commit = false;
      for (int kc = 0; kc < NCHUNK; ++kc) {
        const int bs = kc % BST, ws = kc % WST;
        if (!cwait(&b_full[bs], (kc / BST) & 1, abort, err, 4) || !cwait(&w_full[ws], (kc / WST) & 1, abort, err, 5))
          break;
        fence_after_sync();
        const uint32_t wa = smem_u32(sm + L::OFF_W + ws * W_TILE), ba = smem_u32(sm + L::OFF_B + bs * 2 * L::B_TILE);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int kk = 0; kk < KC / 16; ++kk)
            mma_ss(tmem, smem_desc(wa + kk * 32, 16, 1024, SWIZZLE_128B),
                   smem_desc(ba + part * L::B_TILE + kk * 32, 16, 1024, SWIZZLE_128B), idesc,
                   (kc | part | kk) != 0 ? 1u : 0u);
        mma_commit(&b_free[bs]);
        mma_commit(&w_empty[ws]);
        if (kc == NCHUNK - 1) {
          mma_commit(d_full);
          final_commit = true;
        }
      }
      if (*abort) {  // MMAs in flight finish before TMEM is freed
        if (!final_commit) mma_commit(d_full);
        (void)mbar_wait(d_full, 0);
      }
    } else if (warp == NW + 1 && lane == 0) {
      int pu = 0;  // partial tiles issued so far
      bool ok = true;
      for (int kc = 0; kc < NCHUNK && ok; ++kc) {
        for (int sub = 0; sub < nsub; ++sub, ++pu) {
          const int st = pu % PST;
          ok = cwait(&p_empty[st], ((pu / PST) & 1) ^ 1, abort, err, 1);
          if (!ok) break;
          const int nbox = (min(SEGB, s_hi - s_lo - SEGB * sub) + SBOX - 1) / SBOX;
          mbar_arrive_expect_tx(&p_full[st], (uint32_t)nbox * SBOX * KC * 2);
          for (int j = 0; j < nbox; ++j)
            tma_load_3d(sm + L::OFF_P + st * P_TILE + j * SBOX * KC * 2, &tm_p, KC * kc,
                        s_lo + SEGB * sub + SBOX * j, h, &p_full[st]);
        }
      }
      if (*abort)
        for (int k = max(0, pu - PST); k < pu; ++k) (void)mbar_wait(&p_full[k % PST], (k / PST) & 1);
    }
  } else {
    // ------------------------------------------------------------ merge warps
    const long long orow = b < B ? out_row(b) : -1;
    // ---- the row's softmax weights e^{LSE_s - LSE} into wgt, the row's 8
    // threads sharing the segments (a worker without tiles left no partial:
    // weight 0).  Slots between rows are never read.
    float mx = -INFINITY;
    for (int s = rs.x + u; s <= rs.y; s += 8) {
      const long long w = s - b;
      const float lw = worker_begin(w, T, W) == worker_begin(w + 1, T, W) ? -INFINITY : part_lse[(size_t)s * H + h];
      wgt[s - s_lo] = lw;
      mx = fmaxf(mx, lw);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
    for (int s = rs.x + u; s <= rs.y; s += 8) {
      const float lw = wgt[s - s_lo];
      const float e = lw == -INFINITY ? 0.f : expf(lw - mx);
      wgt[s - s_lo] = e;
      den += e;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int s = rs.x + u; s <= rs.y; s += 8) wgt[s - s_lo] *= inv;
    __syncwarp();  // the row's weights, written by its 8 threads (one warp)
    int pu = 0;
    bool ok = true;
    for (int kc = 0; kc < NCHUNK && ok; ++kc) {
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.f;
      for (int sub = 0; sub < nsub; ++sub, ++pu) {
        const int st = pu % PST;
        if (!cwait(&p_full[st], (pu / PST) & 1, abort, err, 2)) {
          ok = false;
          break;
        }
        const uint16_t* tile = reinterpret_cast<const uint16_t*>(sm + L::OFF_P + st * P_TILE);
        const int base = s_lo + SEGB * sub;
        const int sa = max(rs.x, base), sz = min(rs.y, base + SEGB - 1);
        for (int s0 = sa; s0 <= sz; s0 += 4) {  // four segments' loads at once
          float wv[4];
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool in = s0 + k <= sz;
            wv[k] = in ? wgt[s0 + k - s_lo] : 0.f;
            v[k] = in ? *reinterpret_cast<const uint4*>(tile + (s0 + k - base) * KC + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (wv[k] == 0.f) continue;  // a slot no worker wrote (its contents are undefined)
            const float w = wv[k];
            acc[0] = fmaf(w, bf16lo(v[k].x), acc[0]); acc[1] = fmaf(w, bf16hi(v[k].x), acc[1]);
            acc[2] = fmaf(w, bf16lo(v[k].y), acc[2]); acc[3] = fmaf(w, bf16hi(v[k].y), acc[3]);
            acc[4] = fmaf(w, bf16lo(v[k].z), acc[4]); acc[5] = fmaf(w, bf16hi(v[k].z), acc[5]);
            acc[6] = fmaf(w, bf16lo(v[k].w), acc[6]); acc[7] = fmaf(w, bf16hi(v[k].w), acc[7]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_empty[st]);
      }
      if (!ok) break;
      if (o_lat != nullptr && orow >= 0)
        st_global_v8(o_lat + orow * DC + KC * kc + 8 * u, acc[0], acc[1], acc[2], acc[3], acc[4],
                     acc[5], acc[6], acc[7]);
      // o_lat = hi + lo, both bf16, into the operand tiles of this chunk
      const int bs = kc % BST;
      if (!cwait(&b_free[bs], ((kc / BST) & 1) ^ 1, abort, err, 3)) {
        ok = false;
        break;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        hi[k] = pack2_bf16(acc[2 * k], acc[2 * k + 1]);
        const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi[k]));
        lo[k] = pack2_bf16(acc[2 * k] - hf.x, acc[2 * k + 1] - hf.y);
      }
      const uint32_t off = r * 128 + ((u ^ (r & 7)) << 4);
      uint8_t* bt = sm + L::OFF_B + bs * 2 * L::B_TILE;
      *reinterpret_cast<uint4*>(bt + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(bt + L::B_TILE + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      fence_proxy_async_smem();  // generic writes -> the tensor core's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&b_full[bs]);
    }
    // ---- epilogue: D[out dim][row] -> out[b][h][:] (bf16)
    if (ok && cwait(d_full, 0, abort, err, 6)) {
      fence_after_sync();
      const int q = warp & 3, cg = warp >> 2;  // TMEM lane quadrant (32 out dims), 16-row column group
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * cg, v);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int bb = b0 + 16 * cg + k;
        const long long ob = bb < B ? out_row(bb) : -1;
        if (ob >= 0) {
          const __nv_bfloat16 o = __float2bfloat16_rn(__uint_as_float(v[k]));
          out[ob * DV + 32 * q + lane] = *reinterpret_cast<const uint16_t*>(&o);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (w_loader) {
    fence_after_sync();
    tmem_dealloc(tmem, L::TCOLS);
  }
}

// The exact recompute as its own kernel, after the merge: one CTA per (head of
// the partials, group of 32 plan rows) reads the group's flags and leaves at
// once when none is set (the common case costs one launch of the decode
// chain); otherwise it overwrites the flagged rows' outputs (and o_lat) with
// the exact values, each virtual head over its own causal view.
template <int NT>
__global__ void __launch_bounds__(NT) fix_kernel(const uint16_t* W_UV, int H, int B, QSpec qs, const int* plan,
                                                 uint16_t* out, float* o_lat, int* err) {
  __shared__ float scratch[DK + NT + 32 + DC];
  const int h = blockIdx.x, b0 = blockIdx.y * 32, hr = h % qs.Hr;
  // The flags (and the recompute context) come from the attention step, which
  // completed before the merge let this grid start: read before the wait.  The
  // wait stays, before any exit, so that this grid's completion implies the
  // merge's (the next step's plan kernel waits for this one).
  const int* fixf = plan + plan_off_fix(B);
  const int f = (threadIdx.x < 32 && b0 + (int)threadIdx.x < B) ? fixf[b0 + threadIdx.x] : 0;
  const bool any = __syncthreads_or(f);
  grid_dep_wait();  // flagged rows overwrite the merge's outputs
  grid_dep_launch();
  if (!any) return;
  const FixCtx fx = *reinterpret_cast<const FixCtx*>(plan + PLAN_CTX);
  const int* seq_c = plan + plan_off_seq(B);
  for (int r = 0; r < 32 && b0 + r < B; ++r) {
    const int bv = b0 + r;
    const int t = qs.token(bv, h);
    if (!fixf[bv] || t >= qs.T) continue;  // uniform over the CTA
    const int n = seq_c[bv] - qs.shift(bv, h);
    if (n <= 0) continue;
    const long long orow = ((long long)(bv / qs.NG) * qs.T + t) * qs.Hr + hr;
    exact_head<NT>(fx, bv / qs.NG, n, fx.q_cat + (qs.qrow(bv) + h) * DK, W_UV + (size_t)hr * DV * DC, out + orow * DV,
                   o_lat != nullptr ? o_lat + orow * DC : nullptr, scratch, err);
  }
}

// ---------------------------------------------------------------------------
// The merge and the up-projection for few heads (the 16-head single-query
// decode): the tensor-core kernel above gives each (head, 16..32 rows) one CTA,
// only 32 CTAs for 16 heads and a 32-row batch, and its chunk loop is then
// latency-bound.  Here one CTA per (head, group of 4 rows): W_UV[h] (128 KB)
// arrives by TMA as eight 128B-swizzled [128 out dims][64 latent] tiles before
// the kernel waits for the attention step.  Each row has a quarter of the
// block (4 latent dims per thread) and merges its segments 8 at a time in
// fp32, every load of a chunk (the 8 log-sum-exps and the 8 partials) in
// flight at once, as an online softmax over the segments ("kv_budget.py" part
// C: o_lat = sum_s e^{LSE_s - LSE} o_s with LSE = log sum_s e^{LSE_s}, the
// running maximum moved per chunk).  o_lat is then split into a bf16 high part
// and a bf16 residual, written as 128B-swizzled operand rows (the group's 4,
// then zero rows) of the warp-level tensor-core MMA (mma.sync m16n8k16):
// out[b, h, :] = W_UV[h] o_lat[b, h, :] = W_UV[h] hi + W_UV[h] lo, fp32 accumulation
// (the same roundings as the tensor-core kernel: W_UV's own bf16 and the
// residual's, relative 2^-16), computed as out^T = W_UV[h] . o_lat^T so that
// the 128 out dims are the MMA's M and the 4 rows pad only to its N of 8.
// ---------------------------------------------------------------------------
constexpr int SRB = 4;      // rows per CTA
constexpr int SNT = 512;    // threads: a quarter of the block per row in the merge, 16 out dims x half the latent per warp after it
constexpr int SCH = 8;      // segments per merge chunk

struct __align__(1024) SmallSmem {
  uint8_t w[DC / 64][DV * 128];   // W_UV[h]: [128 out dims][64 latent] per 64-wide chunk, 128B-swizzled
  uint8_t a[2][DC / 64][16 * 128];  // o_lat hi / lo: [16 rows][64 latent] per chunk, 128B-swizzled
  uint64_t w_full;
};

__global__ void __launch_bounds__(SNT) combine_small_kernel(const __grid_constant__ CUtensorMap tm_w, int H, int B,
                                                            const int* __restrict__ plan, int segs,
                                                            const uint16_t* __restrict__ part_o,
                                                            const float* __restrict__ part_lse,
                                                            uint16_t* __restrict__ out, float* __restrict__ o_lat,
                                                            int* err) {
  extern __shared__ uint8_t smem_raw[];
  SmallSmem& S = *reinterpret_cast<SmallSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int h = blockIdx.x, b0 = blockIdx.y * SRB, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&S.w_full, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {  // W_UV[h] is a weight: its copy overlaps the attention step's tail
    prefetch_tmap(&tm_w);
    mbar_arrive_expect_tx(&S.w_full, DV * DC * 2);
    for (int c = 0; c < DC / 64; ++c) tma_load_3d_hint(S.w[c], &tm_w, 64 * c, 0, h, &S.w_full, policy_evict_last());
  }
  // the operand rows past the group's 4 are zeros (12 rows x 8 chunks x hi, lo)
  for (int i = tid; i < 2 * (DC / 64) * 12 * 8; i += SNT) {
    const int u = i & 7, row = 4 + (i >> 3) % 12, t = i / 96;  // t: hi/lo and chunk
    *reinterpret_cast<uint4*>(&S.a[t >> 3][t & 7][row * 128 + u * 16]) = make_uint4(0u, 0u, 0u, 0u);
  }
  // the row's segments [sx, sy] (segment w + b of row b for the workers w whose
  // ranges hold its tiles), read before the wait: every kernel of the decode
  // chain waits for its predecessor before it lets the next start, so the plan
  // kernel has completed once this grid runs
  const long long T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  const int r = tid >> 7, rt = tid & 127;  // the row of the group, latent dims 4 rt .. 4 rt + 3
  const int b = b0 + r;
  int sx = 1, sy = 0;
  if (b < B && prefix[b + 1] > prefix[b]) {
    sx = worker_of_tile(prefix[b], T, W) + b;
    sy = worker_of_tile(prefix[b + 1] - 1, T, W) + b;
  }
  grid_dep_wait();  // the partials and their log-sum-exps
  grid_dep_launch();
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (sx <= sy) {
    // a worker without tiles left no partial: weight 0, its slot's undefined
    // bits loaded with the others and discarded
    const size_t stride = DC / 4;  // one segment, in 4-value units (head-major partials)
    const uint2* po = reinterpret_cast<const uint2*>(part_o + (size_t)h * segs * DC) + rt;
    float m = -INFINITY, den = 0.f;
    for (int c0 = sx; c0 <= sy; c0 += SCH) {
      const int cn = min(SCH, sy - c0 + 1);
      float lk = -INFINITY;  // lane k < cn: the log-sum-exp of segment c0 + k
      if (lane < cn) {
        const long long w = c0 + lane - b;
        if (worker_begin(w, T, W) != worker_begin(w + 1, T, W)) lk = part_lse[(size_t)(c0 + lane) * H + h];
      }
      uint2 v[SCH];
#pragma unroll
      for (int k = 0; k < SCH; ++k) v[k] = k < cn ? po[(size_t)(c0 + k) * stride] : make_uint2(0u, 0u);
      float mc = lk;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
      const float mn = fmaxf(m, __shfl_sync(0xffffffffu, mc, 0));  // finite: the row's first segment has tiles
      const float sc = m == -INFINITY ? 0.f : expf(m - mn);
      const float e = lk == -INFINITY ? 0.f : expf(lk - mn);
      a0 *= sc; a1 *= sc; a2 *= sc; a3 *= sc; den *= sc;
#pragma unroll
      for (int k = 0; k < SCH; ++k) {
        const float ek = __shfl_sync(0xffffffffu, e, k);
        if (ek != 0.f) {
          a0 = fmaf(ek, bf16lo(v[k].x), a0);
          a1 = fmaf(ek, bf16hi(v[k].x), a1);
          a2 = fmaf(ek, bf16lo(v[k].y), a2);
          a3 = fmaf(ek, bf16hi(v[k].y), a3);
          den += ek;
        }
      }
      m = mn;
    }
    const float inv = 1.f / den;  // den >= 1: the largest term is e^0
    a0 *= inv; a1 *= inv; a2 *= inv; a3 *= inv;
  }
  if (o_lat != nullptr && b < B)
    *reinterpret_cast<float4*>(o_lat + ((size_t)b * H + h) * DC + 4 * rt) = make_float4(a0, a1, a2, a3);
  {
    // o_lat = hi + lo (both bf16) into row r of the operand tiles: dims 4 rt .. +3
    // are the half (rt & 1) of 16-byte unit (rt >> 1) & 7 of chunk rt >> 4
    const uint32_t h0 = pack_bf16x2(a0, a1), h1 = pack_bf16x2(a2, a3);
    const uint32_t l0 = pack_bf16x2(a0 - bf16lo(h0), a1 - bf16hi(h0)), l1 = pack_bf16x2(a2 - bf16lo(h1), a3 - bf16hi(h1));
    const int c = rt >> 4, u = (rt >> 1) & 7;
    const int off = r * 128 + ((u ^ r) << 4) + 8 * (rt & 1);  // rows 0..3: swizzle r & 7 = r
    *reinterpret_cast<uint2*>(&S.a[0][c][off]) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(&S.a[1][c][off]) = make_uint2(l0, l1);
  }
  __syncthreads();
  if (!mbar_wait(&S.w_full, 0)) {
    if (tid == 0) raise_error(err, MLA_ERR_TIMEOUT, 150);
    return;
  }
  // ---- out^T = W_UV[h] . hi^T + W_UV[h] . lo^T (M = 128 out dims, N = 8 rows of
  // which the group's 4, K = 512): warp w takes out dims 16 (w % 8) .. + 15 over
  // latent half w / 8, the hi and lo terms in two accumulators; the two halves
  // are added through shared memory
  const int mt = warp & 7, kh = warp >> 3;
  float dh[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int c = 4 * kh; c < 4 * kh + 4; ++c) {
    const uint32_t wb = smem_u32(S.w[c]), ah = smem_u32(S.a[0][c]), al = smem_u32(S.a[1][c]);
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
      // B: rows lane % 8 of o_lat (the 4 of the group, then zeros), latent
      // 32 kp + 8 (lane / 8) (two k-steps); A: out dims 16 mt + lane % 16,
      // latent 32 kp + 16 hk + 8 (lane / 16) of k-step hk
      uint32_t bh[4], bl[4];
      ldsm_x4(bh, ah + sw128(lane & 7, 4 * kp + (lane >> 3)));
      ldsm_x4(bl, al + sw128(lane & 7, 4 * kp + (lane >> 3)));
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        uint32_t fa[4];
        ldsm_x4(fa, wb + sw128(16 * mt + (lane & 15), 4 * kp + 2 * hk + (lane >> 4)));
        mma_bf16_16816(dh, fa, bh[2 * hk], bh[2 * hk + 1]);
        mma_bf16_16816(dl, fa, bl[2 * hk], bl[2 * hk + 1]);
      }
    }
  }
  // d[0], d[1]: out dim 16 mt + lane / 4, rows 2 (lane % 4), + 1; d[2], d[3]: out dim + 8
  float* red = reinterpret_cast<float*>(S.a[0][0]);  // [8 m-tiles][32 lanes][4]: the upper latent half
  __syncthreads();  // every warp has read the operand tiles
  if (kh == 1)
    *reinterpret_cast<float4*>(red + (mt * 32 + lane) * 4) =
        make_float4(dh[0] + dl[0], dh[1] + dl[1], dh[2] + dl[2], dh[3] + dl[3]);
  __syncthreads();
  if (kh == 0 && (lane & 3) < SRB / 2) {
    const float4 u = *reinterpret_cast<const float4*>(red + (mt * 32 + lane) * 4);
    const float o[4] = {dh[0] + dl[0] + u.x, dh[1] + dl[1] + u.y, dh[2] + dl[2] + u.z, dh[3] + dl[3] + u.w};
    const int j = 16 * mt + (lane >> 2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = 2 * (lane & 3) + (k & 1), jj = j + 8 * (k >> 1);
      if (b0 + row < B) {
        const __nv_bfloat16 ob = __float2bfloat16_rn(o[k]);
        out[((size_t)(b0 + row) * H + h) * DV + jj] = *reinterpret_cast<const uint16_t*>(&ob);
      }
    }
  }
}

template <int RB>
cudaError_t launch_rb(const CUtensorMap& tm_w, const CUtensorMap& tm_p, const void* W_UV, int H, int B, const QSpec& qs,
                      const int* plan, const float* part_lse, void* out, float* o_lat, int* err, int max_workers,
                      cudaStream_t s) {
  using L = CombLayout<RB>;
  const size_t smem = L::bytes(max_workers);
  cudaError_t e = cudaFuncSetAttribute(combine_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(combine_kernel<RB>, dim3(H, (B + RB - 1) / RB), dim3(L::THREADS), smem, s, tm_w, tm_p,
                    static_cast<const uint16_t*>(W_UV), H, B, qs, plan, part_lse, static_cast<uint16_t*>(out), o_lat,
                    err);
}

}  // namespace

cudaError_t launch_combine(const void* W_UV, int Hv, int Bv, const QSpec& qs, const int* plan, const uint16_t* part_o,
                           const float* part_lse, void* out, float* o_lat, int* err, int max_workers,
                           cudaStream_t s) {
  if (Bv == 0) return cudaSuccess;
  CUtensorMap tm_w, tm_p;  // W_UV: (512 latent, 128 rows, Hr heads), tiles of 64 x 128, 128B swizzle
  if (!encode_3d(&tm_w, W_UV, DC, DV, qs.Hr, DC * 2, (uint64_t)DV * DC * 2, 64, DV, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (Hv < 128) {
    // the 16-head single-query decode (its attend kernels compute the defined
    // softmax themselves and flag no row, so no exact-recompute pass follows)
    if (qs.T != 1 || qs.G != 1 || qs.NG != 1 || qs.Hr != Hv) return cudaErrorInvalidValue;
    const size_t smem = sizeof(SmallSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(combine_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(combine_small_kernel, dim3(Hv, (Bv + SRB - 1) / SRB), dim3(SNT), smem, s, tm_w, Hv, Bv, plan,
                      max_workers + Bv, part_o, part_lse, static_cast<uint16_t*>(out), o_lat, err);
  }
  // partials (bf16, head-major): (512 latent, segments, Hv heads), boxes of 64 dims x 64 segments x 1 head
  // (segments past the buffer read as zeros, without memory traffic)
  const uint64_t segs = (uint64_t)max_workers + Bv;
  if (!encode_3d_box(&tm_p, part_o, DC, segs, Hv, DC * 2, segs * DC * 2, KC, SBOX, 1,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
    return cudaErrorInvalidValue;
  // rows per CTA: 64 (W_UV of the head loaded whole, one CTA per SM) when one
  // wave of such CTAs covers the grid; else 32 when that still gives every SM
  // a CTA; else 16 (few heads or rows)
  const int sms = device_sm_count();
  cudaError_t e;
  if (Bv > 32 && (long long)Hv * ((Bv + 63) / 64) <= sms)
    e = launch_rb<64>(tm_w, tm_p, W_UV, Hv, Bv, qs, plan, part_lse, out, o_lat, err, max_workers, s);
  else if ((long long)Hv * ((Bv + 31) / 32) >= sms)
    e = launch_rb<32>(tm_w, tm_p, W_UV, Hv, Bv, qs, plan, part_lse, out, o_lat, err, max_workers, s);
  else
    e = launch_rb<16>(tm_w, tm_p, W_UV, Hv, Bv, qs, plan, part_lse, out, o_lat, err, max_workers, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(fix_kernel<256>, dim3(Hv, (Bv + 31) / 32), dim3(256), 0, s, static_cast<const uint16_t*>(W_UV), Hv,
                    Bv, qs, plan, static_cast<uint16_t*>(out), o_lat, err);
}

}  // namespace mla
