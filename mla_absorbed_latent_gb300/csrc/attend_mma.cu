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
// block of the cache is B, with no padding rows.
//
// Layout.  One CTA (288 threads, 9 warps) per (worker, group of 16 heads), two
// CTAs per SM.  A worker walks its contiguous range of 64-token pages (see
// decode_plan.cu) in halves of 32 tokens; each half page arrives by TMA as
// nine [32 tokens][64 dims] boxes with the 128-byte swizzle, double-buffered,
// L2 evict-first.  Per half page:
//   scores   warp c (0..8) owns key dims [64c, 64c+64) (box c): its 16-head x
//            64-dim slice of the query sits in registers as A fragments for
//            the whole segment, and it multiplies it with all 32 tokens of its
//            box (4 token tiles x 4 k-steps, B fragments by ldmatrix); the nine
//            partial score tiles meet in shared memory;
//   softmax  16 threads per head (warps 0..7, two heads each) add the nine
//            partials, mask, and run the online softmax in fp32 with a rescale
//            at every new maximum (as the pages' online softmax does), P in bf16;
//   P.V      warp w (0..7) owns latent dims [64w, 64w+64) of O (16 heads x 64
//            fp32 in registers): 8 dim tiles x 2 token k-steps, P as the A
//            operand (ldmatrix), the box as B (ldmatrix.trans).
// Every byte of a stage is read from shared memory once for the scores and
// the latent part once more for P.V.
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int MH = 16;                     // heads per CTA (the MMA's M)
constexpr int MT = 32;                     // tokens per half page
constexpr int NBOX = DK / 64;              // 9 boxes of 64 key dims
constexpr int MTHREADS = 32 * NBOX;        // 288
constexpr uint32_t BOX_BYTES = MT * 128;   // 4 KB: 32 rows of 64 bf16
constexpr uint32_t HALF_PAGE = NBOX * BOX_BYTES;  // 36,864
constexpr int RED_LD = MT + 8;             // fp32 row pitch of a partial score tile
constexpr int P_LD = MT + 8;               // bf16 row pitch of the P tile (80 B: conflict-free ldmatrix)

struct __align__(1024) SmemMMA {
  uint8_t kv[2][NBOX][BOX_BYTES];          // 73,728 B, 128B-swizzled boxes
  float red[NBOX][MH][RED_LD];             // partial scores of the nine boxes
  uint16_t p[MH][P_LD];                    // P (bf16), the A operand of P.V
  float alpha[MH];                         // rescale factor of this half page
  float lfin[MH];                          // l of each head at a segment's end
  uint64_t full[2];
};

// --- warp-level MMA and shared-memory matrix loads (PTX ISA: mma.sync,
// ldmatrix).  Fragment layouts of m16n8k16 with g = lane / 4, t = lane % 4:
//   A (16 x 16, row-major): {a0a1, a2a3, a4a5, a6a7} = rows g, g+8, g, g+8 at
//       columns 2t..2t+1, 2t..2t+1, 2t+8..2t+9, 2t+8..2t+9
//   B (16 x 8, column-major): {b0b1, b2b3} = rows 2t..2t+1, 2t+8..2t+9 of column g
//   C (16 x 8 fp32): {c0, c1, c2, c3} = (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// byte offset of the 16-byte chunk `chunk` (8 dims) of token row r in a
// 128B-swizzled box: chunk position j ^ (r mod 8)
__device__ __forceinline__ uint32_t sw128(int r, int chunk) { return (uint32_t)r * 128u + ((uint32_t)(chunk ^ (r & 7)) << 4); }

__global__ void __launch_bounds__(MTHREADS, 2)
    attend_mma_kernel(const __grid_constant__ CUtensorMap tm_kv, const uint16_t* __restrict__ q_cat, int H,
                      int num_pages, const int32_t* __restrict__ page_table, int max_pages, int B, float scale_log2,
                      const int* __restrict__ plan, uint16_t* __restrict__ part_o, float* __restrict__ part_lse,
                      int* err) {
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
    mbar_init(&S.full[0], 1);
    mbar_init(&S.full[1], 1);
    fence_barrier_init();
  }
  int lo = 0, hi = B;  // first row whose tiles contain x0: prefix[lo] <= x0 < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x0) lo = mid; else hi = mid;
  }
  __syncthreads();

  const uint64_t policy = policy_evict_first();
  auto issue = [&](const HalfCursor& c, int stage) {
    const int j = c.x - prefix[c.b];
    int phys = page_table[(size_t)c.b * max_pages + j];
    if (phys < 0 || phys >= num_pages) {
      raise_error(err, MLA_ERR_BOUNDS, phys);
      phys = 0;
    }
    mbar_arrive_expect_tx(&S.full[stage], HALF_PAGE);
#pragma unroll 1
    for (int c9 = 0; c9 < NBOX; ++c9)
      tma_load_3d_hint(S.kv[stage][c9], &tm_kv, 64 * c9, MT * c.half, phys, &S.full[stage], policy);
  };

  HalfCursor cons{x0, 0, lo};
  HalfCursor prod = cons;
  if (tid == 0) issue(prod, 0);
  cursor_next(prod, prefix, seq_c, B);
  int issued = 1;

  // the score role: this warp's box, its query slice as A fragments
  const int box = warp;
  uint32_t qa[4][4];
  // the softmax role (warps 0..7): head sh, tokens 2 st, 2 st + 1
  const int sh = 2 * warp + (lane >> 4), st = lane & 15;
  float m_run = -INFINITY, l_run = 0.f;
  // the P.V role (warps 0..7): O of heads g, g+8 over dims 64 warp + 8 j + 2 t, +1
  float o[8][4];

  int seg_b = -1;
  bool aborted = false;
  int it = 0;
  for (; cons.x < x1; ++it) {
    const int stage = it & 1;
    // prefetch the next half page into the other stage (its last reads ended at
    // the closing barrier of the previous iteration)
    if (prod.x < x1) {
      if (tid == 0) issue(prod, stage ^ 1);
      cursor_next(prod, prefix, seq_c, B);
      ++issued;
    }
    if (cons.b != seg_b) {
      // new row: this warp's query slice into A fragments, running state reset
      seg_b = cons.b;
      const uint32_t* q = reinterpret_cast<const uint32_t*>(q_cat + ((size_t)seg_b * H + hg * MH) * DK);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int d = 64 * box + 16 * kk + 2 * t;  // even: a bf16 pair
        qa[kk][0] = q[(g * DK + d) >> 1];
        qa[kk][1] = q[((g + 8) * DK + d) >> 1];
        qa[kk][2] = q[(g * DK + d + 8) >> 1];
        qa[kk][3] = q[((g + 8) * DK + d + 8) >> 1];
      }
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    }
    const int valid = page_valid(prefix, seq_c, cons.b, cons.x);
    const int nvalid = cons.half == 0 ? min(MT, valid) : valid - MT;  // >= 1
    HalfCursor nxt = cons;
    cursor_next(nxt, prefix, seq_c, B);
    const bool seg_end = nxt.x >= x1 || nxt.b != cons.b;

    const bool ok = mbar_wait(&S.full[stage], (it >> 1) & 1);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) raise_error(err, MLA_ERR_TIMEOUT, worker);
      aborted = true;
      break;
    }
    const uint32_t kvs = smem_u32(S.kv[stage][0]);

    // ---- partial scores of box `box`: 16 heads x 32 tokens over 64 dims -------
    {
      const uint32_t bb = kvs + box * BOX_BYTES;
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int kp = 0; kp < 2; ++kp) {
          // tokens 8n..8n+7; matrices: dims 32kp + 8m, m = 0..3 (two k-steps)
          uint32_t b[4];
          const int r = 8 * n + (lane & 7);
          ldsm_x4(b, bb + sw128(r, 4 * kp + (lane >> 3)));
          mma_bf16_16816(acc[n], qa[2 * kp], b[0], b[1]);
          mma_bf16_16816(acc[n], qa[2 * kp + 1], b[2], b[3]);
        }
      }
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        *reinterpret_cast<float2*>(&S.red[box][g][8 * n + 2 * t]) = make_float2(acc[n][0], acc[n][1]);
        *reinterpret_cast<float2*>(&S.red[box][g + 8][8 * n + 2 * t]) = make_float2(acc[n][2], acc[n][3]);
      }
    }
    __syncthreads();

    if (warp < 8) {
      // ---- online softmax of head sh over tokens 2st, 2st+1 --------------------
      float2 s = make_float2(0.f, 0.f);
#pragma unroll
      for (int c9 = 0; c9 < NBOX; ++c9) {
        const float2 v = *reinterpret_cast<const float2*>(&S.red[c9][sh][2 * st]);
        s.x += v.x;
        s.y += v.y;
      }
      // tokens past the sequence end: their rows hold whatever the page slot
      // held, so the score is replaced, not combined
      s.x = 2 * st < nvalid ? s.x * scale_log2 : -INFINITY;
      s.y = 2 * st + 1 < nvalid ? s.y * scale_log2 : -INFINITY;
      float mt = fmaxf(s.x, s.y);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m_run, mt);  // finite: every half page holds a token
      const float alpha = exp2f(m_run - m_new);
      const float p0 = exp2f(s.x - m_new), p1 = exp2f(s.y - m_new);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      *reinterpret_cast<uint32_t*>(&S.p[sh][2 * st]) = pack_bf16x2(p0, p1);
      if (st == 0) {
        S.alpha[sh] = alpha;
        if (seg_end) {
          S.lfin[sh] = l_run;
          part_lse[(size_t)(worker + cons.b) * H + hg * MH + sh] = (m_run + log2f(l_run)) * 0.69314718055994531f;
        }
      }
    } else if (nvalid < MT) {
      // ---- warp 8: value rows past the sequence end to zero (p = 0 there, but
      // 0 x NaN is NaN); every score read of this stage is done
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const int nz = (MT - nvalid) * 8;  // 16-byte units per box
      for (int k = lane; k < 8 * nz; k += 32) {
        const int c8 = k / nz, u = k - c8 * nz;
        *reinterpret_cast<uint4*>(S.kv[stage][c8] + (size_t)nvalid * 128 + (size_t)u * 16) = z;
      }
      fence_proxy_async_smem();  // the next TMA copy into this stage comes after these writes
    }
    __syncthreads();

    if (warp < 8) {
      // ---- O = alpha O + P . V over this warp's 64 latent dims ------------------
      const float ag = S.alpha[g], ag8 = S.alpha[g + 8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j][0] *= ag;
        o[j][1] *= ag;
        o[j][2] *= ag8;
        o[j][3] *= ag8;
      }
      const uint32_t vb = kvs + warp * BOX_BYTES;
      const uint32_t pb = smem_u32(&S.p[0][0]);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4];
        ldsm_x4(pa, pb + (uint32_t)((lane & 15) * P_LD + 16 * kk + 8 * (lane >> 4)) * 2u);
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          // matrices: tokens 16kk + 8(m & 1) + 0..7 at dims 16jp + 8(m >> 1) + 0..7
          uint32_t b[4];
          const int m = lane >> 3, r = 16 * kk + 8 * (m & 1) + (lane & 7);
          ldsm_x4_trans(b, vb + sw128(r, 2 * jp + (m >> 1)));
          mma_bf16_16816(o[2 * jp], pa, b[0], b[1]);
          mma_bf16_16816(o[2 * jp + 1], pa, b[2], b[3]);
        }
      }
      if (seg_end) {
        const float ig = 1.f / S.lfin[g], ig8 = 1.f / S.lfin[g + 8];
        const size_t seg = (size_t)(worker + cons.b);
        uint16_t* dst = part_o + (seg * H + hg * MH) * DC + 64 * warp + 2 * t;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          *reinterpret_cast<uint32_t*>(dst + (size_t)g * DC + 8 * j) = pack_bf16x2(o[j][0] * ig, o[j][1] * ig);
          *reinterpret_cast<uint32_t*>(dst + (size_t)(g + 8) * DC + 8 * j) = pack_bf16x2(o[j][2] * ig8, o[j][3] * ig8);
        }
      }
    }
    cons = nxt;
    __syncthreads();  // stage, partial scores and P free for reuse
  }

  if (aborted && tid == 0) {
    // let the copies still in flight land before the CTA exits (bounded waits)
    for (int k = it; k < issued; ++k) (void)mbar_wait(&S.full[k & 1], (k >> 1) & 1);
  }
}

}  // namespace

int attend_mma_workers(int num_sms) { return 2 * num_sms; }

cudaError_t launch_attend_mma(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                              const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                              int workers, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s) {
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
                    scale * 1.4426950408889634f, plan, part_o, part_lse, err);
}

}  // namespace mla
