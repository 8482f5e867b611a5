// Split-KV absorbed decode on CUDA cores (small head counts, e.g. the
// 16-head V2-Lite layer).
//
// Computes, per split of a row's tokens, the absorbed attention of
// "DeepSeek MLA 吸收式缓存" §2.2–§2.4 over the 576-wide latent cache
// (MQA mode with key width 576 and value width 512, §6.1):
//   s_t = scale * (q_lat . c_t + q_pe . k_pe_t),  online softmax over t,
//   O   = sum_t p_t c_t,  emitted as O / l and LSE = m + ln l per head.
//
// Layout.  One CTA (256 threads) per (worker, group of 16 heads).  A worker
// walks its contiguous range of 64-token pages (see decode_plan.cu) in halves
// of 32 tokens; each half page (32 x 1152 B, contiguous in the pool) arrives
// in shared memory by one bulk async copy, double-buffered, with an L2
// evict-first hint (the cache is streamed once).
//   scores: warp w takes tokens 4w..4w+3, lane l the bf16 pairs l+32k of the
//           576-wide key; 64 partial dot products per lane are summed across
//           the warp by a halving butterfly (62 shuffles, each lane ends with
//           two finished scores);
//   softmax: warp w owns heads 2w, 2w+1, one token per lane;
//   P.V:   thread t owns latent dims 2t, 2t+1 for all 16 heads (32 fp32
//          accumulators), P read as warp-broadcast float4.
#include "mla_common.cuh"

namespace mla {
namespace {

constexpr int HG = 16;                 // heads per CTA
constexpr int HT = 32;                 // tokens per half page
constexpr int PAIRS = DK / 2;          // 288 bf16 pairs per token row
constexpr uint32_t HALF_BYTES = HT * DK * 2;  // 36,864
constexpr int THREADS = 256;

struct __align__(16) SmemCC {
  uint32_t kv[2][HT * PAIRS];   // 2 x 36,864 B
  uint32_t q[HG * PAIRS];       // 18,432 B
  float p[HT][HG];              // probabilities, token-major
  float s[HG][HT + 1];          // scores (log2 domain)
  float m[HG], l[HG], alpha[HG];
  uint64_t full[2];
};

__global__ void __launch_bounds__(THREADS, 2)
    attend_cc_kernel(const uint16_t* __restrict__ q_cat, int H, int num_pages, const uint8_t* __restrict__ pages,
                     const int32_t* __restrict__ page_table, int max_pages, int B, float scale_log2,
                     const int* __restrict__ plan, int seg_cap, uint16_t* __restrict__ part_o,
                     float* __restrict__ part_lse, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SmemCC& S = *reinterpret_cast<SmemCC*>(smem_raw);
  grid_dep_wait();  // the plan, the query and the cache may come from the kernel before this one
  grid_dep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int worker = blockIdx.x, hg = blockIdx.y;
  const int T = plan[0], W = plan[1];
  const int* prefix = plan + PLAN_HDR;
  const int* seq_c = plan + plan_off_seq(B);
  if (worker >= W) return;  // a plan may use fewer workers than this launch has CTAs
  const int x0 = (int)worker_begin(worker, T, W), x1 = (int)worker_begin(worker + 1, T, W);
  if (x0 >= x1) return;

  if (tid == 0) {
    mbar_init(&S.full[0], 1);
    mbar_init(&S.full[1], 1);
    fence_barrier_init();
  }
  // first row whose tiles contain x0
  int lo = 0, hi = B;  // prefix[lo] <= x0 < prefix[hi]
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
    const uint8_t* src = pages + (size_t)phys * PAGE_BYTES_BF16 + (size_t)c.half * HALF_BYTES;
    mbar_arrive_expect_tx(&S.full[stage], HALF_BYTES);
    bulk_g2s_hint(S.kv[stage], src, HALF_BYTES, &S.full[stage], policy);
  };

  HalfCursor cons{x0, 0, lo};
  HalfCursor prod = cons;
  if (tid == 0) issue(prod, 0);
  cursor_next(prod, prefix, seq_c, B);
  int issued = 1;

  float o[HG][2];
  int seg_b = -1;
  bool aborted = false;
  int it = 0;

  for (; cons.x < x1; ++it) {
    const int stage = it & 1;
    // prefetch the next half page into the other stage (freed by the last barrier)
    if (prod.x < x1) {
      if (tid == 0) issue(prod, stage ^ 1);
      cursor_next(prod, prefix, seq_c, B);
      ++issued;
    }
    // new row: load its 16-head query slice, reset the running state
    if (cons.b != seg_b) {
      seg_b = cons.b;
      const uint4* src = reinterpret_cast<const uint4*>(q_cat + ((size_t)seg_b * H + hg * HG) * DK);
      uint4* dst = reinterpret_cast<uint4*>(S.q);
      for (int i = tid; i < HG * DK * 2 / 16; i += THREADS) dst[i] = src[i];
      if (tid < HG) {
        S.m[tid] = -INFINITY;
        S.l[tid] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < HG; ++h) o[h][0] = o[h][1] = 0.f;
    }
    const int valid = page_valid(prefix, seq_c, cons.b, cons.x);
    const int nvalid = cons.half == 0 ? min(HT, valid) : valid - HT;

    const bool ok = mbar_wait(&S.full[stage], (it >> 1) & 1);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) raise_error(err, MLA_ERR_TIMEOUT, worker);
      aborted = true;
      break;
    }
    const uint32_t* kv = S.kv[stage];

    // ---- scores: 16 heads x 4 tokens per warp --------------------------------
    {
      float v[HG * 4];
#pragma unroll
      for (int i = 0; i < HG * 4; ++i) v[i] = 0.f;
#pragma unroll 3
      for (int k = 0; k < PAIRS / 32; ++k) {
        const int j = lane + 32 * k;
        float kx[4], ky[4];
#pragma unroll
        for (int tk = 0; tk < 4; ++tk) {
          const uint32_t w = kv[(warp * 4 + tk) * PAIRS + j];
          kx[tk] = bf16lo(w);
          ky[tk] = bf16hi(w);
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const uint32_t qw = S.q[h * PAIRS + j];
          const float qx = bf16lo(qw), qy = bf16hi(qw);
#pragma unroll
          for (int tk = 0; tk < 4; ++tk) v[h * 4 + tk] = fmaf(qx, kx[tk], fmaf(qy, ky[tk], v[h * 4 + tk]));
        }
      }
      // halving butterfly: lane L ends with entries 2L and 2L+1
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int off = 16 >> step, half = 32 >> step;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      const int h = lane >> 1, tk0 = 2 * (lane & 1);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = warp * 4 + tk0 + r;
        S.s[h][tok] = tok < nvalid ? v[r] * scale_log2 : -INFINITY;
      }
    }
    __syncthreads();

    // ---- online softmax: warp w owns heads 2w, 2w+1 ---------------------------
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = 2 * warp + r;
      const float sv = S.s[h][lane];
      float mt = sv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_old = S.m[h];
      const float m_new = fmaxf(m_old, mt);
      const float p = lane < nvalid ? exp2f(sv - m_new) : 0.f;
      float sum = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      S.p[lane][h] = p;
      __syncwarp();
      if (lane == 0) {
        const float a = exp2f(m_old - m_new);
        S.alpha[h] = a;
        S.l[h] = S.l[h] * a + sum;
        S.m[h] = m_new;
      }
    }
    __syncthreads();

    // ---- O = alpha * O + P . V_c ---------------------------------------------
    {
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float a = S.alpha[h];
        o[h][0] *= a;
        o[h][1] *= a;
      }
      for (int tk = 0; tk < nvalid; ++tk) {
        const uint32_t w = kv[tk * PAIRS + tid];
        const float vx = bf16lo(w), vy = bf16hi(w);
        const float4* pr = reinterpret_cast<const float4*>(S.p[tk]);
#pragma unroll
        for (int q4 = 0; q4 < HG / 4; ++q4) {
          const float4 p4 = pr[q4];
          o[4 * q4 + 0][0] = fmaf(p4.x, vx, o[4 * q4 + 0][0]);
          o[4 * q4 + 0][1] = fmaf(p4.x, vy, o[4 * q4 + 0][1]);
          o[4 * q4 + 1][0] = fmaf(p4.y, vx, o[4 * q4 + 1][0]);
          o[4 * q4 + 1][1] = fmaf(p4.y, vy, o[4 * q4 + 1][1]);
          o[4 * q4 + 2][0] = fmaf(p4.z, vx, o[4 * q4 + 2][0]);
          o[4 * q4 + 2][1] = fmaf(p4.z, vy, o[4 * q4 + 2][1]);
          o[4 * q4 + 3][0] = fmaf(p4.w, vx, o[4 * q4 + 3][0]);
          o[4 * q4 + 3][1] = fmaf(p4.w, vy, o[4 * q4 + 3][1]);
        }
      }
    }

    HalfCursor nxt = cons;
    cursor_next(nxt, prefix, seq_c, B);
    // end of this row's segment: emit O / l and the natural-log LSE
    if (nxt.x >= x1 || nxt.b != cons.b) {
      const int seg = worker + cons.b;
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float inv = 1.f / S.l[h];
        reinterpret_cast<uint32_t*>(part_o + ((size_t)(hg * HG + h) * seg_cap + seg) * DC)[tid] =
            pack_bf16x2(o[h][0] * inv, o[h][1] * inv);  // partials are stored in bf16
      }
      if (tid < HG)
        part_lse[(size_t)seg * H + hg * HG + tid] = (S.m[tid] + log2f(S.l[tid])) * 0.69314718055994531f;
    }
    cons = nxt;
    __syncthreads();  // stage and score buffers free for reuse
  }

  if (aborted && tid == 0) {
    // let the copies still in flight (iterations it .. issued-1) land before
    // the CTA exits; each wait is bounded
    for (int k = it; k < issued; ++k) (void)mbar_wait(&S.full[k & 1], (k >> 1) & 1);
  }
}

}  // namespace

int attend_cc_workers(int num_sms) { return 2 * num_sms; }

cudaError_t launch_attend_cc(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                             const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                             int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s) {
  if (fmt != MLA_FMT_BF16) return cudaErrorNotSupported;
  const size_t smem = sizeof(SmemCC);
  cudaError_t e = cudaFuncSetAttribute(attend_cc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attend_cc_kernel, dim3(workers, H / HG), dim3(THREADS), smem, s,
                    static_cast<const uint16_t*>(q_cat), H, num_pages, static_cast<const uint8_t*>(pages), page_table,
                    max_pages, B, scale * 1.4426950408889634f, plan, seg_cap, part_o, part_lse, err);
}

}  // namespace mla
