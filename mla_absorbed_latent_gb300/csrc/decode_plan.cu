// Split-KV plan for one decode step, computed on the device from the
// sequence lengths (no host round trip, so the step stays asynchronous).
//
// Every row's sequence is cut into 64-token tiles (one cache page each).  The
// tiles of all rows, in row order, form one global list of T tiles which is
// cut into `workers` contiguous, near-equal ranges, one per persistent CTA
// (or CTA pair) of the attend kernel: worker w owns tiles
// [floor(w*T/W), floor((w+1)*T/W)).  A worker whose range crosses row
// boundaries emits one partial (segment) per row it touches; segment (w, b)
// is stored at index w + b, which is unique because ranges are ordered.
// Ragged batches therefore cost the same per SM as uniform ones.
#include "mla_common.cuh"

namespace mla {
namespace {

constexpr int SMEM_ROWS = 8192;  // rows whose tile prefix the worker search reads from shared memory

// B: plan rows (virtual rows); their lengths come from the real rows' lengths
// and the query layout qs (one query token per row: the lengths themselves)
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seqlens, int B, QSpec qs,
                                                     int max_pages, int workers, int* __restrict__ plan, int* err) {
  __shared__ int warp_sums[32];
  __shared__ int s_prefix[SMEM_ROWS + 1];
  const bool in_smem = B <= SMEM_ROWS;
  grid_dep_wait();  // earlier work may still write the lengths or read this plan
  grid_dep_launch();
  const int tid = threadIdx.x;
  const int per = (B + blockDim.x - 1) / blockDim.x;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  const long long cap = (long long)max_pages * PAGE;
  int* prefix = plan + PLAN_HDR;
  int* seq_c = plan + plan_off_seq(B);
  int* fix = plan + plan_off_fix(B);

  int local = 0, first_n = 0;  // first_n: the clamped length of row lo (one row per thread when B <= 1024)
  for (int b = lo; b < hi; ++b) {
    const int br = b / qs.NG;  // the real row
    long long n = seqlens[br];
    if (n < 0 || n > cap) {
      raise_error(err, MLA_ERR_BOUNDS, br);
      n = n < 0 ? 0 : cap;
    }
    if (qs.T > 1) {
      // the row's last T tokens are its queries; this virtual row's view ends
      // with its last query token's
      if (n < qs.T) raise_error(err, MLA_ERR_BOUNDS, br);
      n -= qs.T - 1 - qs.last_token(b);
      if (n < 0) n = 0;
    }
    seq_c[b] = (int)n;
    fix[b] = 0;
    if (b == lo) first_n = (int)n;
    local += (int)((n + PAGE - 1) / PAGE);
  }
  // block-wide exclusive scan of the per-thread tile counts
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x / 32) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? warp_sums[warp - 1] : 0);
  for (int b = lo; b < hi; ++b) {
    prefix[b] = run;
    if (in_smem) s_prefix[b] = run;
    run += ((b == lo ? first_n : seq_c[b]) + PAGE - 1) / PAGE;
  }
  if (tid == blockDim.x - 1) {
    prefix[B] = run;
    if (in_smem) s_prefix[B] = run;
    plan[0] = run;
    plan[1] = workers;
    plan[2] = B;
    plan[3] = 0;
  }
  __syncthreads();  // the prefix is complete (block-wide visibility of the global writes)
  // first row of each worker's range: the largest b with prefix[b] <= its first
  // tile (so a worker starts its cursor with one load instead of a search)
  const int* pf = in_smem ? s_prefix : prefix;
  int* wrow = plan + plan_off_wrow(B);
  const long long T = pf[B];
  for (int w = tid; w < workers; w += blockDim.x) {
    const long long x = worker_begin(w, T, workers);
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pf[mid] <= x) lo = mid; else hi = mid;
    }
    wrow[w] = lo;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seqlens, int B, const QSpec& qs, int max_pages, int workers, int* plan,
                        int* err, cudaStream_t s) {
  return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s, seqlens, B * qs.NG, qs, max_pages, workers, plan, err);
}

}  // namespace mla
