// Shared definitions of the CUDA side of libmla: dimensions, the decode
// workspace layout, the device error word, and thin inline-PTX wrappers for
// mbarriers and bulk async copies (sm_90+ forms, used on sm_103a).
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/mla.h"

namespace mla {

constexpr int DC = MLA_D_C;        // 512
constexpr int DR = MLA_D_R;        // 64
constexpr int DK = DC + DR;        // 576: key width of the absorbed (MQA-style) attention
constexpr int DN = MLA_D_NOPE;     // 128
constexpr int DV = MLA_D_V;        // 128
constexpr int PAGE = MLA_PAGE;     // 64 tokens per page

constexpr size_t PAGE_BYTES_BF16 = (size_t)PAGE * DK * 2;                       // 73,728
constexpr size_t PAGE_BYTES_INT8 = (size_t)PAGE * (DC + DR + 2 * 16 + 2 * 8);   // 39,936
constexpr size_t PAGE_BYTES_INT4 = (size_t)PAGE * (DC / 2 + DR + 4 * 16 + 2 * 8);  // 25,600

// the page layout (and decode kernel) a cache format uses: the per-token INT8
// quantizer writes INT8 pages, the symmetric INT4 latent and the INT4 RoPE key
// quantizers INT4 pages
__host__ __device__ constexpr int layout_fmt(int fmt) {
  return fmt == MLA_FMT_INT8_TOKEN ? MLA_FMT_INT8 : (fmt == MLA_FMT_INT4_SYM || fmt == MLA_FMT_INT4_PE4) ? MLA_FMT_INT4 : fmt;
}

// section offsets inside a quantized page
constexpr int I8_C_CODE = 0, I8_PE_CODE = 32768, I8_C_SCALE = 36864, I8_PE_SCALE = 38912;
constexpr int I4_C_CODE = 0, I4_PE_CODE = 16384, I4_C_SCALE = 20480, I4_C_ZERO = 22528,
              I4_PE_SCALE = 24576;

// device error word: [0] = first mla_status_t recorded, [1] = detail
__device__ __forceinline__ void raise_error(int* err, int code, int info) {
  if (err != nullptr && atomicCAS(err, 0, code) == 0) {
    atomicExch(err + 1, info);
  }
}

// ---------------------------------------------------------------------------
// decode workspace: [q_cat bf16 B*H*576][plan int32][partial O bf16][partial lse fp32].
// The partial O is head-major, bf16 [heads][max_segments][512] (segment s of
// head h at (h * max_segments + s) * 512): the merge of a head reads its rows'
// segments from one contiguous block; the partial LSE is fp32
// [max_segments][heads].
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t q_cat, plan, part_o, part_lse, total;
  int max_segments;
};

// plan block (int32):
//   [0] total tiles, [1] workers, [2] B, [3] reserved,
//   [4 .. 14)  the exact-recompute context (FixCtx, written by the tcgen05 attend kernel),
//   [PLAN_HDR .. +B+1)      tile prefix (B+1 entries),
//   then B clamped sequence lengths,
//   then B exact-recompute flags (zeroed by the plan, set by the attend kernel for a row
//        whose weights it could not form exactly; the combine kernel recomputes it),
//   then W first rows, one per worker's tile range.
constexpr int PLAN_HDR = 20;
constexpr int PLAN_CTX = 4;  // int offset of the FixCtx record (byte offset 16: 8-byte aligned)
__host__ __device__ constexpr int plan_off_seq(int B) { return PLAN_HDR + B + 1; }
__host__ __device__ constexpr int plan_off_fix(int B) { return PLAN_HDR + 2 * B + 1; }
__host__ __device__ constexpr int plan_off_wrow(int B) { return PLAN_HDR + 3 * B + 1; }
__host__ __device__ constexpr long long plan_ints(int B, int W) { return (long long)PLAN_HDR + 3LL * B + 1 + W; }

// Several query tokens per row ("手搓 MLA" §四 with its query-token axis t;
// causal as in "DeepSeek MLA 吸收式缓存" §3.4's prefill and incremental decode):
// row b holds n_b cached tokens whose last T are its queries, and query t sees
// tokens 0 .. n_b - T + t.  The attend kernel's MMA has 128 rows, so G = 128 / Hr
// query tokens of a row share one pass over its cache (a "virtual row" of G
// tokens x Hr heads = 128 virtual heads, virtual head v = token (v / Hr) of the
// group, head v % Hr); NG = ceil(T / G) virtual rows per row.  A virtual row's
// length is that of its last token's view; each virtual head sees a prefix of
// it (shorter by the tokens after its own query), and virtual heads past T are
// padding (they see nothing).  One query token per row is T = G = NG = 1 with
// Hr = 128, or the H = 16 CUDA-core path.
struct QSpec {
  int T, G, NG, Hr;
  // flat q_cat row ([B][T][Hr][576] bf16) of virtual row r's first virtual head
  __host__ __device__ __forceinline__ long long qrow(int r) const {
    return ((long long)(r / NG) * T + (long long)(r % NG) * G) * Hr;
  }
  // query token (0 .. T-1, or >= T for padding) of virtual head v of virtual row r
  __host__ __device__ __forceinline__ int token(int r, int v) const { return (r % NG) * G + v / Hr; }
  // the last query token of virtual row r
  __host__ __device__ __forceinline__ int last_token(int r) const {
    const int e = (r % NG) * G + G;
    return (e < T ? e : T) - 1;
  }
  // tokens of virtual row r's view that virtual head v does not see (huge for padding)
  __host__ __device__ __forceinline__ int shift(int r, int v) const {
    const int t = token(r, v), tl = last_token(r);
    return t <= tl ? tl - t : (1 << 30);
  }
};
__host__ __device__ inline QSpec qspec_single(int H) { return QSpec{1, 1, 1, H}; }

// What the combine kernel needs to recompute a flagged row from the cache: the
// attend kernel's cache, page table, query operand, scale and query layout.
struct FixCtx {
  const uint8_t* pages;
  const int32_t* page_table;
  const uint16_t* q_cat;  // flat rows of 576 bf16: q_lat then q_pe
  int max_pages, num_pages, fmt;
  float scale_log2;       // softmax scale times log2(e)
  QSpec qs;
};
static_assert(sizeof(FixCtx) <= (PLAN_HDR - PLAN_CTX) * 4, "FixCtx fits the plan header");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bv plan rows (virtual rows), Hv heads of the partials, q_rows flat query rows
inline WsLayout ws_layout_q(int Bv, int Hv, long long q_rows, int max_workers) {
  WsLayout L;
  size_t off = 0;
  L.q_cat = off;
  off = align_up(off + (size_t)q_rows * DK * 2, 1024);
  L.plan = off;
  off = align_up(off + (size_t)plan_ints(Bv, max_workers) * 4, 1024);
  L.max_segments = max_workers + Bv;
  L.part_o = off;
  off = align_up(off + (size_t)L.max_segments * Hv * DC * 2, 1024);  // bf16 partials
  L.part_lse = off;
  off = align_up(off + (size_t)L.max_segments * Hv * 4, 1024);
  L.total = off;
  return L;
}
inline WsLayout ws_layout(int B, int H, int max_workers) { return ws_layout_q(B, H, (long long)B * H, max_workers); }

// Largest worker count <= want whose decode workspace for B rows and H heads
// fits in cap bytes; 0 when even one worker does not fit.
inline int fitting_workers(int B, int H, int want, size_t cap) {
  if (want < 1) return 0;
  if (ws_layout(B, H, want).total <= cap) return want;
  if (ws_layout(B, H, 1).total > cap) return 0;
  int lo = 1, hi = want;  // layout(lo) fits, layout(hi) does not
  while (hi - lo > 1) {
    const int mid = lo + (hi - lo) / 2;
    if (ws_layout(B, H, mid).total <= cap) lo = mid; else hi = mid;
  }
  return lo;
}

// worker that owns global tile x when T tiles are cut into W contiguous ranges
// [floor(w*T/W), floor((w+1)*T/W))
__host__ __device__ __forceinline__ int worker_of_tile(long long x, long long T, long long W) {
  return (int)(((x + 1) * W + T - 1) / T - 1);
}
__host__ __device__ __forceinline__ long long worker_begin(long long w, long long T, long long W) {
  return (w * T) / W;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A bounded wait gives up after this long (far above any legal wait).
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with `parity` to complete; false after WAIT_LIMIT_NS.
// (the polling loop out of line: call sites stay small, most waits end at the
// first probe)
__device__ __noinline__ static bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity);
}

// 1-D bulk async copy global -> shared, completion counted on `bar` (bytes),
// with an L2 cache policy.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// host-side launchers (one per translation unit)
// ---------------------------------------------------------------------------
cudaError_t launch_absorb_weights(const void* wkv_b, int H, void* W_UK, void* W_UV, cudaStream_t s);
cudaError_t launch_cache_append(int fmt, int num_pages, void* pages, const void* c_kv, const void* k_pe,
                                const int32_t* page_table, int max_pages, const int32_t* pos, int B, int T,
                                int* err, cudaStream_t s);
// fused producer of the cache payload (cache_project.cu): down-projection on the
// tensor cores, RMSNorm, RoPE, page write; ksplit pairs per 128-token tile
cudaError_t launch_cache_project(const void* x, int hidden, const void* wkv_a, const void* kv_norm_w, float eps,
                                 float rope_theta, int fmt, int num_pages, void* pages, const int32_t* page_table,
                                 int max_pages, const int32_t* pos, int B, int T, void* latent_out, int ksplit,
                                 bool small, void* workspace, int* err, cudaStream_t s);
// CTA pairs per token tile that the producer uses (`requested` > 0 forces it, capped at hidden/64)
int project_splits(long long ntok, int hidden, int sms, int requested);
// workspace of the producer for ntok tokens and ksplit pairs per tile (0 when ksplit is 1)
size_t project_workspace_bytes(long long ntok, int ksplit);
// at most 64 tokens (small = true above): the warp-level projection's slices of
// the hidden dimension per 64-column group, and its workspace (one fp32
// partial payload per slice and token)
constexpr int PROJECT_SMALL_TOKENS = 64;
int project_small_splits(int hidden, int sms);
size_t project_small_workspace_bytes(long long ntok, int ksplit);
// after_plan: launched right after the plan kernel of the same decode (the
// fused entry points), so the kernel need not wait for it before it starts
cudaError_t launch_q_absorb(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* q_cat,
                            bool after_plan, cudaStream_t s);
// B real rows, query layout qs (B * qs.NG plan rows)
cudaError_t launch_plan(const int32_t* seqlens, int B, const QSpec& qs, int max_pages, int workers, int* plan,
                        int* err, cudaStream_t s);
cudaError_t launch_attend_cc(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                             const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                             int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s);
int attend_cc_workers(int num_sms);
cudaError_t launch_attend_mma(const void* q_cat, int H, int fmt, int num_pages, const void* pages,
                              const int32_t* page_table, int max_pages, int B, float scale, const int* plan,
                              int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s);
int attend_mma_workers(int num_sms);
// Bv virtual rows of the query layout qs (q_cat: Bv / qs.NG * qs.T * qs.Hr flat rows)
cudaError_t launch_attend_tc(const void* q_cat, const QSpec& qs, int fmt, int num_pages, const void* pages,
                             const int32_t* page_table, int max_pages, int Bv, float scale, int* plan,
                             int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s);
int attend_tc_workers(int num_sms);
// a CTA pair whose bounded wait runs out on purpose (see mla_wait_selftest)
cudaError_t launch_wait_selftest(int* err, cudaStream_t s);
// library-internal accessors (defined in mla_api.cu)
int* device_error_word();            // this device's error word, nullptr on failure
int device_sm_count();               // SMs of the current device, 0 on failure
int attend_kernel_kind(int H, int fmt);  // an mla_kernel_t value, -1 = unsupported
int attend_workers(int kind, int sms);   // persistent workers of that kernel
// the single-query attend step with the kernel `kind` (B rows, H heads)
cudaError_t launch_attend_kind(int kind, const void* q_cat, int H, const mla_cache_t* cache,
                               const int32_t* page_table, int max_pages, int B, float scale, int* plan, int workers,
                               int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s);

// Hv heads of the partials (virtual heads), Bv plan rows, query layout qs;
// unabsorbed causal prefill (prefill.cu): expand the rows' latents into per-head
// keys and values in the workspace, then flash attention over them
size_t prefill_workspace_bytes(int B, int H, int max_pages);
cudaError_t launch_prefill(const void* q_nope, const void* q_pe, const void* wkv_b, int H, int T, int num_pages,
                           const void* pages, const int32_t* page_table, int max_pages, const int32_t* seqlens, int B,
                           float scale, void* workspace, void* out, int* err, cudaStream_t s);
// the output projection after W_UV (out_proj.cu): y [R][hidden] = o [R][K] . W_O^T
int out_proj_splits(int R, int K, int hidden, int sms);
size_t out_proj_workspace_bytes(int R, int K, int hidden, int sms);
cudaError_t launch_out_proj(const void* o, const void* W_O, int R, int K, int hidden, void* y, void* workspace,
                            int* err, cudaStream_t s);
// max_workers: the partial buffer holds max_workers + Bv segment slots
cudaError_t launch_combine(const void* W_UV, int Hv, int Bv, const QSpec& qs, const int* plan, const uint16_t* part_o,
                           const float* part_lse, void* out, float* o_lat, int* err, int max_workers,
                           cudaStream_t s);

// 3-D TMA tensor map (tensor_map.cu): dims (d0 fastest), byte strides of dims 1
// and 2, box (b0, b1, 1); false when the driver refuses the description
bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
               uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
// the same with a box extent in all three dims
bool encode_3d_box(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                   uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw,
                   CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

// Programmatic dependent launch.  A kernel of the decode chain is launched
// with launch_pdl, so it may start while the kernel before it in the stream is
// still running; it must call grid_dep_wait before touching any memory that
// earlier work may write (or read), and calls grid_dep_launch after that wait,
// letting the next kernel of the chain begin its own prologue.
// Walk over a worker's pages in halves of 32 tokens (the CUDA-core and
// warp-MMA decode kernels): page tile x of row b, half 0 or 1; a page's second
// half is visited only when it holds tokens.
struct HalfCursor {
  int x, half, b;
};
__device__ __forceinline__ int page_valid(const int* prefix, const int* seq_c, int b, int x) {
  return min(PAGE, seq_c[b] - PAGE * (x - prefix[b]));
}
__device__ __forceinline__ void cursor_next(HalfCursor& c, const int* prefix, const int* seq_c, int B) {
  if (c.half == 0 && page_valid(prefix, seq_c, c.b, c.x) > PAGE / 2) {
    c.half = 1;
    return;
  }
  c.half = 0;
  ++c.x;
  while (c.b < B - 1 && c.x >= prefix[c.b + 1]) ++c.b;
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace mla
