// C ABI of libmla: argument checks, workspace layout, kernel dispatch and the
// device error word.  Declarations and the contract live in include/mla.h.
#include <atomic>
#include <mutex>

#include "mla_common.cuh"

namespace mla {

// First device-detected error: [0] status, [1] detail.  One copy per device.
__device__ int g_error_word[2];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
int* g_err_ptr[MAX_DEVICES] = {};
int g_sms[MAX_DEVICES] = {};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1;
  return dev;
}

// device address of this device's error word (resolved once per device)
int* err_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool heads_ok(int H) { return H == 16 || H == 128; }
bool fmt_ok(int fmt) { return fmt >= MLA_FMT_BF16 && fmt <= MLA_FMT_INT4_PE4; }
// hidden width of the cache producer's input: whole 64-wide chunks of the projection's K
bool hidden_ok(int hidden) { return hidden >= 64 && hidden <= 65536 && hidden % 64 == 0; }
// the producer indexes tokens with 32-bit integers
constexpr long long MAX_PROJECT_TOKENS = 2147483647LL - 128;

size_t page_bytes(int fmt) {
  switch (layout_fmt(fmt)) {
    case MLA_FMT_BF16: return PAGE_BYTES_BF16;
    case MLA_FMT_INT8: return PAGE_BYTES_INT8;
    case MLA_FMT_INT4: return PAGE_BYTES_INT4;
    default: return 0;
  }
}

// the kernel of 16-head decodes over bf16 pages (mla_decode_select_kernel)
std::atomic<int> g_small_head_kernel{MLA_KERNEL_MMA};

// attend kernel for H heads over a `fmt` cache (an mla_kernel_t value), -1 = none
int attend_kind(int H, int fmt) {
  if (!heads_ok(H) || !fmt_ok(fmt)) return -1;
  if (H == 128) return MLA_KERNEL_TCGEN05;  // every format: quantized pages are dequantized in the load stage
  return fmt == MLA_FMT_BF16 ? g_small_head_kernel.load() : -1;
}

int max_workers(int sms) {
  int w = attend_tc_workers(sms);
  if (attend_cc_workers(sms) > w) w = attend_cc_workers(sms);
  if (attend_mma_workers(sms) > w) w = attend_mma_workers(sms);
  return w;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

bool cache_ok(const mla_cache_t* c) {
  return c != nullptr && fmt_ok(c->fmt) && c->num_pages > 0 && c->pages != nullptr && aligned(c->pages, 256);
}

int check_ws(int B, int H, void* ws, size_t ws_bytes, WsLayout* L) {
  const int sms = num_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  *L = ws_layout(B, H, max_workers(sms));
  if (ws == nullptr || !aligned(ws, 256)) return MLA_ERR_INVALID;
  if (ws_bytes < L->total) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

}  // namespace

// accessors for other translation units of the library
int* device_error_word() { return err_ptr(); }
int device_sm_count() { return num_sms(); }
int attend_kernel_kind(int H, int fmt) { return attend_kind(H, fmt); }
int attend_workers(int kind, int sms) {
  return kind == MLA_KERNEL_TCGEN05 ? attend_tc_workers(sms)
         : kind == MLA_KERNEL_MMA   ? attend_mma_workers(sms)
                                    : attend_cc_workers(sms);
}
cudaError_t launch_attend_kind(int kind, const void* q_cat, int H, const mla_cache_t* cache,
                               const int32_t* page_table, int max_pages, int B, float scale, int* plan, int workers,
                               int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s) {
  switch (kind) {
    case MLA_KERNEL_TCGEN05:
      return launch_attend_tc(q_cat, qspec_single(H), layout_fmt(cache->fmt), cache->num_pages, cache->pages,
                              page_table, max_pages, B, scale, plan, workers, seg_cap, part_o, part_lse, err, s);
    case MLA_KERNEL_MMA:
      return launch_attend_mma(q_cat, H, cache->fmt, cache->num_pages, cache->pages, page_table, max_pages, B, scale,
                               plan, workers, seg_cap, part_o, part_lse, err, s);
    case MLA_KERNEL_CUDA_CORES:
      return launch_attend_cc(q_cat, H, cache->fmt, cache->num_pages, cache->pages, page_table, max_pages, B, scale,
                              plan, workers, seg_cap, part_o, part_lse, err, s);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_cache_page_bytes(int fmt) { return page_bytes(fmt); }

int mla_absorb_weights(const void* wkv_b, int H, void* W_UK, void* W_UV, cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (!wkv_b || !W_UK || !W_UV || !aligned(wkv_b, 16) || !aligned(W_UK, 16) || !aligned(W_UV, 16))
    return MLA_ERR_INVALID;
  return status_of(launch_absorb_weights(wkv_b, H, W_UK, W_UV, stream));
}

int mla_cache_append(const mla_cache_t* cache, const void* c_kv, const void* k_pe, const int32_t* page_table,
                     int max_pages, const int32_t* pos, int B, int T, cudaStream_t stream) {
  if (cache == nullptr || !fmt_ok(cache->fmt)) return cache == nullptr ? MLA_ERR_INVALID : MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache) || B < 0 || T < 0 || max_pages <= 0) return MLA_ERR_INVALID;
  if ((long long)B * T == 0) return MLA_OK;
  if (!c_kv || !k_pe || !page_table || !pos || !aligned(c_kv, 16) || !aligned(k_pe, 16) || !aligned(page_table, 4) ||
      !aligned(pos, 4))
    return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  return status_of(launch_cache_append(cache->fmt, cache->num_pages, cache->pages, c_kv, k_pe, page_table, max_pages,
                                       pos, B, T, err, stream));
}

size_t mla_cache_project_workspace_bytes(int B, int T, int hidden, int k_splits) {
  if (B < 0 || T < 0 || k_splits < 0 || !hidden_ok(hidden)) return 0;
  const long long ntok = (long long)B * T;
  if (ntok > MAX_PROJECT_TOKENS) return 0;
  const int sms = num_sms();
  if (sms <= 0) return 0;
  if (k_splits == 0 && ntok <= PROJECT_SMALL_TOKENS)
    return project_small_workspace_bytes(ntok, project_small_splits(hidden, sms));
  return project_workspace_bytes(ntok, project_splits(ntok, hidden, sms, k_splits));
}

int mla_cache_project_append(const mla_cache_t* cache, const void* x, int hidden, const void* wkv_a,
                             const void* kv_norm_w, float eps, float rope_theta, const int32_t* page_table,
                             int max_pages, const int32_t* pos, int B, int T, void* latent_out, int k_splits,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (cache == nullptr) return MLA_ERR_INVALID;
  if (!fmt_ok(cache->fmt) || !hidden_ok(hidden) || layout_fmt(cache->fmt) != cache->fmt) return MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache) || B < 0 || T < 0 || max_pages <= 0 || k_splits < 0) return MLA_ERR_INVALID;
  const long long ntok = (long long)B * T;
  if (ntok == 0) return MLA_OK;
  if (ntok > MAX_PROJECT_TOKENS) return MLA_ERR_UNSUPPORTED;
  if (!x || !wkv_a || !kv_norm_w || !page_table || !pos || !aligned(x, 16) || !aligned(wkv_a, 16) ||
      !aligned(kv_norm_w, 16) || !aligned(page_table, 4) || !aligned(pos, 4) ||
      (latent_out != nullptr && !aligned(latent_out, 16)))
    return MLA_ERR_INVALID;
  if (!(eps >= 0.f) || eps == INFINITY || !(rope_theta > 0.f) || rope_theta == INFINITY) return MLA_ERR_INVALID;
  const int sms = num_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  // at most 64 tokens with the automatic split: the warp-level projection
  const bool small = k_splits == 0 && ntok <= PROJECT_SMALL_TOKENS;
  const int ksplit = small ? project_small_splits(hidden, sms) : project_splits(ntok, hidden, sms, k_splits);
  if (2 * ((ntok + 127) / 128) * (long long)ksplit > 2147483647LL) return MLA_ERR_UNSUPPORTED;  // one CTA per grid x
  const size_t need = small ? project_small_workspace_bytes(ntok, ksplit) : project_workspace_bytes(ntok, ksplit);
  if (need > 0) {
    if (workspace == nullptr || !aligned(workspace, 256)) return MLA_ERR_INVALID;
    if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  }
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  return status_of(launch_cache_project(x, hidden, wkv_a, kv_norm_w, eps, rope_theta, cache->fmt, cache->num_pages,
                                        cache->pages, page_table, max_pages, pos, B, T, latent_out, ksplit, small,
                                        workspace, err, stream));
}

size_t mla_decode_workspace_bytes(int B, int H) {
  if (B < 0 || !heads_ok(H)) return 0;
  const int sms = num_sms();
  if (sms <= 0) return 0;
  return ws_layout(B, H, max_workers(sms)).total;
}

}  // extern "C"

namespace {
// step 1 with its checks; after_plan: called by mla_decode right after its plan step
int absorb_q_checked(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* workspace,
                     size_t workspace_bytes, bool after_plan, cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (B < 0) return MLA_ERR_INVALID;
  WsLayout L;
  int st = check_ws(B, H, workspace, workspace_bytes, &L);
  if (st != MLA_OK) return st;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !W_UK || !aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(W_UK, 16))
    return MLA_ERR_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return status_of(launch_q_absorb(q_nope, q_pe, W_UK, H, B, ws + L.q_cat, after_plan, stream));
}
}  // namespace

extern "C" {

int mla_decode_absorb_q(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return absorb_q_checked(q_nope, q_pe, W_UK, H, B, workspace, workspace_bytes, false, stream);
}

}  // extern "C"

namespace {
// Step 0 with `req` split workers (0: the attend kernel's default count; else
// 1 <= req <= that count)
int decode_plan(int H, int fmt, const int32_t* seqlens, int B, int max_pages, int req, void* workspace,
                size_t workspace_bytes, cudaStream_t stream) {
  if (!heads_ok(H) || !fmt_ok(fmt)) return MLA_ERR_UNSUPPORTED;
  const int kind = attend_kind(H, fmt);
  if (kind < 0) return MLA_ERR_UNSUPPORTED;
  if (B < 0 || max_pages <= 0 || req < 0) return MLA_ERR_INVALID;
  WsLayout L;
  int st = check_ws(B, H, workspace, workspace_bytes, &L);
  if (st != MLA_OK) return st;
  const int sms = num_sms();
  const int workers = attend_workers(kind, sms);
  if (req > workers) return MLA_ERR_INVALID;
  if (B == 0) return MLA_OK;
  if (!seqlens || !aligned(seqlens, 4)) return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  int* plan = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + L.plan);
  return status_of(launch_plan(seqlens, B, qspec_single(H), max_pages, req > 0 ? req : workers, plan, err, stream));
}
}  // namespace

extern "C" {

int mla_decode_plan(int H, int fmt, const int32_t* seqlens, int B, int max_pages, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
  return decode_plan(H, fmt, seqlens, B, max_pages, 0, workspace, workspace_bytes, stream);
}

int mla_decode_plan_workers(int H, int fmt, const int32_t* seqlens, int B, int max_pages, int workers,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (workers < 1) return MLA_ERR_INVALID;
  return decode_plan(H, fmt, seqlens, B, max_pages, workers, workspace, workspace_bytes, stream);
}

int mla_decode_max_workers(int H, int fmt) {
  const int kind = attend_kind(H, fmt);
  if (kind < 0) return MLA_ERR_UNSUPPORTED;
  const int sms = num_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  return attend_workers(kind, sms);
}

int mla_decode_attend(int H, const mla_cache_t* cache, const int32_t* page_table, int max_pages,
                      const int32_t* seqlens, int B, float scale, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (cache == nullptr || B < 0 || max_pages <= 0) return MLA_ERR_INVALID;
  if (!fmt_ok(cache->fmt)) return MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache)) return MLA_ERR_INVALID;
  const int kind = attend_kind(H, cache->fmt);
  if (kind < 0) return MLA_ERR_UNSUPPORTED;
  WsLayout L;
  int st = check_ws(B, H, workspace, workspace_bytes, &L);
  if (st != MLA_OK) return st;
  if (B == 0) return MLA_OK;
  if (!page_table || !seqlens || !aligned(page_table, 4) || !aligned(seqlens, 4)) return MLA_ERR_INVALID;
  if (!(scale > 0.f) || scale == INFINITY) return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* plan = reinterpret_cast<int*>(ws + L.plan);
  uint16_t* part_o = reinterpret_cast<uint16_t*>(ws + L.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  const int sms = num_sms();
  const int workers = attend_workers(kind, sms);
  return status_of(launch_attend_kind(kind, ws + L.q_cat, H, cache, page_table, max_pages, B, scale, plan, workers,
                                      L.max_segments, part_o, part_lse, err, stream));
}

int mla_decode_combine(const void* W_UV, int H, int B, void* workspace, size_t workspace_bytes, void* out,
                       float* o_lat_out, cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (B < 0) return MLA_ERR_INVALID;
  WsLayout L;
  int st = check_ws(B, H, workspace, workspace_bytes, &L);
  if (st != MLA_OK) return st;
  if (B == 0) return MLA_OK;
  if (!W_UV || !out || !aligned(W_UV, 16) || !aligned(out, 16) || (o_lat_out && !aligned(o_lat_out, 16)))
    return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return status_of(launch_combine(W_UV, H, B, qspec_single(H), reinterpret_cast<const int*>(ws + L.plan),
                                  reinterpret_cast<const uint16_t*>(ws + L.part_o),
                                  reinterpret_cast<const float*>(ws + L.part_lse), out, o_lat_out, err,
                                  L.max_segments - B, stream));
}

int mla_decode(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H,
               const mla_cache_t* cache, const int32_t* page_table, int max_pages, const int32_t* seqlens, int B,
               float scale, void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (cache == nullptr || B < 0 || max_pages <= 0) return MLA_ERR_INVALID;
  if (!fmt_ok(cache->fmt)) return MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache)) return MLA_ERR_INVALID;
  if (attend_kind(H, cache->fmt) < 0) return MLA_ERR_UNSUPPORTED;
  WsLayout L;
  int st = check_ws(B, H, workspace, workspace_bytes, &L);
  if (st != MLA_OK) return st;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !W_UK || !W_UV || !out || !page_table || !seqlens) return MLA_ERR_INVALID;
  st = mla_decode_plan(H, cache->fmt, seqlens, B, max_pages, workspace, workspace_bytes, stream);
  if (st != MLA_OK) return st;
  st = absorb_q_checked(q_nope, q_pe, W_UK, H, B, workspace, workspace_bytes, true, stream);
  if (st != MLA_OK) return st;
  st = mla_decode_attend(H, cache, page_table, max_pages, seqlens, B, scale, workspace, workspace_bytes, stream);
  if (st != MLA_OK) return st;
  return mla_decode_combine(W_UV, H, B, workspace, workspace_bytes, out, nullptr, stream);
}

}  // extern "C"

namespace {
constexpr int MAX_Q_LEN = 65536;
// T query tokens per row for H heads on the tcgen05 kernel's 128 MMA rows
QSpec qspec_multi(int H, int T) {
  const int G = 128 / H;
  return QSpec{T, G, (T + G - 1) / G, H};
}
WsLayout ws_layout_multi(int B, int H, int T, int workers) {
  const QSpec qs = qspec_multi(H, T);
  return ws_layout_q(B * qs.NG, 128, (long long)B * T * H, workers);
}
bool multi_ok(int B, int H, int T) {
  if (!heads_ok(H) || T < 1 || T > MAX_Q_LEN || B < 0) return false;
  const long long rows = (long long)B * T * H;  // flat query rows: TMA coordinates
  return rows <= 2147483647LL - 256 && (long long)B * qspec_multi(H, T).NG <= 2147483647LL / 4;
}
}  // namespace

extern "C" {

size_t mla_decode_q_workspace_bytes(int B, int H, int T) {
  if (!multi_ok(B, H, T)) return 0;
  const int sms = num_sms();
  if (sms <= 0) return 0;
  return ws_layout_multi(B, H, T, attend_tc_workers(sms)).total;
}

int mla_decode_q(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H, int T,
                 const mla_cache_t* cache, const int32_t* page_table, int max_pages, const int32_t* seqlens, int B,
                 float scale, void* workspace, size_t workspace_bytes, void* out, float* o_lat_out,
                 cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (cache == nullptr || B < 0 || max_pages <= 0 || T < 1) return MLA_ERR_INVALID;
  if (!multi_ok(B, H, T)) return MLA_ERR_UNSUPPORTED;
  if (!fmt_ok(cache->fmt)) return MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache)) return MLA_ERR_INVALID;
  const int sms = num_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  const int workers = attend_tc_workers(sms);
  const WsLayout L = ws_layout_multi(B, H, T, workers);
  if (workspace == nullptr || !aligned(workspace, 256)) return MLA_ERR_INVALID;
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !W_UK || !W_UV || !out || !page_table || !seqlens) return MLA_ERR_INVALID;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(W_UK, 16) || !aligned(W_UV, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(seqlens, 4) || (o_lat_out && !aligned(o_lat_out, 16)))
    return MLA_ERR_INVALID;
  if (!(scale > 0.f) || scale == INFINITY) return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  const QSpec qs = qspec_multi(H, T);
  const int Bv = B * qs.NG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* plan = reinterpret_cast<int*>(ws + L.plan);
  uint16_t* part_o = reinterpret_cast<uint16_t*>(ws + L.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  cudaError_t e = launch_plan(seqlens, B, qs, max_pages, workers, plan, err, stream);
  if (e == cudaSuccess) e = launch_q_absorb(q_nope, q_pe, W_UK, H, B * T, ws + L.q_cat, true, stream);
  if (e == cudaSuccess)
    e = launch_attend_tc(ws + L.q_cat, qs, layout_fmt(cache->fmt), cache->num_pages, cache->pages, page_table, max_pages, Bv,
                         scale, plan, workers, L.max_segments, part_o, part_lse, err, stream);
  if (e == cudaSuccess)
    e = launch_combine(W_UV, 128, Bv, qs, plan, part_o, part_lse, out, o_lat_out, err, L.max_segments - Bv, stream);
  return status_of(e);
}

size_t mla_prefill_workspace_bytes(int B, int H, int max_pages) {
  if (B < 0 || !heads_ok(H) || max_pages <= 0) return 0;
  if ((long long)B * max_pages * PAGE > 2147483647LL - 256) return 0;  // key rows are TMA coordinates
  return prefill_workspace_bytes(B, H, max_pages);
}

int mla_prefill(const void* q_nope, const void* q_pe, const void* wkv_b, int H, int T, const mla_cache_t* cache,
                const int32_t* page_table, int max_pages, const int32_t* seqlens, int B, float scale,
                void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (cache == nullptr || B < 0 || T < 1 || max_pages <= 0) return MLA_ERR_INVALID;
  if (cache->fmt != MLA_FMT_BF16) return MLA_ERR_UNSUPPORTED;
  if (!cache_ok(cache)) return MLA_ERR_INVALID;
  if ((long long)B * T > 2147483647LL - 256 || (long long)B * max_pages * PAGE > 2147483647LL - 256)
    return MLA_ERR_UNSUPPORTED;
  const size_t need = prefill_workspace_bytes(B, H, max_pages);
  if (workspace == nullptr || !aligned(workspace, 256)) return MLA_ERR_INVALID;
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !wkv_b || !out || !page_table || !seqlens) return MLA_ERR_INVALID;
  if (!aligned(q_nope, 16) || !aligned(q_pe, 16) || !aligned(wkv_b, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(seqlens, 4))
    return MLA_ERR_INVALID;
  if (!(scale > 0.f) || scale == INFINITY) return MLA_ERR_INVALID;
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  return status_of(launch_prefill(q_nope, q_pe, wkv_b, H, T, cache->num_pages, cache->pages, page_table, max_pages,
                                  seqlens, B, scale, workspace, out, err, stream));
}

size_t mla_output_projection_workspace_bytes(int R, int H, int hidden) {
  if (R < 0 || !heads_ok(H) || hidden <= 0 || hidden % 128 != 0) return 0;
  const int sms = num_sms();
  if (sms <= 0) return 0;
  return out_proj_workspace_bytes(R, H * DV, hidden, sms);
}

int mla_output_projection(const void* o, const void* W_O, int R, int H, int hidden, void* y, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  if (!heads_ok(H) || hidden <= 0 || hidden % 128 != 0 || hidden > 65536) return MLA_ERR_UNSUPPORTED;
  if (R < 0) return MLA_ERR_INVALID;
  if (R == 0) return MLA_OK;
  if (!o || !W_O || !y || !aligned(o, 16) || !aligned(W_O, 16) || !aligned(y, 16)) return MLA_ERR_INVALID;
  const int sms = num_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  const size_t need = out_proj_workspace_bytes(R, H * DV, hidden, sms);
  if (need > 0) {
    if (workspace == nullptr || !aligned(workspace, 256)) return MLA_ERR_INVALID;
    if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  }
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  return status_of(launch_out_proj(o, W_O, R, H * DV, hidden, y, workspace, err, stream));
}

int mla_get_device_status(cudaStream_t stream, int* info) {
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  int host[2] = {0, 0};
  if (cudaMemcpyAsync(host, err, sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (host[0] != 0) {
    if (cudaMemsetAsync(err, 0, sizeof(host), stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  }
  if (info != nullptr) *info = host[1];
  return host[0];
}

int mla_wait_selftest(cudaStream_t stream) {
  int* err = err_ptr();
  if (err == nullptr) return MLA_ERR_CUDA;
  return status_of(launch_wait_selftest(err, stream));
}

int mla_decode_kernel_kind(int H) { return attend_kind(H, MLA_FMT_BF16); }

int mla_decode_select_kernel(int H, int kind) {
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  if (H == 128) return kind == MLA_KERNEL_TCGEN05 ? MLA_OK : MLA_ERR_UNSUPPORTED;
  if (kind != MLA_KERNEL_MMA && kind != MLA_KERNEL_CUDA_CORES) return MLA_ERR_UNSUPPORTED;
  g_small_head_kernel.store(kind);
  return MLA_OK;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_BOUNDS: return "page id or sequence length out of bounds";
    case MLA_ERR_TIMEOUT: return "bounded device wait timed out";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

}  // extern "C"
