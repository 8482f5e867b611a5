// mla_decode_noalloc: the decode step for callers that cannot allocate device
// memory.
//
// Some hosts of this library cannot hand it a workspace: an inference engine
// whose custom-operator interface passes only the op's inputs and outputs, a
// runtime that has given all device memory to its own pool and offers no
// allocation hook, or a serving loop that forbids cudaMalloc (a device-wide,
// synchronising call) once it is running.  For them this entry point keeps
// its scratch (the split plan, the query-side latent and the split partials)
// in one fixed array of device global memory that belongs to the library
// image itself, so neither the caller nor the library allocates anything.
//
// Costs of that choice, stated for the user:
//  * every GPU that loads the library holds the array (MLA_NOALLOC_SCRATCH_BYTES)
//    until the process exits;
//  * all calls on a device share the one array and it keeps whatever the last
//    call left there: two calls whose work overlaps on the GPU (different
//    streams, or different host threads, without ordering between them) race
//    on it and corrupt each other's results — serialise them on one stream;
//  * nothing in the array has to start at zero: every byte a call reads was
//    written earlier in the same call (plan, then query latent, then partials);
//  * the first call on a device looks up the array's device address (once per
//    device, with that device current); make that first call before any stream
//    capture begins;
//  * when the batch does not fit, the call is rejected with MLA_ERR_WORKSPACE;
//    to fit, the call may use fewer split workers than mla_decode, so its
//    results can differ from mla_decode's in the last bits (same tolerance).
#include <mutex>

#include "mla_common.cuh"

namespace mla {
namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a usable address: host code passes on the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; resolved once
// per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_decode_noalloc(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H,
                                  const mla_cache_t* cache, const int32_t* page_table, int max_pages,
                                  const int32_t* seqlens, int B, float scale, void* out, cudaStream_t stream) {
  if (H != 16 && H != 128) return MLA_ERR_UNSUPPORTED;
  if (cache == nullptr || B < 0 || max_pages <= 0) return MLA_ERR_INVALID;
  const int kind = attend_kernel_kind(H, cache->fmt);
  if (kind < 0) return MLA_ERR_UNSUPPORTED;
  if (cache->num_pages <= 0 || cache->pages == nullptr || !aligned_to(cache->pages, 256)) return MLA_ERR_INVALID;
  if (B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !W_UK || !W_UV || !out || !page_table || !seqlens) return MLA_ERR_INVALID;
  if (!aligned_to(q_nope, 16) || !aligned_to(q_pe, 16) || !aligned_to(W_UK, 16) || !aligned_to(W_UV, 16) ||
      !aligned_to(out, 16) || !aligned_to(page_table, 4) || !aligned_to(seqlens, 4))
    return MLA_ERR_INVALID;
  if (!(scale > 0.f) || scale == INFINITY) return MLA_ERR_INVALID;  // the same rule as mla_decode

  const int sms = device_sm_count();
  if (sms <= 0) return MLA_ERR_CUDA;
  const int want = attend_workers(kind, sms);
  const int workers = fitting_workers(B, H, want, kScratchBytes);
  if (workers < 1) return MLA_ERR_WORKSPACE;  // batch too large for the fixed scratch

  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != MLA_OK) return st;
  int* err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;

  const WsLayout L = ws_layout(B, H, workers);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  int* plan = reinterpret_cast<int*>(ws + L.plan);
  uint16_t* part_o = reinterpret_cast<uint16_t*>(ws + L.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + L.part_lse);

  if (launch_plan(seqlens, B, qspec_single(H), max_pages, workers, plan, err, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_q_absorb(q_nope, q_pe, W_UK, H, B, ws + L.q_cat, true, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_attend_kind(kind, ws + L.q_cat, H, cache, page_table, max_pages, B, scale, plan, workers,
                         L.max_segments, part_o, part_lse, err, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (launch_combine(W_UV, H, B, qspec_single(H), plan, part_o, part_lse, out, nullptr, err, workers, stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}
