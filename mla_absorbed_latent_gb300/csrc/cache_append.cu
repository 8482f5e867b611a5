// Append new tokens (c_KV, k_pe) into the paged latent cache, quantizing per
// the cache format.
//
// The absorbed cache keeps one 512-wide latent and one 64-wide RoPE key per
// token ("DeepSeek MLA 吸收式缓存" §2.4, §4.1).  Quantized formats follow the
// block sizes of "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化" §3.2: INT8 over
// 32-channel groups of c_KV, asymmetric INT4 (scale + zero) over 32-channel
// groups, and INT8 over 8-dim groups of k_pe.  The rounding rules (fp32,
// round-half-even, bf16 scales) are stated in include/mla.h and are bit-exact
// by construction: every decision is one IEEE fp32 operation (quant.cuh).
//
// One warp per token.  bf16: lanes copy 16-byte chunks.  Quantized: lane g < 16
// owns c_KV group g, lanes 16..23 own the k_pe groups.  The per-token INT8 and
// symmetric INT4 quantizers write INT8 and INT4 pages (include/mla.h).
#include "quant.cuh"

namespace mla {
namespace {

__device__ __forceinline__ void load32(const uint16_t* src, float* x) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v = s[i];
    x[8 * i + 0] = bf16lo(v.x); x[8 * i + 1] = bf16hi(v.x);
    x[8 * i + 2] = bf16lo(v.y); x[8 * i + 3] = bf16hi(v.y);
    x[8 * i + 4] = bf16lo(v.z); x[8 * i + 5] = bf16hi(v.z);
    x[8 * i + 6] = bf16lo(v.w); x[8 * i + 7] = bf16hi(v.w);
  }
}

__global__ void __launch_bounds__(256) append_kernel(int fmt, int num_pages, uint8_t* __restrict__ pages,
                                                      const uint16_t* __restrict__ c_kv,
                                                      const uint16_t* __restrict__ k_pe,
                                                      const int32_t* __restrict__ page_table, int max_pages,
                                                      const int32_t* __restrict__ pos, int B, int T, int* err) {
  const int lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (tok >= (long long)B * T) return;
  const int b = (int)(tok / T), t = (int)(tok % T);
  const int p0 = pos[b];
  const long long p = (long long)p0 + t;
  if (p0 < 0 || p >= (long long)max_pages * PAGE) {
    if (lane == 0) raise_error(err, MLA_ERR_BOUNDS, b);
    return;
  }
  const int lp = (int)(p / PAGE), slot = (int)(p % PAGE);
  const int phys = page_table[(size_t)b * max_pages + lp];
  if (phys < 0 || phys >= num_pages) {
    if (lane == 0) raise_error(err, MLA_ERR_BOUNDS, phys);
    return;
  }
  const uint16_t* c = c_kv + (size_t)tok * DC;
  const uint16_t* pe = k_pe + (size_t)tok * DR;

  if (fmt == MLA_FMT_BF16) {
    uint8_t* dst = pages + (size_t)phys * PAGE_BYTES_BF16 + (size_t)slot * DK * 2;
    const uint4* cs = reinterpret_cast<const uint4*>(c);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[lane] = cs[lane];
    d4[lane + 32] = cs[lane + 32];
    if (lane < 8) d4[64 + lane] = reinterpret_cast<const uint4*>(pe)[lane];
    return;
  }

  const bool i8 = layout_fmt(fmt) == MLA_FMT_INT8;
  const size_t pb = i8 ? PAGE_BYTES_INT8 : PAGE_BYTES_INT4;
  uint8_t* page = pages + (size_t)phys * pb;
  const int pe_code_off = i8 ? I8_PE_CODE : I4_PE_CODE;
  const int pe_scale_off = i8 ? I8_PE_SCALE : I4_PE_SCALE;

  // per-token INT8: the token's one scale over all 512 channels (lanes 0..15
  // own the 32-channel groups; the maximum is reduced over them)
  float tok_amax = 0.f;
  float x[32];
  if (lane < 16) {
    load32(c + lane * 32, x);
#pragma unroll
    for (int i = 0; i < 32; ++i) tok_amax = fmaxf(tok_amax, fabsf(x[i]));
  }
  if (fmt == MLA_FMT_INT8_TOKEN) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tok_amax = fmaxf(tok_amax, __shfl_xor_sync(0xffffffffu, tok_amax, o));
  }

  if (lane < 16) {
    const int g = lane;
    if (fmt == MLA_FMT_INT8_TOKEN) {
      const __nv_bfloat16 sb = __float2bfloat16_rn(tok_amax / 127.0f);
      int8_t code[32];
      quant_i8_scaled<32>(x, __bfloat162float(sb), code);
      uint8_t* dst = page + I8_C_CODE + slot * DC + g * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) store_i8x8(dst + 8 * i, code + 8 * i);
      reinterpret_cast<uint16_t*>(page + I8_C_SCALE)[slot * 16 + g] = __bfloat16_as_ushort(sb);
    } else if (fmt == MLA_FMT_INT4_SYM) {
      uint32_t w[4];
      uint16_t sb, zb;
      quant_i4sym_32(x, w, &sb, &zb);
      *reinterpret_cast<uint4*>(page + I4_C_CODE + slot * (DC / 2) + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint16_t*>(page + I4_C_SCALE)[slot * 16 + g] = sb;
      reinterpret_cast<uint16_t*>(page + I4_C_ZERO)[slot * 16 + g] = zb;
    } else if (fmt == MLA_FMT_INT8) {
      int8_t code[32];
      const uint16_t sb = quant_i8<32>(x, code);
      uint8_t* dst = page + I8_C_CODE + slot * DC + g * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) store_i8x8(dst + 8 * i, code + 8 * i);
      reinterpret_cast<uint16_t*>(page + I8_C_SCALE)[slot * 16 + g] = sb;
    } else {
      uint32_t w[4];
      uint16_t sb, zb;
      quant_i4_32(x, w, &sb, &zb);
      *reinterpret_cast<uint4*>(page + I4_C_CODE + slot * (DC / 2) + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint16_t*>(page + I4_C_SCALE)[slot * 16 + g] = sb;
      reinterpret_cast<uint16_t*>(page + I4_C_ZERO)[slot * 16 + g] = zb;
    }
  } else if (lane < 24) {
    const int g = lane - 16;
    const uint4 v = reinterpret_cast<const uint4*>(pe)[g];
    float x[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                  bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
    int8_t code[8];
    const uint16_t sb = fmt == MLA_FMT_INT4_PE4 ? quant_i4sym_i8<8>(x, code) : quant_i8<8>(x, code);
    store_i8x8(page + pe_code_off + slot * DR + g * 8, code);
    reinterpret_cast<uint16_t*>(page + pe_scale_off)[slot * 8 + g] = sb;
  }
}

}  // namespace

cudaError_t launch_cache_append(int fmt, int num_pages, void* pages, const void* c_kv, const void* k_pe,
                                const int32_t* page_table, int max_pages, const int32_t* pos, int B, int T,
                                int* err, cudaStream_t s) {
  const long long ntok = (long long)B * T;
  if (ntok == 0) return cudaSuccess;
  const int warps = 8;
  const long long blocks = (ntok + warps - 1) / warps;
  append_kernel<<<(unsigned)blocks, warps * 32, 0, s>>>(fmt, num_pages, static_cast<uint8_t*>(pages),
                                                        static_cast<const uint16_t*>(c_kv),
                                                        static_cast<const uint16_t*>(k_pe), page_table, max_pages,
                                                        pos, B, T, err);
  return cudaGetLastError();
}

}  // namespace mla
