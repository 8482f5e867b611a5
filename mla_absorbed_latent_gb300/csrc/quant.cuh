// The cache quantizers of the page formats (include/mla.h), shared by the
// kernels that write pages (mla_cache_append and the fused producer of
// mla_cache_project_append).  Every decision is one IEEE fp32 operation on
// bf16-representable inputs, so the codes and scales are bit-exact and
// deterministic: INT8 over 32-channel groups of c_KV and 8-dim groups of k_pe,
// asymmetric INT4 (scale + zero) over 32-channel groups of c_KV, and the
// per-token INT8, symmetric INT4 and 4-bit RoPE-key variants
// ("DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化" §3.2 names the block sizes; the
// rounding rules are the library's, stated in include/mla.h).
#pragma once

#include "mla_common.cuh"

namespace mla {

// Symmetric INT8 of N values: returns the bf16 scale bits, writes the codes.
template <int N>
__device__ __forceinline__ uint16_t quant_i8(const float* x, int8_t* code) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const __nv_bfloat16 sb = __float2bfloat16_rn(amax / 127.0f);
  const float s = __bfloat162float(sb);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float q = 0.f;
    if (s != 0.f) q = fminf(fmaxf(rintf(x[i] / s), -127.f), 127.f);
    code[i] = static_cast<int8_t>(q);
  }
  return __bfloat16_as_ushort(sb);
}

// Asymmetric INT4 of 32 values: the codes packed two per byte (element 2i in
// the low nibble, 2i+1 in the high) into w[0..3]; bf16 scale and zero bits out.
__device__ __forceinline__ void quant_i4_32(const float* x, uint32_t* w, uint16_t* scale_bits, uint16_t* zero_bits) {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
  const __nv_bfloat16 sb = __float2bfloat16_rn((mx - mn) / 15.0f);
  const __nv_bfloat16 zb = __float2bfloat16_rn(mn);
  const float s = __bfloat162float(sb), z = __bfloat162float(zb);
  w[0] = w[1] = w[2] = w[3] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t q = 0u;
    if (s != 0.f) q = (uint32_t)fminf(fmaxf(rintf((x[i] - z) / s), 0.f), 15.f);
    w[i / 8] |= q << (4 * (i % 8));
  }
  *scale_bits = __bfloat16_as_ushort(sb);
  *zero_bits = __bfloat16_as_ushort(zb);
}

// INT8 codes of N values with a given scale (bf16 value s): the per-token
// quantizer's groups, which share the token's scale
template <int N>
__device__ __forceinline__ void quant_i8_scaled(const float* x, float s, int8_t* code) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float q = 0.f;
    if (s != 0.f) q = fminf(fmaxf(rintf(x[i] / s), -127.f), 127.f);
    code[i] = static_cast<int8_t>(q);
  }
}

// Symmetric INT4 of 32 values, written in the asymmetric INT4 page form: the
// nibbles hold q + 8 (q = clamp(rint(x / s), -7, 7), s = bf16(amax / 7)) and
// the zero is -8 s, so that code * s + zero = q * s exactly.
__device__ __forceinline__ void quant_i4sym_32(const float* x, uint32_t* w, uint16_t* scale_bits, uint16_t* zero_bits) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const __nv_bfloat16 sb = __float2bfloat16_rn(amax / 7.0f);
  const float s = __bfloat162float(sb);
  w[0] = w[1] = w[2] = w[3] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float q = 0.f;
    if (s != 0.f) q = fminf(fmaxf(rintf(x[i] / s), -7.f), 7.f);
    w[i / 8] |= (uint32_t)(q + 8.f) << (4 * (i % 8));
  }
  *scale_bits = __bfloat16_as_ushort(sb);
  *zero_bits = __bfloat16_as_ushort(__float2bfloat16_rn(-8.f * s));  // exact: a power-of-two multiple
}

// Symmetric INT4 of N values as INT8 codes (-7..7): returns the bf16 scale bits
// (s = bf16(amax / 7)); the 4-bit RoPE-key quantizer, stored in the INT8 code
// section of a page
template <int N>
__device__ __forceinline__ uint16_t quant_i4sym_i8(const float* x, int8_t* code) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const __nv_bfloat16 sb = __float2bfloat16_rn(amax / 7.0f);
  const float s = __bfloat162float(sb);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float q = 0.f;
    if (s != 0.f) q = fminf(fmaxf(rintf(x[i] / s), -7.f), 7.f);
    code[i] = static_cast<int8_t>(q);
  }
  return __bfloat16_as_ushort(sb);
}

__device__ __forceinline__ void store_i8x8(uint8_t* dst, const int8_t* c) {
  uint2 v;
  v.x = (uint32_t)(uint8_t)c[0] | ((uint32_t)(uint8_t)c[1] << 8) | ((uint32_t)(uint8_t)c[2] << 16) |
        ((uint32_t)(uint8_t)c[3] << 24);
  v.y = (uint32_t)(uint8_t)c[4] | ((uint32_t)(uint8_t)c[5] << 8) | ((uint32_t)(uint8_t)c[6] << 16) |
        ((uint32_t)(uint8_t)c[7] << 24);
  *reinterpret_cast<uint2*>(dst) = v;
}

}  // namespace mla
