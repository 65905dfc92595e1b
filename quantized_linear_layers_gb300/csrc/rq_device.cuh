// rq_device.cuh -- device helpers shared by the librq kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace rq {

constexpr int kQK = 256;          // weights per GGUF super-block
constexpr int kQ4KBytes = 144;    // Q4_K super-block size
constexpr int kQ6KBytes = 210;    // Q6_K super-block size

// ---------------------------------------------------------------- E4M3 ----
//
// FP32 -> E4M3 byte with the rules of realizar 0.8.4,
// cublas_prefill/mod.rs, F32_TO_E4M3_PTX: exponent rebias 127 -> 7, mantissa
// rounded to 3 bits with round-to-nearest-even, |v| < 2^-6 flushed to 0x00,
// NaN / Inf / overflow saturated to sign|0x7E, and (the one deviation from
// that code) 0x7F / 0xFF never produced.
//
// Formulation used here: for 2^-6 <= |v| < Inf, (|v|bits - 120<<23) >> 20 is
// exactly the 7-bit code exponent:mantissa; rounding that integer to nearest
// even on the 20 dropped bits also performs the mantissa carry into the
// exponent, and one clamp to 0x7E covers both 0x7F and exponent overflow.
__device__ __forceinline__ uint32_t e4m3_from_bits(uint32_t bits) {
  const uint32_t sign = (bits >> 24) & 0x80u;
  const uint32_t mag = bits & 0x7FFFFFFFu;
  if (mag >= 0x7F800000u) return sign | 0x7Eu;   // NaN, +-Inf
  if (mag < 0x3C800000u) return 0u;               // below 2^-6 (incl. +-0)
  const uint32_t r = mag - 0x3C000000u;           // exponent rebias by 120
  uint32_t code = r >> 20;
  const uint32_t rem = r & 0xFFFFFu;
  code += (rem > 0x80000u) | ((rem == 0x80000u) & (code & 1u));
  code = code < 0x7Eu ? code : 0x7Eu;
  return sign | code;
}

// Scaled element encode: non-finite inputs keep their own sign and saturate,
// +-0 gives 0x00 (both decided before the multiply); otherwise one
// correctly rounded fp32 multiply by s (no FMA contraction) and the encoder.
__device__ __forceinline__ uint32_t e4m3_scaled(float x, float s) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t mag = b & 0x7FFFFFFFu;
  if (mag >= 0x7F800000u) return ((b >> 24) & 0x80u) | 0x7Eu;
  if (mag == 0u) return 0u;
  return e4m3_from_bits(__float_as_uint(__fmul_rn(x, s)));
}

// Quantization scale from the absmax word: A' = (A == 0 ? 1 : A),
// s = 448 / A' (IEEE division), dequant = A' / 448.
__device__ __forceinline__ float absmax_prime(uint32_t absmax_bits) {
  const float a = __uint_as_float(absmax_bits);
  return a == 0.0f ? 1.0f : a;
}

// |x| bits with NaN mapped to 0 (NaNs are skipped by the absmax).
__device__ __forceinline__ uint32_t abs_bits_skip_nan(float x) {
  const uint32_t m = __float_as_uint(x) & 0x7FFFFFFFu;
  return m > 0x7F800000u ? 0u : m;
}

// ------------------------------------------------------------ loads -------

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Two fp16 values packed in a 32-bit word (low half first) -> floats.
__device__ __forceinline__ float2 half_pair(uint32_t v) {
  return make_float2(__half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(v >> 16))));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace rq
