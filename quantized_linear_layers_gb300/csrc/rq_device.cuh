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
// Formulation used here: the sm_89+ conversion cvt.rn.satfinite.e4m3x2.f32
// rounds to nearest even among E4M3FN values and saturates finite overflow
// and +-Inf to +-448, which is exactly the rule for 2^-6 <= |v|; values below
// 2^-6 (and NaN, which only arises from 0 * Inf here) are replaced by +0
// before the conversion, and non-finite inputs are handled before the
// multiply by the callers below.

// Two codes: low byte from `lo`, high byte from `hi`.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// +0 unless 2^-6 <= |v| (NaN fails the comparison too).
__device__ __forceinline__ float flush_small(float v) {
  return fabsf(v) >= 0x1p-6f ? v : 0.0f;
}

__device__ __forceinline__ bool non_finite(float x) {
  return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

__device__ __forceinline__ uint32_t saturated_code(float x) {
  return ((__float_as_uint(x) >> 24) & 0x80u) | 0x7Eu;
}

// Scaled element encode: non-finite inputs keep their own sign and saturate,
// +-0 gives 0x00 (both decided before the multiply); otherwise one
// correctly rounded fp32 multiply by s (no FMA contraction) and the encoder.
__device__ __forceinline__ uint32_t e4m3_scaled(float x, float s) {
  if (non_finite(x)) return saturated_code(x);
  return cvt_e4m3x2(0.0f, flush_small(__fmul_rn(x, s))) & 0xFFu;
}

// Four elements -> four codes (element i in byte i).
__device__ __forceinline__ uint32_t e4m3_scaled4(float4 v, float s) {
  const float a = flush_small(__fmul_rn(v.x, s)), b = flush_small(__fmul_rn(v.y, s));
  const float c = flush_small(__fmul_rn(v.z, s)), d = flush_small(__fmul_rn(v.w, s));
  uint32_t r = cvt_e4m3x2(b, a) | (cvt_e4m3x2(d, c) << 16);
  if (non_finite(v.x) | non_finite(v.y) | non_finite(v.z) | non_finite(v.w)) {
    if (non_finite(v.x)) r = (r & 0xFFFFFF00u) | saturated_code(v.x);
    if (non_finite(v.y)) r = (r & 0xFFFF00FFu) | (saturated_code(v.y) << 8);
    if (non_finite(v.z)) r = (r & 0xFF00FFFFu) | (saturated_code(v.z) << 16);
    if (non_finite(v.w)) r = (r & 0x00FFFFFFu) | (saturated_code(v.w) << 24);
  }
  return r;
}

// The same for four finite values (no non-finite fix-ups).
__device__ __forceinline__ uint32_t e4m3_scaled4_finite(float4 v, float s) {
  const float a = flush_small(__fmul_rn(v.x, s)), b = flush_small(__fmul_rn(v.y, s));
  const float c = flush_small(__fmul_rn(v.z, s)), d = flush_small(__fmul_rn(v.w, s));
  return cvt_e4m3x2(b, a) | (cvt_e4m3x2(d, c) << 16);
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

// ------------------------------------------------------ mbarrier / TMA ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, at most limit_ns
// nanoseconds.  On expiry, sets bit 0 of *err and returns false.
__device__ __noinline__ inline bool mbar_wait(uint32_t bar, uint32_t parity,
                                              uint64_t limit_ns, unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(err, 1u);
      return false;
    }
  }
}

// mbar_wait with its first test inline: the call is made only when the
// phase has not completed yet (for waits in loops that are bound by issue).
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               unsigned int* err) {
  return mbar_try_wait(bar, parity) || mbar_wait(bar, parity, limit_ns, err);
}

// An L2 cache policy that evicts the lines it loads first (for data that is
// read once and should not push other lines out of L2).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// An L2 cache policy that keeps the lines it loads longest (data read again
// soon).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte read-only load with an L2 cache policy.
__device__ __forceinline__ float4 ldg_f4_policy(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on bar.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s for any pipeline wait

// Programmatic dependent launch.  pdl_wait: block until the grids this
// launch depends on have completed and their memory operations are visible;
// pdl_trigger: let the next launch in the stream start being scheduled.
// Both are no-ops for launches made without programmatic serialization.
// Every kernel of the library calls pdl_wait before it reads anything an
// earlier launch may write (activations, scales, outputs) and calls
// pdl_trigger only after its own pdl_wait, so that whatever a kernel may
// read before its wait (constant weights) was written by launches that
// completed before its predecessor passed its own wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace rq
