// rq_quant.cu -- per-tensor absmax and scaled FP32 -> E4M3 quantization.
//
// realizar 0.8.4, cublas_prefill/mod.rs: ABSMAX_REDUCE_PTX (block max of |x|
// folded into a pre-zeroed word with an unsigned atomic max, valid because
// non-negative float bit patterns order like their values) and
// F32_TO_E4M3_DEVICE_SCALED_PTX (scale read from device memory, thread 0
// writes absmax/448).  Both are HBM-bound streaming kernels: 16-byte loads,
// grid sized to a multiple of the SM count, grid-stride loops.
#include <algorithm>
#include <cstdlib>

#include "rq_device.cuh"
#include "rq_internal.h"

namespace rq {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t max4(uint32_t m, float4 v) {
  m = max(m, abs_bits_skip_nan(v.x));
  m = max(m, abs_bits_skip_nan(v.y));
  m = max(m, abs_bits_skip_nan(v.z));
  return max(m, abs_bits_skip_nan(v.w));
}

// Block-wide max of the per-thread values, folded into *out by one atomic.
__device__ __forceinline__ void block_max_to(uint32_t m, uint32_t* out) {
  __shared__ uint32_t warp_max[kThreads / 32];
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_max[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kThreads / 32 ? warp_max[lane] : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0 && m != 0u) atomicMax(out, m);
  }
}

// VEC: x is 16-byte aligned, so the body is read as float4, four per
// iteration to keep 64 bytes per thread in flight; the tail (n % 4) and the
// unaligned case go element by element.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
absmax_kernel(const float* __restrict__ x, int64_t n, uint32_t* out) {
  pdl_wait();
  pdl_trigger();
  uint32_t m = 0;
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * kThreads;
  int64_t done = 0;
  if (VEC) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t n4 = n >> 2;
    int64_t i = tid;
    for (; i + 3 * nthreads < n4; i += 4 * nthreads) {
      const float4 a = __ldg(x4 + i), b = __ldg(x4 + i + nthreads);
      const float4 c = __ldg(x4 + i + 2 * nthreads), d = __ldg(x4 + i + 3 * nthreads);
      m = max4(max4(m, a), b);
      m = max4(max4(m, c), d);
    }
    for (; i < n4; i += nthreads) m = max4(m, __ldg(x4 + i));
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < n; i += nthreads)
    m = max(m, abs_bits_skip_nan(__ldg(x + i)));
  block_max_to(m, out);
}

__device__ __forceinline__ uint32_t pack4(float4 v, float s) { return e4m3_scaled4(v, s); }

// VEC: x 16-byte aligned and out 4-byte aligned; each thread turns a float4
// into one 32-bit store of four codes.  Elements n..n_out-1 are zero-filled
// (the rows that pad M up to a multiple of 16).
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
quant_kernel(const float* __restrict__ x, int64_t n, int64_t n_out,
             const uint32_t* __restrict__ absmax_bits, uint8_t* __restrict__ out,
             float* __restrict__ dequant_out) {
  pdl_wait();
  pdl_trigger();
  const float a = absmax_prime(*absmax_bits);
  const float s = __fdiv_rn(448.0f, a);
  if (dequant_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *dequant_out = __fdiv_rn(a, 448.0f);
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * kThreads;
  int64_t done = 0;
  if (VEC) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint32_t* o4 = reinterpret_cast<uint32_t*>(out);
    const int64_t n4 = n >> 2;
    int64_t i = tid;
    for (; i + 3 * nthreads < n4; i += 4 * nthreads) {
      const float4 v0 = __ldg(x4 + i), v1 = __ldg(x4 + i + nthreads);
      const float4 v2 = __ldg(x4 + i + 2 * nthreads), v3 = __ldg(x4 + i + 3 * nthreads);
      o4[i] = pack4(v0, s);
      o4[i + nthreads] = pack4(v1, s);
      o4[i + 2 * nthreads] = pack4(v2, s);
      o4[i + 3 * nthreads] = pack4(v3, s);
    }
    for (; i < n4; i += nthreads) o4[i] = pack4(__ldg(x4 + i), s);
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < n; i += nthreads)
    out[i] = (uint8_t)e4m3_scaled(__ldg(x + i), s);
  for (int64_t i = n + tid; i < n_out; i += nthreads) out[i] = 0;
}

// ------------------------------------------------------ one-pass variant --
//
// One wave of CTAs (one per SM).  Each CTA holds a stash of up to `stash4`
// float4s of x in shared memory (one bulk copy; the stashes are the last
// float4s of x), and the CTAs stream the rest, the head at the front of x,
// together through registers while the copies land, reducing the max of
// both; all CTAs meet at a grid barrier that publishes the tensor max; the
// head is then read again, newest lines first (they are the likeliest to be
// in L2), and encoded with each CTA's stash from shared memory.  When the
// stashes hold all of x (the activations of 2048 tokens x 3584) x is read
// from HBM once; the launcher takes this kernel only while the head is
// small enough to stay largely in L2 between the passes.  Same arithmetic
// as absmax_kernel + quant_kernel, so the bytes are identical.
//
// Grid barrier of the one-pass kernel, on 64-bit words that each carry a
// launch tag (high half) and a maximum |x| bits (low half), written and read
// whole, so no fences or atomics are needed:
// state: the tag of the last launch and its tensor maximum (zero before the
//        first launch); a launch's tag is that tag + 1, read by every CTA
//        at its start;
// slots: one word per SM; CTA i of a launch writes (tag, its maximum) to
//        slot i.  CTA 0 waits until the slots of all CTAs carry the tag,
//        then writes (tag, tensor maximum) to `state`, which the other CTAs
//        wait for.  (Every CTA has read `state` before CTA 0 can write it,
//        since CTA 0 first waits for every CTA's slot.)
// Launches that share the words run one after another (one stream).

__device__ unsigned int g_quant_error;

constexpr int kFusedThreads = 1024;
constexpr int kFusedParts = 1;               // bulk copies (and barriers) per CTA
constexpr int64_t kFusedMinChunk = 4096;     // floats: fewer CTAs for small tensors
constexpr int64_t kFusedSmemMax = 220 * 1024;

__device__ __forceinline__ uint64_t ld_relaxed_u64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Running max |x| over four values, NaN skipped (fmaxf returns the other
// operand; no flush of subnormals in this build, so the bits of the result
// are the largest non-NaN |x| bits), and a running sum of x * 0, which
// stays zero while every value is finite and is NaN once one is not.
__device__ __forceinline__ void max4_f(float& mf, float& nf, float4 v) {
  mf = fmaxf(mf, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  nf = fmaf(v.x, 0.0f, nf);
  nf = fmaf(v.y, 0.0f, nf);
  nf = fmaf(v.z, 0.0f, nf);
  nf = fmaf(v.w, 0.0f, nf);
}

// Block maximum and non-finite flag of the threads' running values (mf, nf
// of max4_f), then the grid barrier on the tagged words described above.
// On return (after a block barrier) absmax_s holds the tensor's maximum |x|
// bits and nonfinite_s whether this CTA's part of x held a NaN or an
// infinity.  tag_s: this launch's tag, read from `state` before the call.
// NW: warps of the block.
template <int NW>
__device__ __forceinline__ void one_pass_grid_max(float mf, float nf, uint32_t (&warp_max)[NW],
                                                  uint32_t (&warp_nf)[NW], const uint32_t& tag_s,
                                                  unsigned long long* state,
                                                  unsigned long long* slots, uint32_t& absmax_s,
                                                  uint32_t& nonfinite_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mf));
  const uint32_t bad = __any_sync(0xFFFFFFFFu, !(nf == 0.0f)) ? 1u : 0u;
  if (lane == 0) {
    warp_max[warp] = m;
    warp_nf[warp] = bad;
  }
  __syncthreads();

  if (warp == 0) {
    m = __reduce_max_sync(0xFFFFFFFFu, lane < NW ? warp_max[lane] : 0u);
    const uint32_t any_bad = __reduce_or_sync(0xFFFFFFFFu, lane < NW ? warp_nf[lane] : 0u);
    const uint32_t tag = tag_s;
    if (lane == 0) {
      nonfinite_s = any_bad;
      st_relaxed_u64(slots + blockIdx.x, ((uint64_t)tag << 32) | m);
    }
    uint32_t all = 0;
    const uint64_t t0 = globaltimer();
    if (blockIdx.x == 0) {
      // every CTA's maximum, then the tensor's for the others
      while (true) {
        bool done = true;
        uint32_t mm = 0;
        for (int i = lane; i < (int)gridDim.x; i += 32) {
          const uint64_t v = ld_relaxed_u64(slots + i);
          done = done && (uint32_t)(v >> 32) == tag;
          mm = max(mm, (uint32_t)v);
        }
        all = __reduce_max_sync(0xFFFFFFFFu, mm);
        if (__all_sync(0xFFFFFFFFu, done)) break;
        if (globaltimer() - t0 > kWaitLimitNs) {
          if (lane == 0) atomicOr(&g_quant_error, 2u);
          break;
        }
      }
      if (lane == 0) st_relaxed_u64(state, ((uint64_t)tag << 32) | all);
    } else {
      uint64_t v = ld_relaxed_u64(state);
      while ((uint32_t)(v >> 32) != tag) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          if (lane == 0) atomicOr(&g_quant_error, 2u);
          break;
        }
        v = ld_relaxed_u64(state);
      }
      all = (uint32_t)v;
    }
    if (lane == 0) absmax_s = all;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFusedThreads, 1)
act_quant_fused_kernel(const float* __restrict__ x, int64_t n, int64_t n_out,
                       int64_t chunk, int64_t stash4, uint8_t* __restrict__ out,
                       uint32_t* __restrict__ absmax_out, float* __restrict__ dequant_out,
                       unsigned long long* state, unsigned long long* slots) {
  extern __shared__ __align__(128) float4 stash[];
  __shared__ __align__(8) uint64_t bars[kFusedParts];
  __shared__ uint32_t warp_max[kFusedThreads / 32], warp_nf[kFusedThreads / 32];
  __shared__ uint32_t absmax_s, nonfinite_s, tag_s;

  // The whole float4s of x: the last G * S of them are the CTAs' stashes
  // (CTA i holds [hs + i*S, hs + (i+1)*S) in shared memory, the last one
  // possibly fewer); the first hs, the head, are streamed by all CTAs
  // together (thread g of the grid takes float4s g, g + T, ...), once for
  // the max and once to encode.  The n % 4 last values go to the last CTA.
  (void)chunk;
  const int64_t n4 = n >> 2;
  const int64_t G = gridDim.x;
  const int64_t S = min(stash4, (n4 + G - 1) / G);
  const int64_t hs = n4 - min(n4, G * S);
  const int64_t s_lo = min(n4, hs + (int64_t)blockIdx.x * S);
  const int64_t s4 = min(n4, s_lo + S) - s_lo;  // this CTA's stash
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const int tid = threadIdx.x;
  const int64_t g = (int64_t)blockIdx.x * kFusedThreads + tid, T = G * kFusedThreads;
  const bool last_cta = blockIdx.x == gridDim.x - 1;

  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    for (int p = 0; p < kFusedParts; ++p) mbar_init(smem_u32(&bars[p]), 1);
    mbar_fence_init();
    for (int p = 0; p < kFusedParts; ++p) {
      const int64_t lo = s4 * p / kFusedParts, hi = s4 * (p + 1) / kFusedParts;
      const uint32_t bytes = (uint32_t)((hi - lo) * 16);
      mbar_arrive_expect_tx(smem_u32(&bars[p]), bytes);
      // read once: evict_first
      if (bytes != 0)
        bulk_g2s_hint(smem_u32(stash + lo), x4 + s_lo + lo, bytes, smem_u32(&bars[p]),
                      l2_policy_evict_first());
    }
  }
  if (tid == 32) tag_s = (uint32_t)(ld_relaxed_u64(state) >> 32) + 1u;
  __syncthreads();

  float mf = 0.0f, nf = 0.0f;
  {
    // the head is read again after the barrier: ask L2 to keep it
    const uint64_t keep = l2_policy_evict_last();
    int64_t i = g;
    for (; i + 3 * T < hs; i += 4 * T) {
      const float4 v0 = ldg_f4_policy(x4 + i, keep);
      const float4 v1 = ldg_f4_policy(x4 + i + T, keep);
      const float4 v2 = ldg_f4_policy(x4 + i + 2 * T, keep);
      const float4 v3 = ldg_f4_policy(x4 + i + 3 * T, keep);
      max4_f(mf, nf, v0);
      max4_f(mf, nf, v1);
      max4_f(mf, nf, v2);
      max4_f(mf, nf, v3);
    }
    for (; i < hs; i += T) max4_f(mf, nf, ldg_f4_policy(x4 + i, keep));
  }
  for (int p = 0; p < kFusedParts; ++p) {
    mbar_wait(smem_u32(&bars[p]), 0, kWaitLimitNs, &g_quant_error);
    const int64_t lo = s4 * p / kFusedParts, hi = s4 * (p + 1) / kFusedParts;
    for (int64_t i = lo + tid; i < hi; i += kFusedThreads) max4_f(mf, nf, stash[i]);
  }
  if (last_cta)
    for (int64_t i = (n4 << 2) + tid; i < n; i += kFusedThreads) {
      const float v = __ldg(x + i);
      mf = fmaxf(mf, fabsf(v));
      nf = fmaf(v, 0.0f, nf);
    }
  one_pass_grid_max<kFusedThreads / 32>(mf, nf, warp_max, warp_nf, tag_s, state, slots, absmax_s,
                                        nonfinite_s);

  const float a = absmax_prime(absmax_s);
  const float s = __fdiv_rn(448.0f, a);
  if (blockIdx.x == 0 && tid == 0) {
    if (absmax_out != nullptr) *absmax_out = absmax_s;
    if (dequant_out != nullptr) *dequant_out = __fdiv_rn(a, 448.0f);
  }
  uint32_t* o4 = reinterpret_cast<uint32_t*>(out);
  const uint64_t last_use = l2_policy_evict_first();
  // this thread's head float4s again, the last rounds first (the lines read
  // last are the likeliest to be in L2)
  const bool finite = nonfinite_s == 0u;  // every value this CTA read is finite
  if (hs > 0)
    for (int64_t base = ((hs - 1) / (4 * T)) * (4 * T); base >= 0; base -= 4 * T) {
      float4 v[4];
#pragma unroll
      for (int u = 3; u >= 0; --u) {
        const int64_t i = base + u * T + g;
        if (i < hs) v[u] = ldg_f4_policy(x4 + i, last_use);
      }
#pragma unroll
      for (int u = 3; u >= 0; --u) {
        const int64_t i = base + u * T + g;
        if (i < hs) o4[i] = finite ? e4m3_scaled4_finite(v[u], s) : pack4(v[u], s);
      }
    }
  if (finite) {
    for (int64_t i = tid; i < s4; i += kFusedThreads)
      o4[s_lo + i] = e4m3_scaled4_finite(stash[i], s);
  } else {
    for (int64_t i = tid; i < s4; i += kFusedThreads) o4[s_lo + i] = pack4(stash[i], s);
  }
  if (last_cta)
    for (int64_t i = (n4 << 2) + tid; i < n; i += kFusedThreads)
      out[i] = (uint8_t)e4m3_scaled(__ldg(x + i), s);
  const int64_t stride = (int64_t)gridDim.x * kFusedThreads;
  for (int64_t i = n + (int64_t)blockIdx.x * kFusedThreads + tid; i < n_out; i += stride)
    out[i] = 0;
}

// ------------------------------------------- one-pass, register variant --
//
// For tensors that fit on chip in one wave: each CTA holds up to 512 x 24
// float4s of x in its threads' registers (7.47 M values on 152 SMs, the
// 2048 x 3584 activations included) and up to 220 KB more in shared memory
// (63 MB in all: the 4096 x 3584 activations).  Each thread loads its
// float4s straight into registers (all loads in flight at once, read once:
// evict_first), the rest of the CTA's part arrives by one bulk copy; the
// maximum is taken as they land, the CTAs meet at the same grid barrier as
// act_quant_fused_kernel, and each encodes from its registers and shared
// memory.  The register part is not read from shared memory twice (once for
// the maximum, once to encode) as the shared-memory stash is.  CTA i owns
// float4s [i*per4, (i+1)*per4): thread t takes float4s t, t + 512, ... of
// its first 512 * 24, the bulk copy the rest.  Same arithmetic as
// absmax_kernel + quant_kernel, so the bytes are identical.

constexpr int kRegThreads = 512;
constexpr int kRegVec = 24;  // float4s of x per thread

__global__ void __launch_bounds__(kRegThreads, 1)
act_quant_reg_kernel(const float* __restrict__ x, int64_t n, int64_t n_out, int64_t per4,
                     uint8_t* __restrict__ out, uint32_t* __restrict__ absmax_out,
                     float* __restrict__ dequant_out, unsigned long long* state,
                     unsigned long long* slots) {
  extern __shared__ __align__(128) float4 rstash[];
  __shared__ __align__(8) uint64_t rbar;
  __shared__ uint32_t warp_max[kRegThreads / 32], warp_nf[kRegThreads / 32];
  __shared__ uint32_t absmax_s, nonfinite_s, tag_s;
  const int64_t n4 = n >> 2;
  const int64_t lo = min(n4, (int64_t)blockIdx.x * per4);
  const int64_t cnt = min(n4, lo + per4) - lo;  // this CTA's float4s
  const int64_t rcnt = min(cnt, (int64_t)kRegThreads * kRegVec);  // in registers
  const int64_t scnt = cnt - rcnt;  // in shared memory, <= kFusedSmemMax / 16
  const float4* x4 = reinterpret_cast<const float4*>(x) + lo;
  const int tid = threadIdx.x;
  const bool last_cta = blockIdx.x == gridDim.x - 1;

  pdl_wait();
  pdl_trigger();
  if (tid == 0 && scnt > 0) {
    const uint32_t b = smem_u32(&rbar);
    mbar_init(b, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(b, (uint32_t)(scnt * 16));
    bulk_g2s_hint(smem_u32(rstash), x4 + rcnt, (uint32_t)(scnt * 16), b, l2_policy_evict_first());
  }
  if (tid == 32) tag_s = (uint32_t)(ld_relaxed_u64(state) >> 32) + 1u;
  const uint64_t once = l2_policy_evict_first();
  float4 v[kRegVec];
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) {
    const int64_t i = tid + (int64_t)k * kRegThreads;
    v[k] = i < rcnt ? ldg_f4_policy(x4 + i, once) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float mf = 0.0f, nf = 0.0f;  // the zeros of absent float4s change neither
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) max4_f(mf, nf, v[k]);
  __syncthreads();  // the barrier's initialization is visible to every thread
  if (scnt > 0) {
    mbar_wait(smem_u32(&rbar), 0, kWaitLimitNs, &g_quant_error);
    for (int64_t i = tid; i < scnt; i += kRegThreads) max4_f(mf, nf, rstash[i]);
  }
  if (last_cta)
    for (int64_t i = (n4 << 2) + tid; i < n; i += kRegThreads) {
      const float w = __ldg(x + i);
      mf = fmaxf(mf, fabsf(w));
      nf = fmaf(w, 0.0f, nf);
    }
  one_pass_grid_max<kRegThreads / 32>(mf, nf, warp_max, warp_nf, tag_s, state, slots, absmax_s,
                                      nonfinite_s);

  const float a = absmax_prime(absmax_s);
  const float s = __fdiv_rn(448.0f, a);
  if (blockIdx.x == 0 && tid == 0) {
    if (absmax_out != nullptr) *absmax_out = absmax_s;
    if (dequant_out != nullptr) *dequant_out = __fdiv_rn(a, 448.0f);
  }
  uint32_t* o4 = reinterpret_cast<uint32_t*>(out) + lo;
  if (nonfinite_s == 0u) {  // every value this CTA read is finite
#pragma unroll
    for (int k = 0; k < kRegVec; ++k) {
      const int64_t i = tid + (int64_t)k * kRegThreads;
      if (i < rcnt) o4[i] = e4m3_scaled4_finite(v[k], s);
    }
    for (int64_t i = tid; i < scnt; i += kRegThreads)
      o4[rcnt + i] = e4m3_scaled4_finite(rstash[i], s);
  } else {
#pragma unroll
    for (int k = 0; k < kRegVec; ++k) {
      const int64_t i = tid + (int64_t)k * kRegThreads;
      if (i < rcnt) o4[i] = pack4(v[k], s);
    }
    for (int64_t i = tid; i < scnt; i += kRegThreads) o4[rcnt + i] = pack4(rstash[i], s);
  }
  if (last_cta)
    for (int64_t i = (n4 << 2) + tid; i < n; i += kRegThreads)
      out[i] = (uint8_t)e4m3_scaled(__ldg(x + i), s);
  const int64_t stride = (int64_t)gridDim.x * kRegThreads;
  for (int64_t i = n + (int64_t)blockIdx.x * kRegThreads + tid; i < n_out; i += stride)
    out[i] = 0;
}

int64_t fused_chunk(int64_t n) {
  const int64_t sms = device_sm_count();
  int64_t c = (n + sms - 1) / sms;
  c = (c + 3) & ~int64_t(3);
  return c < kFusedMinChunk ? kFusedMinChunk : c;
}

// ------------------------------------------------- two-pass, slot variant --
//
// For the activation cache: absmax_slots_kernel writes each CTA's partial
// maximum to its own slot (no zeroing and no atomics needed), and
// quant_slots_kernel reduces the slots at its start and then encodes the
// tensor walking it backwards, so that whatever of x the first pass left in
// L2 (what it read last) is read first.  Same arithmetic as absmax_kernel +
// quant_kernel, hence the same bytes.

constexpr int kSlotUnroll = 4;  // float4 loads in flight per thread


// Each slot: the CTA's maximum |x| bits (NaN skipped) in bits 0..30, and
// bit 31 set when its part of x holds a NaN or an infinity.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
absmax_slots_kernel(const float* __restrict__ x, int64_t n, uint32_t* __restrict__ slots) {
  pdl_wait();
  pdl_trigger();
  float mf = 0.0f, nf = 0.0f;
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * kThreads;
  int64_t done = 0;
  if (VEC) {
    // streamed with L2 priority evict_first (measured on GB300: asking L2
    // to keep the tail of x for the encoder with evict_last made the pair
    // of kernels slower, 55.4 -> 57.1 us at 2048 x 18944)
    const uint64_t pol = l2_policy_evict_first();
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t n4 = n >> 2;
    int64_t i = tid;
    for (; i + (kSlotUnroll - 1) * nthreads < n4; i += kSlotUnroll * nthreads) {
      float4 v[kSlotUnroll];
#pragma unroll
      for (int u = 0; u < kSlotUnroll; ++u) v[u] = ldg_f4_policy(x4 + i + u * nthreads, pol);
#pragma unroll
      for (int u = 0; u < kSlotUnroll; ++u) max4_f(mf, nf, v[u]);
    }
    for (; i < n4; i += nthreads) max4_f(mf, nf, __ldg(x4 + i));
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < n; i += nthreads) {
    const float v = __ldg(x + i);
    mf = fmaxf(mf, fabsf(v));
    nf = fmaf(v, 0.0f, nf);
  }
  __shared__ uint32_t warp_max[kThreads / 32];
  uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mf));
  if (__any_sync(0xFFFFFFFFu, !(nf == 0.0f))) m |= 0x80000000u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_max[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kThreads / 32 ? warp_max[lane] : 0u;
    const uint32_t bad = __reduce_or_sync(0xFFFFFFFFu, m) & 0x80000000u;
    m = __reduce_max_sync(0xFFFFFFFFu, m & 0x7FFFFFFFu);
    if (lane == 0) slots[blockIdx.x] = m | bad;
  }
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
quant_slots_kernel(const float* __restrict__ x, int64_t n, int64_t n_out,
                   const uint32_t* __restrict__ slots, int nslots, uint8_t* __restrict__ out,
                   uint32_t* __restrict__ absmax_out, float* __restrict__ dequant_out) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t warp_max[kThreads / 32];
  __shared__ uint32_t absmax_s, bad_s;
  uint32_t m = 0, bad = 0;
  for (int i = threadIdx.x; i < nslots; i += kThreads) {
    const uint32_t v = slots[i];
    m = max(m, v & 0x7FFFFFFFu);
    bad |= v;
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m) | (__reduce_or_sync(0xFFFFFFFFu, bad) & 0x80000000u);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_max[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kThreads / 32 ? warp_max[lane] : 0u;
    bad = __reduce_or_sync(0xFFFFFFFFu, m) >> 31;
    m = __reduce_max_sync(0xFFFFFFFFu, m & 0x7FFFFFFFu);
    if (lane == 0) {
      absmax_s = m;
      bad_s = bad;
    }
  }
  __syncthreads();
  const uint32_t bits = absmax_s;
  const float a = absmax_prime(bits);
  const float s = __fdiv_rn(448.0f, a);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (absmax_out != nullptr) *absmax_out = bits;
    if (dequant_out != nullptr) *dequant_out = __fdiv_rn(a, 448.0f);
  }
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * kThreads;
  int64_t done = 0;
  if (VEC) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint32_t* o4 = reinterpret_cast<uint32_t*>(out);
    const int64_t n4 = n >> 2;
    // rounds of kSlotUnroll * nthreads float4s, the last (partial) round
    // first, then backwards
    const int64_t per_round = kSlotUnroll * nthreads;
    const uint64_t last_use = l2_policy_evict_first();
    const bool finite = bad_s == 0u;  // no NaN or infinity anywhere in x
    for (int64_t base = ((n4 - 1) / per_round) * per_round; base >= 0 && n4 > 0;
         base -= per_round) {
      float4 v[kSlotUnroll];
#pragma unroll
      for (int u = 0; u < kSlotUnroll; ++u) {
        const int64_t i = base + u * nthreads + tid;
        if (i < n4) v[u] = ldg_f4_policy(x4 + i, last_use);
      }
      if (finite) {
#pragma unroll
        for (int u = 0; u < kSlotUnroll; ++u) {
          const int64_t i = base + u * nthreads + tid;
          if (i < n4) o4[i] = e4m3_scaled4_finite(v[u], s);
        }
      } else {
#pragma unroll
        for (int u = 0; u < kSlotUnroll; ++u) {
          const int64_t i = base + u * nthreads + tid;
          if (i < n4) o4[i] = pack4(v[u], s);
        }
      }
    }
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < n; i += nthreads)
    out[i] = (uint8_t)e4m3_scaled(__ldg(x + i), s);
  for (int64_t i = n + tid; i < n_out; i += nthreads) out[i] = 0;
}

// ------------------------------------------------- one-cluster variant --
//
// Small activations (the inputs of a few tokens) in one launch: a single
// thread-block cluster streams x for the max, exchanges the CTAs' maxima
// through distributed shared memory behind the cluster barrier, and reads x
// again, now from L2, to encode it.  No grid barrier and no second launch;
// the same arithmetic as absmax_kernel + quant_kernel, hence the same bytes.

constexpr int kClusterThreads = 1024;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// A word in the shared memory of CTA `rank` of the cluster, at the offset of
// `local` in this CTA.
__device__ __forceinline__ uint32_t ld_peer_u32(const uint32_t* local, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// x 16-byte and out 4-byte aligned (the launcher checks).
__global__ void __launch_bounds__(kClusterThreads, 1)
act_quant_cluster_kernel(const float* __restrict__ x, int64_t n, int64_t n_out,
                         uint8_t* __restrict__ out, uint32_t* __restrict__ absmax_out,
                         float* __restrict__ dequant_out) {
  __shared__ uint32_t warp_max[kClusterThreads / 32];
  __shared__ uint32_t cta_max, all_max;
  pdl_wait();
  pdl_trigger();
  const uint32_t rank = cluster_ctarank(), ncta = cluster_nctarank();
  const int64_t tid = (int64_t)rank * kClusterThreads + threadIdx.x;
  const int64_t nthreads = (int64_t)ncta * kClusterThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const int64_t n4 = n >> 2;

  // pass 1: this CTA's max, from HBM (or from L2 when x was just written)
  uint32_t m = 0;
  {
    int64_t i = tid;
    for (; i + 3 * nthreads < n4; i += 4 * nthreads) {
      const float4 a = __ldg(x4 + i), b = __ldg(x4 + i + nthreads);
      const float4 c = __ldg(x4 + i + 2 * nthreads), d = __ldg(x4 + i + 3 * nthreads);
      m = max4(max4(m, a), b);
      m = max4(max4(m, c), d);
    }
    for (; i < n4; i += nthreads) m = max4(m, __ldg(x4 + i));
    for (int64_t j = (n4 << 2) + tid; j < n; j += nthreads)
      m = max(m, abs_bits_skip_nan(__ldg(x + j)));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) warp_max[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = warp_max[lane];
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) cta_max = m;
  }
  // every CTA's maximum is in its shared memory
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (warp == 0) {
    m = (uint32_t)lane < ncta ? ld_peer_u32(&cta_max, (uint32_t)lane) : 0u;
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) all_max = m;
  }
  // this CTA has read its peers' maxima; it waits at the end of the kernel
  // until every CTA has, so that no shared memory is read after it is gone
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  __syncthreads();

  // pass 2: encode with the tensor's scale; x is read again from L2
  const uint32_t bits = all_max;
  const float a = absmax_prime(bits);
  const float s = __fdiv_rn(448.0f, a);
  if (rank == 0 && threadIdx.x == 0) {
    if (absmax_out != nullptr) *absmax_out = bits;
    if (dequant_out != nullptr) *dequant_out = __fdiv_rn(a, 448.0f);
  }
  {
    uint32_t* o4 = reinterpret_cast<uint32_t*>(out);
    int64_t i = tid;
    for (; i + 3 * nthreads < n4; i += 4 * nthreads) {
      const float4 v0 = __ldg(x4 + i), v1 = __ldg(x4 + i + nthreads);
      const float4 v2 = __ldg(x4 + i + 2 * nthreads), v3 = __ldg(x4 + i + 3 * nthreads);
      o4[i] = pack4(v0, s);
      o4[i + nthreads] = pack4(v1, s);
      o4[i + 2 * nthreads] = pack4(v2, s);
      o4[i + 3 * nthreads] = pack4(v3, s);
    }
    for (; i < n4; i += nthreads) o4[i] = pack4(__ldg(x4 + i), s);
    for (int64_t j = (n4 << 2) + tid; j < n; j += nthreads)
      out[j] = (uint8_t)e4m3_scaled(__ldg(x + j), s);
    for (int64_t j = n + tid; j < n_out; j += nthreads) out[j] = 0;
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

int grid_for(int64_t work_items) {
  const int64_t per_wave = (int64_t)device_sm_count() * 4;  // 4 CTAs / SM
  int64_t blocks = (work_items + kThreads - 1) / kThreads;
  if (blocks > per_wave) blocks = per_wave;
  return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

rq_status launch_absmax(const float* x, int64_t n, uint32_t* absmax_bits,
                        cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(absmax_bits, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return RQ_ERR_CUDA;
  if (n == 0) return RQ_OK;
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const int grid = grid_for(vec ? (n + 3) / 4 : n);
  if (vec) return launch_kernel(absmax_kernel<true>, grid, kThreads, 0, st, x, n, absmax_bits);
  return launch_kernel(absmax_kernel<false>, grid, kThreads, 0, st, x, n, absmax_bits);
}

rq_status launch_quant(const float* x, int64_t n, int64_t n_out,
                       const uint32_t* absmax_bits, uint8_t* out,
                       float* dequant_out, cudaStream_t st) {
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 3) == 0;
  const int grid = grid_for(vec ? (n_out + 3) / 4 : n_out);
  if (vec)
    return launch_kernel(quant_kernel<true>, grid, kThreads, 0, st, x, n, n_out, absmax_bits,
                         out, dequant_out);
  return launch_kernel(quant_kernel<false>, grid, kThreads, 0, st, x, n, n_out, absmax_bits, out,
                       dequant_out);
}

int act_quant_slots() { return device_sm_count() * 4; }

rq_status launch_act_quant_two_pass(const float* x, int64_t n, int64_t n_out, uint8_t* out,
                                    uint32_t* slots, uint32_t* absmax_out,
                                    float* dequant_out, cudaStream_t st) {
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 3) == 0;
  const int nslots = act_quant_slots();
  int g1 = grid_for(vec ? (n + 3) / 4 : n);
  if (g1 > nslots) g1 = nslots;
  rq_status s = vec ? launch_kernel(absmax_slots_kernel<true>, g1, kThreads, 0, st, x, n, slots)
                    : launch_kernel(absmax_slots_kernel<false>, g1, kThreads, 0, st, x, n, slots);
  if (s != RQ_OK) return s;
  const int g2 = grid_for(vec ? (n_out + 3) / 4 : n_out);
  if (vec)
    return launch_kernel(quant_slots_kernel<true>, g2, kThreads, 0, st, x, n, n_out,
                         (const uint32_t*)slots, g1, out, absmax_out, dequant_out);
  return launch_kernel(quant_slots_kernel<false>, g2, kThreads, 0, st, x, n, n_out,
                       (const uint32_t*)slots, g1, out, absmax_out, dequant_out);
}

// CTAs of the one-cluster kernel: 16 (a size beyond the portable 8) where
// the GPU schedules such a cluster of these CTAs, else 8.
int act_quant_cluster_ctas() {
  static int ctas = 0;
  if (ctas != 0) return ctas;
  ctas = 8;
  if (cudaFuncSetAttribute(act_quant_cluster_kernel,
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(kClusterThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, act_quant_cluster_kernel, &cfg) ==
            cudaSuccess &&
        n >= 1)
      ctas = 16;
  }
  cudaGetLastError();  // a refused attribute or query leaves no error behind
  return ctas;
}

rq_status launch_act_quant_cluster(const float* x, int64_t n, int64_t n_out, uint8_t* out,
                                   uint32_t* absmax_out, float* dequant_out,
                                   cudaStream_t st) {
  if ((reinterpret_cast<uintptr_t>(x) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 3) != 0)
    return RQ_ERR_SHAPE;
  const int ctas = act_quant_cluster_ctas();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, act_quant_cluster_kernel, x, n, n_out, out,
                                        absmax_out, dequant_out));
}

// Heads (the parts of the chunks beyond shared memory) up to this many bytes
// in all.  The heads are loaded with L2 priority evict_last on the first
// pass and evict_first on the second, the on-chip parts with evict_first.
// Measured on GB300 (graph-replayed, alone; one kernel against two): 512 x
// 18944, 5 MB of heads: 11.9 against 17.9 us; 1024 x 18944, 54 MB: 22.6
// against 30.4; 4096 x 3584, 25 MB: 17.4 against 24.3; 2048 x 18944,
// 121 MB: 55.7 against 54.2.  In the 28-layer stack, whose weights share L2
// (eager ms per pass, 16 MB cap against 128 MB): 1024 tokens 6.84 / 6.67,
// 2048 tokens 12.53 / 12.44, but 4096 tokens 23.4 / 23.8, the 25 MB heads
// of its 4096 x 3584 activations costing the GEMMs after them more than
// they save.  So up to 16 MB of heads in general, up to 128 MB for tensors
// of at least 2^24 elements; RQ_ONE_PASS_HEAD_MB sets one cap for all
// (tuning).
constexpr int64_t kFusedHeadMax = 16ll << 20;
constexpr int64_t kFusedHeadMaxLarge = 128ll << 20;
constexpr int64_t kFusedLargeElems = 1ll << 24;

int64_t fused_stash4(int64_t chunk) {
  return std::min<int64_t>(chunk / 4, kFusedSmemMax / 16);
}

// The register form of the one-pass kernel takes x when every CTA of one
// wave of g keeps its part on chip (at least one float4 per thread, at most
// 512 x 24 in registers plus 220 KB in shared memory); *per4 gets the
// float4s per CTA.  RQ_QUANT_REG=0 turns it off (tuning).
bool act_quant_reg_fits(int64_t n, int g, int64_t* per4) {
  const char* e = std::getenv("RQ_QUANT_REG");
  if (g <= 0 || (e != nullptr && std::atoi(e) == 0)) return false;
  const int64_t n4 = n >> 2;
  *per4 = (n4 + g - 1) / g;
  return n4 >= (int64_t)g * kRegThreads &&
         *per4 <= (int64_t)kRegThreads * kRegVec + kFusedSmemMax / 16;
}

bool act_quant_fused_fits(const float* x, int64_t n, const uint8_t* out) {
  if (n <= 0 || (reinterpret_cast<uintptr_t>(x) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(out) & 3) != 0)
    return false;
  int64_t per4 = 0;
  if (act_quant_reg_fits(n, device_sm_count(), &per4)) return true;
  const int64_t chunk = fused_chunk(n);
  const int64_t grid = (n + chunk - 1) / chunk;
  const int64_t head_bytes = 4 * n - 16 * grid * fused_stash4(chunk);
  static int64_t cap = -2;
  if (cap == -2) {
    const char* e = std::getenv("RQ_ONE_PASS_HEAD_MB");
    cap = e != nullptr ? (int64_t)std::atoll(e) << 20 : -1;
  }
  if (cap >= 0) return head_bytes <= cap;
  return head_bytes <= (n >= kFusedLargeElems ? kFusedHeadMaxLarge : kFusedHeadMax);
}

rq_status launch_act_quant_fused(const float* x, int64_t n, int64_t n_out,
                                 uint8_t* out, uint32_t* absmax_out,
                                 float* dequant_out, unsigned long long* state,
                                 unsigned long long* slots, int nslots, cudaStream_t st) {
  if (!act_quant_fused_fits(x, n, out)) return RQ_ERR_SHAPE;
  {
    // x held on chip in registers (and shared memory) when it fits one wave.
    // Measured on GB300 (graph-replayed, against the shared-memory form or,
    // where that does not take x, the two kernels): 2048 x 3584 10.3 -> 9.3
    // us (all in registers), 4096 x 3584 24.4 -> 15.6 us; the 28-layer stack
    // at 4096 tokens ~22.1 -> 21.5 ms eager, at 512 tokens 4.57 -> 4.51 ms.
    int64_t per4 = 0;
    if (act_quant_reg_fits(n, std::min(device_sm_count(), nslots), &per4)) {
      const int64_t s4 = per4 - (int64_t)kRegThreads * kRegVec;
      const size_t smem = s4 > 0 ? (size_t)s4 * 16 : 0;
      static bool reg_attr = false;
      if (!reg_attr) {
        if (cudaFuncSetAttribute(act_quant_reg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kFusedSmemMax) != cudaSuccess)
          return launch_status();
        reg_attr = true;
      }
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(((n >> 2) + per4 - 1) / per4));
      cfg.blockDim = dim3(kRegThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = st;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = pdl_enabled() ? 2 : 1;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, act_quant_reg_kernel, x, n, n_out, per4,
                                               out, absmax_out, dequant_out, state, slots);
      if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return RQ_ERR_SHAPE;
      }
      return cuda_status(e);
    }
  }
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(act_quant_fused_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFusedSmemMax) != cudaSuccess)
      return launch_status();
    attr_set = true;
  }
  int64_t chunk = fused_chunk(n);
  const int grid = (int)((n + chunk - 1) / chunk);
  if (grid > nslots) return RQ_ERR_SHAPE;
  const int64_t stash4 = fused_stash4(chunk);
  const size_t smem = (size_t)stash4 * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, act_quant_fused_kernel, x, n, n_out, chunk,
                                           stash4, out, absmax_out, dequant_out, state, slots);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return RQ_ERR_SHAPE;
  }
  return cuda_status(e);
}

rq_status read_and_clear_quant_error() {
  unsigned int v = 0;
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(v)) != cudaSuccess) return RQ_ERR_CUDA;
  if (v == 0) return RQ_OK;
  if (cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(zero)) != cudaSuccess) return RQ_ERR_CUDA;
  return RQ_ERR_TIMEOUT;
}

}  // namespace rq
