// rq_wcache.cu -- one-time FP8 weight-cache build from GGUF Q4_K / Q6_K.
//
// realizar 0.8.4, cublas_prefill/gemm.rs, get_or_cache_fp8_weight: dequant
// the packed weight, take its absmax, encode with 448/absmax', keep
// absmax'/448 as the weight's dequant scale.  Here the dequant scale stays in
// device memory and no fp32 scratch is used: pass 1 decodes and reduces the
// absmax, pass 2 decodes again and encodes.  Both passes evaluate every weight
// in the same fixed fp32 order, w = (d*sc)*q - dmin*m for Q4_K and
// (d*scale)*(q-32) for Q6_K, each operation correctly rounded and never
// contracted into an FMA, so the E4M3 bytes are reproducible bit for bit.
#include "rq_device.cuh"
#include "rq_internal.h"

namespace rq {
namespace {

constexpr int kThreads = 256;

// Q4_K: one thread per 64-weight group (super-block sb, group g): weights
// 64g + l (low nibbles, sub-block 2g) and 64g + 32 + l (high, 2g+1).
struct Q4Group {
  float d, dmin, sc_lo, sc_hi, m_lo, m_hi;
  uint32_t q[8];
};

__device__ __forceinline__ Q4Group q4_group(const uint8_t* __restrict__ W,
                                            int64_t unit) {
  const int64_t blk = unit >> 2;
  const int g = (int)(unit & 3);
  const uint8_t* p = W + blk * kQ4KBytes;
  const uint4 h = ldg_nc_v4(p);
  const uint4 a = ldg_nc_v4(p + 16 + 32 * g);
  const uint4 b = ldg_nc_v4(p + 32 + 32 * g);
  Q4Group o;
  const float2 dd = half_pair(h.x);
  o.d = dd.x;
  o.dmin = dd.y;
  const uint8_t s[12] = {
      (uint8_t)h.y, (uint8_t)(h.y >> 8), (uint8_t)(h.y >> 16), (uint8_t)(h.y >> 24),
      (uint8_t)h.z, (uint8_t)(h.z >> 8), (uint8_t)(h.z >> 16), (uint8_t)(h.z >> 24),
      (uint8_t)h.w, (uint8_t)(h.w >> 8), (uint8_t)(h.w >> 16), (uint8_t)(h.w >> 24)};
  int sc[2], mn[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int j = 2 * g + t;
    if (j < 4) {
      sc[t] = s[j] & 63;
      mn[t] = s[j + 4] & 63;
    } else {
      sc[t] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      mn[t] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
  }
  o.sc_lo = (float)sc[0];
  o.sc_hi = (float)sc[1];
  o.m_lo = (float)mn[0];
  o.m_hi = (float)mn[1];
  o.q[0] = a.x; o.q[1] = a.y; o.q[2] = a.z; o.q[3] = a.w;
  o.q[4] = b.x; o.q[5] = b.y; o.q[6] = b.z; o.q[7] = b.w;
  return o;
}

// Weight i (0..63) of the group: i < 32 low nibble of byte i, else high
// nibble of byte i - 32.
__device__ __forceinline__ float q4_weight(const Q4Group& o, int i) {
  const int byte = i & 31;
  const uint32_t word = o.q[byte >> 2] >> (8 * (byte & 3));
  const bool hi = i >= 32;
  const float q = (float)(hi ? ((word >> 4) & 15u) : (word & 15u));
  const float dsc = __fmul_rn(o.d, hi ? o.sc_hi : o.sc_lo);
  return __fsub_rn(__fmul_rn(dsc, q), __fmul_rn(o.dmin, hi ? o.m_hi : o.m_lo));
}

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

__global__ void __launch_bounds__(kThreads)
q4_absmax_kernel(const uint8_t* __restrict__ W, int64_t units, uint32_t* out) {
  pdl_wait();
  pdl_trigger();
  uint32_t m = 0;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * kThreads) {
    const Q4Group o = q4_group(W, u);
#pragma unroll 8
    for (int i = 0; i < 64; ++i) m = max(m, abs_bits_skip_nan(q4_weight(o, i)));
  }
  block_max_to(m, out);
}

// Output position of group u: row n = u / (4*nsb), k = (u % (4*nsb)) * 64;
// the 64 codes are contiguous, written as four 16-byte stores.
__global__ void __launch_bounds__(kThreads)
q4_encode_kernel(const uint8_t* __restrict__ W, int64_t units,
                 const uint32_t* __restrict__ absmax_bits, uint8_t* __restrict__ out,
                 float* __restrict__ dequant_out) {
  pdl_wait();
  pdl_trigger();
  const float a = absmax_prime(*absmax_bits);
  const float s = __fdiv_rn(448.0f, a);
  if (blockIdx.x == 0 && threadIdx.x == 0) *dequant_out = __fdiv_rn(a, 448.0f);
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * kThreads) {
    const Q4Group o = q4_group(W, u);
    uint4* dst = reinterpret_cast<uint4*>(out + u * 64);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint32_t wd[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          word |= e4m3_scaled(q4_weight(o, 16 * v + 4 * c + b), s) << (8 * b);
        wd[c] = word;
      }
      dst[v] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
  }
}

// Q6_K: one thread per 32-weight unit (block, half h, l-quad lq): weights
// 128h + 32i + 8lq + j, i = 0..3, j = 0..7.  Byte loads (one-time pass).
__device__ __forceinline__ float q6_weight(const uint8_t* __restrict__ blk, int h,
                                           int lq, int i, int j, float d) {
  const int l = 8 * lq + j;
  const uint8_t* ql = blk + 64 * h;
  const uint8_t qh = __ldg(blk + 128 + 32 * h + l);
  int q;
  switch (i) {
    case 0: q = (__ldg(ql + l) & 15) | (((qh >> 0) & 3) << 4); break;
    case 1: q = (__ldg(ql + l + 32) & 15) | (((qh >> 2) & 3) << 4); break;
    case 2: q = (__ldg(ql + l) >> 4) | (((qh >> 4) & 3) << 4); break;
    default: q = (__ldg(ql + l + 32) >> 4) | (((qh >> 6) & 3) << 4); break;
  }
  const int8_t sc = (int8_t)__ldg(blk + 192 + 8 * h + l / 16 + 2 * i);
  return __fmul_rn(__fmul_rn(d, (float)sc), (float)(q - 32));
}

__device__ __forceinline__ float q6_d(const uint8_t* blk) {
  const uint32_t lo = __ldg(blk + 208), hi = __ldg(blk + 209);
  return __half2float(__ushort_as_half((unsigned short)(lo | (hi << 8))));
}

__global__ void __launch_bounds__(kThreads)
q6_absmax_kernel(const uint8_t* __restrict__ W, int64_t units, uint32_t* out) {
  pdl_wait();
  pdl_trigger();
  uint32_t m = 0;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * kThreads) {
    const uint8_t* blk = W + (u >> 3) * kQ6KBytes;
    const int h = (int)((u >> 2) & 1), lq = (int)(u & 3);
    const float d = q6_d(blk);
    for (int i = 0; i < 4; ++i)
      for (int j = 0; j < 8; ++j)
        m = max(m, abs_bits_skip_nan(q6_weight(blk, h, lq, i, j, d)));
  }
  block_max_to(m, out);
}

__global__ void __launch_bounds__(kThreads)
q6_encode_kernel(const uint8_t* __restrict__ W, int64_t units,
                 const uint32_t* __restrict__ absmax_bits, uint8_t* __restrict__ out,
                 float* __restrict__ dequant_out) {
  pdl_wait();
  pdl_trigger();
  const float a = absmax_prime(*absmax_bits);
  const float s = __fdiv_rn(448.0f, a);
  if (blockIdx.x == 0 && threadIdx.x == 0) *dequant_out = __fdiv_rn(a, 448.0f);
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * kThreads) {
    const int64_t blkid = u >> 3;
    const uint8_t* blk = W + blkid * kQ6KBytes;
    const int h = (int)((u >> 2) & 1), lq = (int)(u & 3);
    const float d = q6_d(blk);
    uint8_t* dst = out + blkid * kQK + 128 * h + 8 * lq;  // rows are K contiguous
    for (int i = 0; i < 4; ++i) {
      uint32_t w0 = 0, w1 = 0;
      for (int j = 0; j < 4; ++j) {
        w0 |= e4m3_scaled(q6_weight(blk, h, lq, i, j, d), s) << (8 * j);
        w1 |= e4m3_scaled(q6_weight(blk, h, lq, i, j + 4, d), s) << (8 * j);
      }
      *reinterpret_cast<uint2*>(dst + 32 * i) = make_uint2(w0, w1);
    }
  }
}

int grid_for(int64_t units) {
  const int64_t cap = (int64_t)device_sm_count() * 8;
  int64_t b = (units + kThreads - 1) / kThreads;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

rq_status launch_dequant_absmax(int qtype, const uint8_t* w, int N, int K,
                                uint32_t* absmax_bits, cudaStream_t st) {
  const int64_t blocks = (int64_t)N * (K / kQK);
  if (qtype == RQ_Q4K) {
    const int64_t units = blocks * 4;
    return launch_kernel(q4_absmax_kernel, grid_for(units), kThreads, 0, st, w, units,
                         absmax_bits);
  } else if (qtype == RQ_Q6K) {
    const int64_t units = blocks * 8;
    return launch_kernel(q6_absmax_kernel, grid_for(units), kThreads, 0, st, w, units,
                         absmax_bits);
  }
  return RQ_ERR_QTYPE;
}

rq_status launch_dequant_encode(int qtype, const uint8_t* w, int N, int K,
                                const uint32_t* absmax_bits, uint8_t* out,
                                float* dequant_out, cudaStream_t st) {
  const int64_t blocks = (int64_t)N * (K / kQK);
  if (qtype == RQ_Q4K) {
    const int64_t units = blocks * 4;
    return launch_kernel(q4_encode_kernel, grid_for(units), kThreads, 0, st, w, units,
                         absmax_bits, out, dequant_out);
  } else if (qtype == RQ_Q6K) {
    const int64_t units = blocks * 8;
    return launch_kernel(q6_encode_kernel, grid_for(units), kThreads, 0, st, w, units,
                         absmax_bits, out, dequant_out);
  }
  return RQ_ERR_QTYPE;
}

}  // namespace rq
