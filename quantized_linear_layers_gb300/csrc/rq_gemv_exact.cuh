// rq_gemv_exact.cuh -- the accuracy guarantee of the decode GEMVs.
//
// The GEMV kernels compute y[n] = sum_k x[k] w(n, k) on fast paths whose
// rounding error is not a fixed fraction of sum_k |x[k] w(n, k)|: the x
// planes are fixed-point relative to a sub-block's largest |x|, and the Q4_K
// factorisation d*sc*sum(q x) - dmin*m*sum(x) cancels when a weight's two
// terms are equal.  Each fast path therefore carries a certificate per
// output: every lane bounds the error of its partial dot product p by E
// (from the magnitudes of the row's scales and of x; see each kernel) and
// contributes D = E - tau * |p|.  With D summed over the row,
//
//   sum E <= tau * sum |p|   implies   |y - y_exact| <= 1e-4 * sum_k |x_k w_k|
//
// (|p| <= sum over the lane's weights of |x_k w_k| + E, and the fp32 sums of
// y and D add far less than the 5e-6 margin between tau and 1e-4).  An output
// whose certificate fails (D > 0, or D not finite: non-finite or extreme x,
// overflow) is recomputed here in fp64: every weight is decoded exactly, each
// product x*w is exact in fp64 and the sum is rounded once to fp32 at the end.
// The recomputation is slow (fp64 on GB300) and meant for adversarial inputs;
// on the decoder's data the certificate holds with a wide margin.
#pragma once

#include "rq_device.cuh"

namespace rq {

// tau of the certificate (see above).
constexpr float kCertTau = 0.95e-4f;

// Sub-block maxima below this take the exact path: the planes' scale and its
// inverse stay normal fp32 numbers above it.
constexpr float kCertTinyMax = 0x1p-100f;

// True when an output's summed certificate D does not prove the bound.
__device__ __forceinline__ bool cert_fails(float D) {
  return !(D <= 0.0f) || !(D > -INFINITY);
}

// 16 per-lane values summed over the warp (transpose pattern: 8 + 4 + 2 + 1
// exchanging shuffles, then one plain): lane l ends with the total of slot
// (l >> 1) & 15.
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 16;
    const float send = up ? v[i] : v[i + 8], keep = up ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 8;
    const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 4;
    const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  }
  {
    const bool up = lane & 2;
    const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 2);
  }
  v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
  return v[0];
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float half_at(const uint8_t* p) {
  return __half2float(__ushort_as_half(
      (unsigned short)(p[0] | ((unsigned)p[1] << 8))));
}

// Exact dot product of one Q4_K row (K/256 super-blocks of 144 bytes: fp16
// d, fp16 dmin, 12 bytes packing eight 6-bit scales and eight 6-bit mins,
// 128 bytes of 4-bit quants) with x, by one warp; every lane returns the sum.
// Weight 64c + l (l < 32) of a super-block is the low nibble of quant byte
// 32c + l with sub-block 2c, weight 64c + 32 + l the high nibble with
// sub-block 2c + 1; the weight is d*sc_j*q - dmin*m_j, formed in fp64 from
// the exact fp32 products d*sc_j and dmin*m_j.
__device__ __noinline__ inline double q4k_row_exact(const uint8_t* row, const float* x, int K,
                                                    int lane) {
  double acc = 0.0;
  const int groups = K >> 6;  // 64-weight groups (super-block, chunk c)
  for (int u = lane; u < groups; u += 32) {
    const int sb = u >> 2, c = u & 3;
    const uint8_t* blk = row + (size_t)sb * kQ4KBytes;
    const uint8_t* s = blk + 4;
    const float d = half_at(blk), dmin = half_at(blk + 2);
    int sc[2], mn[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * c + t;
      if (j < 4) {
        sc[t] = s[j] & 63;
        mn[t] = s[j + 4] & 63;
      } else {
        sc[t] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        mn[t] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
      }
    }
    const double a0 = (double)(d * (float)sc[0]), b0 = (double)(dmin * (float)mn[0]);
    const double a1 = (double)(d * (float)sc[1]), b1 = (double)(dmin * (float)mn[1]);
    const uint8_t* qs = blk + 16 + 32 * c;
    const float* xr = x + (size_t)sb * kQK + 64 * c;
    for (int l = 0; l < 32; ++l) {
      const int b = qs[l];
      acc = fma((double)xr[l], fma(a0, (double)(b & 15), -b0), acc);
      acc = fma((double)xr[32 + l], fma(a1, (double)(b >> 4), -b1), acc);
    }
  }
  return warp_sum_f64(acc);
}

// Exact dot product of one Q6_K row (K/256 super-blocks of 210 bytes:
// ql[128], qh[64], 16 int8 scales, fp16 d) with x, by one warp.  In half h
// (weights 128h .. 128h+127) with l = 0..31, the quarters i = 0..3 hold
// weights 128h + 32i + l: the low nibble of ql[64h + l] (i = 0), of
// ql[64h + 32 + l] (i = 1), the high nibbles of the same bytes (i = 2, 3),
// with bits 2i, 2i+1 of qh[32h + l] on top, and scale 8h + l/16 + 2i; the
// weight d*scale*(q - 32) is exact in fp32.
__device__ __noinline__ inline double q6k_row_exact(const uint8_t* row, const float* x, int K,
                                                    int lane) {
  double acc = 0.0;
  for (int k = lane; k < K; k += 32) {
    const uint8_t* blk = row + (size_t)(k >> 8) * kQ6KBytes;
    const int j = k & 255, h = j >> 7, i = (j >> 5) & 3, l = j & 31;
    const uint8_t* ql = blk + 64 * h;
    const int lowbyte = ql[l + 32 * (i & 1)];
    const int low = (i < 2) ? (lowbyte & 15) : (lowbyte >> 4);
    const int high = (blk[128 + 32 * h + l] >> (2 * i)) & 3;
    const int q = low | (high << 4);
    const int scale = (int)(int8_t)blk[192 + 8 * h + l / 16 + 2 * i];
    const float d = half_at(blk + 208);
    const float w = d * (float)scale * (float)(q - 32);
    acc = fma((double)x[k], (double)w, acc);
  }
  return warp_sum_f64(acc);
}

}  // namespace rq
