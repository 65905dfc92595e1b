// rq_gemv_mma.cu -- few-token (M = 2..8) Q4_K GEMV with the dot products on
// the tensor cores.
//
// realizar 0.8.4, cublas_prefill/mod.rs (cublas_gemm_threshold: below the
// threshold the batched GEMV reads the Q4_K weights directly, 0.5625 B per
// weight) and q6k_gemv_indexed.rs (q4k_gemv_into, batched over M tokens).
// The Q4_K weight of sub-block j of a super-block is d*sc_j*q - dmin*m_j, so
//
//   sum_k x_k w_k = sum_j [ d*sc_j * sum_{k in j} q_k x_k - dmin*m_j * sum_{k in j} x_k ].
//
// With M tokens the inner sums sum_{k in j} q_k x[m, k] are a 16-row x 8-token
// x 32-weight matrix product per sub-block, which this kernel hands to
// mma.sync.m16n8k16 (f16 inputs, f32 accumulation) with exact operands:
//
//  * A (weights): the 4-bit quant itself.  A nibble in the low bits of an
//    fp16 word is the subnormal q * 2^-24, exact; a high nibble masked in
//    place (bits 4..7) is 16 q * 2^-24.  One AND per two weights (plus one
//    shift per four), no conversion; the 2^24 and 16 go into the scales.
//  * B (tokens): x times a power of two s (per token and super-block, so the
//    scaled maximum lies in [2^14, 2^15)), split into two fp16 terms
//    hi + lo with |x*s - hi - lo| <= 2^-22 |x*s| (Veltkamp's split, FP32
//    arithmetic only).  The products q*hi and q*lo are exact.  For M <= 4
//    the MMA's 8 columns hold (token, hi) and (token, lo), one MMA per
//    step; for M <= 8 the columns are tokens and hi and lo take one MMA each.
//  * The per-sub-block scale cannot ride inside the MMA's accumulation, so
//    each sub-block starts a fresh accumulator, and P = sum_j sc_j D_j is
//    formed in registers.  The min term sum_j m_j S_j (S_j = sum of the
//    scaled x over sub-block j) is one more m16n8k8 MMA with A = the mins
//    (6-bit integers as f16 subnormals) and B = S as fp16 hi + lo.  Per row
//    and token: y = (d 2^24 P - dmin 2^30 Qd) / s.
//
// Which 16 weights form one MMA step is free (the sum over k does not care),
// so the steps follow the byte layout: quad lane q owns bytes 8q..8q+7 of
// each 32-byte quant group, step h of sub-block 2g (low nibbles) or 2g+1
// (high nibbles) uses bytes 8q+4h..8q+4h+3, and the x fragments are built in
// the same order.
//
// Work split.  A cluster of `ks` CTAs owns a block of 16-row tiles; CTA
// rank r of the cluster owns super-blocks [r*S, (r+1)*S) of every row (a
// K-slice), one compute warp per super-block, so each warp keeps its x
// fragments in registers for the whole kernel.  A producer warp streams
// [16 rows x S super-blocks] tiles with one 3-D TMA copy each into a ring of
// stages; the compute warps add their partial 16 x 8 results into a
// shared-memory accumulator with shared atomics.  With ks > 1 the K-slices
// of a cluster are summed at the end through distributed shared memory, in
// rank order.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstdio>
#include <cstdlib>
#include <map>
#include <tuple>

#include "rq_device.cuh"
#include "rq_internal.h"

namespace rq {
namespace {

__device__ unsigned int g_ft_error;  // bit 0: a pipeline wait timed out

constexpr int kTileRows = 16;
constexpr int kMaxSlice = 15;   // super-blocks per K-slice (compute warps); with
                                // the producer, 16 warps keep 128 registers
constexpr int kMaxKs = 8;       // K-slices per cluster
constexpr int kTok = 8;         // MMA N: tokens (M <= 8, padded with zeros)

// The weights of one launch: `nseg` members that share x, member i owning
// tiles [tile_start[i], tile_start[i+1]) of the launch's 16-row tiles (its
// N_i rows, padded to whole tiles) and writing y_i [M x N_i].
struct FtArgs {
  const float* x;
  int M, K;
  int nseg;
  int tile_start[RQ_MAX_GROUP + 1];
  int seg_n[RQ_MAX_GROUP];
  float* seg_y[RQ_MAX_GROUP];
  int nsb;         // super-blocks per row (K / 256)
  int S;           // super-blocks per K-slice = compute warps per CTA
  int tiles;       // 16-row tiles of all members
  int clusters;
  int stages;
  int max_tiles;   // most tiles any cluster owns (accumulator rows / 16)
  int perm;        // 1: spread a half-warp's four rows over distinct banks
  uint64_t wait_limit_ns;
};

// One 3-D tensor map per member (box: 16 rows x S super-blocks x 144 B).
struct FtMaps {
  CUtensorMap m[RQ_MAX_GROUP];
};

__device__ __forceinline__ int ft_seg(const FtArgs& a, int tile) {
  int i = 0;
  while (i + 1 < a.nseg && tile >= a.tile_start[i + 1]) ++i;
  return i;
}

// Output element (token m, row `row` of the launch's tile rows): its member's
// y and row, or nullptr for a padding row past the member's N.
__device__ __forceinline__ float* ft_out(const FtArgs& a, int m, int row) {
  const int t = row / kTileRows;
  const int sg = ft_seg(a, t);
  const int r = (t - a.tile_start[sg]) * kTileRows + row % kTileRows;
  return r < a.seg_n[sg] ? a.seg_y[sg] + (size_t)m * a.seg_n[sg] + r : nullptr;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// d += A * B for one m16n8k16 step (f16 x f16 -> f32).
__device__ __forceinline__ void mma_step(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);  // .x (low 16 bits) = lo
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Split v into a part with at most 11 significant bits and the rest
// (Veltkamp's splitting with the factor 2^13 + 1; the operations are kept
// apart so no FMA contraction changes them): v = hi + lo exactly, and hi is
// exact in fp16 when |hi| >= 2^-14.  FP32-pipe arithmetic only.
__device__ __forceinline__ void split11(float v, float& hi, float& lo) {
  const float c = __fmul_rn(v, 8193.0f);
  hi = __fsub_rn(c, __fsub_rn(c, v));
  lo = __fsub_rn(v, hi);
}

// Byte b (0 or 1) of a 16-bit pair, as a float, without an int->float
// conversion: the byte goes into the mantissa of 2^23.
__device__ __forceinline__ float byte_f(uint32_t pair, int b) {
  return __uint_as_float(__byte_perm(pair, 0x4B000000u, b ? 0x7441u : 0x7440u)) - 8388608.0f;
}

// 6-bit scales (byte 0: sub-block 2g, byte 1: 2g+1) and mins of group g of a
// Q4_K header (12 bytes of scales and mins packed as in GGML's
// get_scale_min_k4, after the fp16 d and dmin).
__device__ __forceinline__ void q4_scale_min_pair(const uint4& h, int g, uint32_t& scp,
                                                  uint32_t& mp) {
  const int sh = (g & 1) * 16;
  const uint32_t a16 = h.y >> sh, b16 = h.z >> sh, c16 = h.w >> sh;
  if (g < 2) {
    scp = a16 & 0x3F3Fu;
    mp = b16 & 0x3F3Fu;
  } else {
    scp = (c16 & 0x0F0Fu) | ((a16 >> 2) & 0x3030u);
    mp = ((c16 >> 4) & 0x0F0Fu) | ((b16 >> 2) & 0x3030u);
  }
}

// d += A * B for one m16n8k8 step (f16 x f16 -> f32).
__device__ __forceinline__ void mma_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// byte_f with the byte divided by 16 (mantissa of 2^19 instead of 2^23).
__device__ __forceinline__ float byte_f16th(uint32_t pair, int b) {
  return __uint_as_float(__byte_perm(pair, 0x49000000u, b ? 0x7441u : 0x7440u)) - 524288.0f;
}

// 6-bit mins of sub-blocks 2g, 2g+1 (bytes 0, 1) for a group index g known
// only at run time (no divergent branch).
__device__ __forceinline__ uint32_t q4_min_pair(const uint4& h, int g) {
  const int sh = (g & 1) * 16;
  const uint32_t b16 = h.z >> sh, c16 = h.w >> sh;
  const uint32_t lo = b16 & 0x3F3Fu;
  const uint32_t hi = ((c16 >> 4) & 0x0F0Fu) | ((b16 >> 2) & 0x3030u);
  return g < 2 ? lo : hi;
}

// PACK (M <= 4): the MMA's 8 columns are (token, hi) and (token, lo) pairs,
// so one MMA per step covers both halves of the split and each lane holds
// only its column's half of x.  Otherwise (M <= 8) the columns are tokens
// and the hi and lo halves take one MMA each.
template <bool PACK>
__global__ void __launch_bounds__((kMaxSlice + 1) * 32, 1)
q4k_gemv_ft_kernel(const __grid_constant__ FtMaps maps, const __grid_constant__ FtArgs a) {
  extern __shared__ __align__(128) uint8_t smem_ft[];
  const int S = a.S;
  const uint32_t stage_bytes = (uint32_t)(kTileRows * S * kQ4KBytes);
  uint8_t* ring = smem_ft;
  float* acc = reinterpret_cast<float*>(ring + (size_t)a.stages * stage_bytes);
  const int acc_n = a.max_tiles * kTileRows * kTok;
  uint64_t* bars = reinterpret_cast<uint64_t*>(acc + acc_n);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + a.stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int ks = (int)(gridDim.x / a.clusters);
  const int cid = (int)blockIdx.x / ks;
  const int t0 = (int)((int64_t)cid * a.tiles / a.clusters);
  const int t1 = (int)((int64_t)(cid + 1) * a.tiles / a.clusters);
  const int ntiles = t1 - t0;
  const int sb0 = (int)rank * S;

  for (int i = threadIdx.x; i < acc_n; i += blockDim.x) acc[i] = 0.f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, S);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  // The first ring's worth of weight copies goes out before the wait for
  // the previous launch; x and y are touched only after it.
  uint32_t issued = 0, parity_bits = 0;
  const bool producer = warp == S && lane == 0;
  const int first = ntiles < a.stages ? ntiles : a.stages;
  auto load_tile = [&](int it, int s) {
    const int t = t0 + it, sg = ft_seg(a, t);
    tma_load_3d(smem_u32(ring + (size_t)s * stage_bytes), &maps.m[sg], full0 + 8 * s, 0, sb0,
                (t - a.tile_start[sg]) * kTileRows);
  };
  if (producer) {
    for (int it = 0; it < first; ++it) {
      mbar_arrive_expect_tx(full0 + 8 * it, stage_bytes);
      load_tile(it, it);
      issued |= 1u << it;
    }
  }
  pdl_wait();
  pdl_trigger();
  if (warp == S) {
    if (lane == 0) {
      for (int it = first; it < ntiles; ++it) {
        const int s = it % a.stages;
        const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, a.wait_limit_ns, &g_ft_error)) break;
        mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
        load_tile(it, s);
        issued |= 1u << s;
        parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
      }
      // every issued copy has landed before the CTA can exit
      for (int s = 0; s < a.stages; ++s)
        if (issued & (1u << s))
          mbar_wait(full0 + 8 * s, (parity_bits >> s) & 1u, a.wait_limit_ns, &g_ft_error);
    }
  } else {
    // ------------------------------------------------- x fragments (prologue)
    // Lane (n, q): MMA column n = lane / 4, quad lane q.  Column n is token
    // n (or, with PACK, token n / 2 and half n % 2 of its split).
    const int n = lane >> 2, q = lane & 3;
    const int tok = PACK ? (n >> 1) : n;
    const bool lo_half = PACK && (n & 1);
    const int sb = sb0 + warp;
    const bool have = sb < a.nsb && tok < a.M;
    const float* xr = a.x + (size_t)tok * a.K + (size_t)sb * kQK + 8 * q;
    float4 xv[16];  // i = g*4 + hn*2 + h
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (have)
        xv[i] = __ldg(reinterpret_cast<const float4*>(
            xr + 64 * (i >> 2) + 32 * ((i >> 1) & 1) + 4 * (i & 1)));
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(xv[i].x), fabsf(xv[i].y)),
                           fmaxf(fabsf(xv[i].z), fabsf(xv[i].w))));
    }
    // The token's scale for this warp's super-block: s = 2^(14 - E) for
    // max |x| in [2^E, 2^(E+1)), so every scaled value is below 2^15 (NaN is
    // ignored by the max; an all-zero or non-finite maximum keeps s = 1).
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    const uint32_t mb = __float_as_uint(mx);
    int es = 127;
    if (mb != 0u && mb < 0x7F800000u) {
      es = 268 - (int)(mb >> 23);
      es = es > 253 ? 253 : es;
    }
    const float s = __int_as_float(es << 23);
    const float inv = __int_as_float((254 - es) << 23);
    // 1/s of the tokens of this lane's accumulator columns 2q, 2q+1 (with
    // PACK both columns are token q, read from lane 8q)
    const float inv0 = __shfl_sync(0xFFFFFFFFu, inv, 8 * q);
    const float inv1 = __shfl_sync(0xFFFFFFFFu, inv, 8 * q + 4);
    // bx[p][j][h][r]: half p (hi, lo), sub-block j = 2g + hn, step h,
    // register r (0: bytes 0 and 2 of the 4-byte chunk, 1: bytes 1 and 3);
    // with PACK only this lane's half is kept
    constexpr int NP = PACK ? 1 : 2;
    uint32_t bx[NP][8][2][2];
    float ps[8];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int hn = (i >> 1) & 1, h = i & 1, j = 2 * (i >> 2) + hn;
      const float4 v = make_float4(xv[i].x * s, xv[i].y * s, xv[i].z * s, xv[i].w * s);
      float h0, l0, h1, l1, h2, l2, h3, l3;
      split11(v.x, h0, l0);
      split11(v.y, h1, l1);
      split11(v.z, h2, l2);
      split11(v.w, h3, l3);
      if (PACK) {
        bx[0][j][h][0] = lo_half ? half2_bits(l0, l2) : half2_bits(h0, h2);
        bx[0][j][h][1] = lo_half ? half2_bits(l1, l3) : half2_bits(h1, h3);
      } else {
        bx[0][j][h][0] = half2_bits(h0, h2);
        bx[0][j][h][1] = half2_bits(h1, h3);
        bx[NP - 1][j][h][0] = half2_bits(l0, l2);
        bx[NP - 1][j][h][1] = half2_bits(l1, l3);
      }
      const float sum = (v.x + v.y) + (v.z + v.w);
      ps[j] = h ? ps[j] + sum : sum;
    }
    // Min term as m16n8k8 steps: B = (S_2q, S_2q+1) of the column's token,
    // the scaled sub-block sums times 2^-6 (below 2^14), split into fp16
    // hi + lo.  S_j sums the scaled x itself; hi + lo of the main fragments
    // differ from it by at most 2^-22 of each value, far inside the
    // tolerance.
    float S0 = 0.f, S1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float t = ps[j];
      t += __shfl_xor_sync(0xFFFFFFFFu, t, 1);
      t += __shfl_xor_sync(0xFFFFFFFFu, t, 2);
      if (j == 2 * q) S0 = t;
      if (j == 2 * q + 1) S1 = t;
    }
    float sh0, sl0, sh1, sl1;
    split11(S0 * 0.015625f, sh0, sl0);
    split11(S1 * 0.015625f, sh1, sl1);
    uint32_t bq[NP];
    if (PACK) {
      bq[0] = lo_half ? half2_bits(sl0, sl1) : half2_bits(sh0, sh1);
    } else {
      bq[0] = half2_bits(sh0, sh1);
      bq[NP - 1] = half2_bits(sl0, sl1);
    }

    // ------------------------------------------------------------ compute --
    const int rA = a.perm ? (((n & 3) << 1) | (n >> 2)) : n;  // stage row of MMA row n
    const int rB = rA + 8;
    const int rs = S * kQ4KBytes;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % a.stages;
      const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(full0 + 8 * st, ph, a.wait_limit_ns, &g_ft_error)))
        break;
      const uint8_t* pA = ring + (size_t)st * stage_bytes + rA * rs + warp * kQ4KBytes;
      const uint8_t* pB = pA + 8 * rs;
      const uint4 hA = *reinterpret_cast<const uint4*>(pA);
      const uint4 hB = *reinterpret_cast<const uint4*>(pB);
      // P = sum_j sc_j * D_j per accumulator entry (row A column 2q, row A
      // column 2q+1, row B column 2q, row B column 2q+1).  High nibbles enter
      // the MMA as 16 q (one AND, no shift), so their scales carry 1/16.
      float P[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint2 uA = *reinterpret_cast<const uint2*>(pA + 16 + 32 * g + 8 * q);
        const uint2 uB = *reinterpret_cast<const uint2*>(pB + 16 + 32 * g + 8 * q);
        uint32_t scA, scB, unused;
        q4_scale_min_pair(hA, g, scA, unused);
        q4_scale_min_pair(hB, g, scB, unused);
#pragma unroll
        for (int hn = 0; hn < 2; ++hn) {
          const int j = 2 * g + hn;
          const uint32_t mask = hn ? 0x00F000F0u : 0x000F000Fu;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wA = h ? uA.y : uA.x, wB = h ? uB.y : uB.x;
            const uint32_t a0 = wA & mask, a1 = wB & mask;                // bytes 0, 2
            const uint32_t a2 = (wA >> 8) & mask, a3 = (wB >> 8) & mask;  // bytes 1, 3
#pragma unroll
            for (int p = 0; p < NP; ++p)
              mma_step(d, a0, a1, a2, a3, bx[p][j][h][0], bx[p][j][h][1]);
          }
          const float sA = hn ? byte_f16th(scA, 1) : byte_f(scA, 0);
          const float sB = hn ? byte_f16th(scB, 1) : byte_f(scB, 0);
          P[0] = fmaf(sA, d[0], P[0]);
          P[1] = fmaf(sA, d[1], P[1]);
          P[2] = fmaf(sB, d[2], P[2]);
          P[3] = fmaf(sB, d[3], P[3]);
        }
      }
      // Qd = 2^-30 sum_j m_j S_j: A = the mins of sub-blocks 2q, 2q+1 of the
      // two rows as f16 subnormals m * 2^-24
      float Qd[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t qa0 = __byte_perm(q4_min_pair(hA, q), 0u, 0x4140u);
        const uint32_t qa1 = __byte_perm(q4_min_pair(hB, q), 0u, 0x4140u);
#pragma unroll
        for (int p = 0; p < NP; ++p) mma_k8(Qd, qa0, qa1, bq[p]);
      }
      const float2 ddA = half_pair(hA.x), ddB = half_pair(hB.x);  // (d, dmin)
      const float dA = ddA.x * 16777216.0f, dB = ddB.x * 16777216.0f;
      const float mA = ddA.y * 1073741824.0f, mB = ddB.y * 1073741824.0f;
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      float* accA = acc + (it * kTileRows + rA) * kTok;
      float* accB = acc + (it * kTileRows + rB) * kTok;
      if (PACK) {
        // columns 2q and 2q+1 are the hi and lo halves of token q
        atomicAdd(accA + q, fmaf(dA, P[0] + P[1], -mA * (Qd[0] + Qd[1])) * inv0);
        atomicAdd(accB + q, fmaf(dB, P[2] + P[3], -mB * (Qd[2] + Qd[3])) * inv0);
      } else {
        atomicAdd(accA + 2 * q, fmaf(dA, P[0], -mA * Qd[0]) * inv0);
        atomicAdd(accA + 2 * q + 1, fmaf(dA, P[1], -mA * Qd[1]) * inv1);
        atomicAdd(accB + 2 * q, fmaf(dB, P[2], -mB * Qd[2]) * inv0);
        atomicAdd(accB + 2 * q + 1, fmaf(dB, P[3], -mB * Qd[3]) * inv1);
      }
    }
  }
  __syncthreads();

  const int r0 = t0 * kTileRows;
  const int rows = (t1 - t0) * kTileRows;
  if (ks == 1) {
    for (int i = threadIdx.x; i < rows * a.M; i += blockDim.x) {
      const int m = i / rows, row = i % rows;
      float* out = ft_out(a, m, r0 + row);
      if (out != nullptr) *out = acc[row * kTok + m];
    }
    return;
  }
  // sum the K-slices of the cluster in rank order
  cluster_sync();
  const int lo = (int)((int64_t)rank * rows / ks), hi = (int)((int64_t)(rank + 1) * rows / ks);
  const int nr = hi - lo;
  for (int i = threadIdx.x; i < nr * a.M; i += blockDim.x) {
    const int m = i / nr, row = lo + i % nr;
    const float* p = acc + row * kTok + m;
    float v = 0.f;
    for (int r = 0; r < ks; ++r) v += ld_cluster_f32(p, (uint32_t)r);
    float* out = ft_out(a, m, r0 + row);
    if (out != nullptr) *out = v;
  }
  cluster_sync();  // no CTA leaves while a peer may still read its memory
}

// ----------------------------------------------------------- host side --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D view [N rows][nsb super-blocks][144 bytes] of a Q4_K matrix; a box is
// 16 rows x S super-blocks; rows past N read as zero.  Maps are cached per
// (weight, N, K, S).
const CUtensorMap* weight_map(const uint8_t* w, int N, int K, int S) {
  static std::map<std::tuple<const void*, int, int, int>, CUtensorMap> cache;
  const auto key = std::make_tuple(static_cast<const void*>(w), N, K, S);
  auto it = cache.find(key);
  if (it != cache.end()) return &it->second;
  auto fn = encode_fn();
  if (fn == nullptr) return nullptr;
  const int nsb = K / kQK;
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)kQ4KBytes, (cuuint64_t)nsb, (cuuint64_t)N};
  const cuuint64_t strides[2] = {(cuuint64_t)kQ4KBytes, (cuuint64_t)nsb * kQ4KBytes};
  const cuuint32_t box[3] = {(cuuint32_t)kQ4KBytes, (cuuint32_t)S, (cuuint32_t)kTileRows};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(w), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return nullptr;
  if (cache.size() > 4096) cache.clear();
  return &cache.emplace(key, map).first->second;
}

constexpr size_t kSmemLimit = 227 * 1024;

size_t ft_smem(int S, int stages, int max_tiles) {
  return (size_t)stages * kTileRows * S * kQ4KBytes + (size_t)max_tiles * kTileRows * kTok * 4 +
         16 * (size_t)stages;
}

// Clusters of `ks` CTAs (one per SM) that fit on the GPU at once.
int resident_clusters(int ks, int threads, size_t smem) {
  static std::map<std::tuple<int, int, size_t>, int> cache;
  const auto key = std::make_tuple(ks, threads, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ks * (device_sm_count() / ks));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, q4k_gemv_ft_kernel<false>, &cfg) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 0;
  }
  cache.emplace(key, n);
  return n;
}

}  // namespace

rq_status launch_q4k_gemv_mma_group(int count, const uint8_t* const* ws, const int* Ns,
                                    float* const* ys, const float* x, int M, int K,
                                    cudaStream_t st) {
  if (M < 2 || M > kTok || count < 1 || count > RQ_MAX_GROUP) return RQ_ERR_SHAPE;
  const int nsb = K / kQK;
  const int sms = device_sm_count();
  int tile_start[RQ_MAX_GROUP + 1];
  tile_start[0] = 0;
  for (int i = 0; i < count; ++i) tile_start[i + 1] = tile_start[i] + (Ns[i] + kTileRows - 1) / kTileRows;
  const int tiles = tile_start[count];
  const int ks_min = (nsb + kMaxSlice - 1) / kMaxSlice;
  if (ks_min > kMaxKs) return RQ_ERR_SHAPE;
  int ks = ks_min;
  // few row tiles: split K further so that more SMs stream weights
  if (tiles * ks < sms) {
    int want = sms / tiles;
    want = want > kMaxKs ? kMaxKs : want;
    want = want > nsb ? nsb : want;
    if (want > ks) ks = want;
  }
  const char* env = std::getenv("RQ_GEMV_MMA_KS");
  if (env != nullptr) {
    const int v = std::atoi(env);
    if (v >= ks_min && v <= kMaxKs && v <= nsb) ks = v;  // tuning runs
  }
  const int S = (nsb + ks - 1) / ks;
  ks = (nsb + S - 1) / S;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(q4k_gemv_ft_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemLimit) != cudaSuccess ||
        cudaFuncSetAttribute(q4k_gemv_ft_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemLimit) != cudaSuccess)
      return RQ_ERR_CUDA;
    attr_set = true;
  }
  const int threads = (S + 1) * 32;
  const size_t stage_bytes = (size_t)kTileRows * S * kQ4KBytes;

  // stages and clusters: as many stages as fit next to the accumulator of
  // the resulting tile share
  int stages = 8;
  int clusters = 0, max_tiles = 0;
  for (; stages >= 2; --stages) {
    const size_t probe = ft_smem(S, stages, 1);
    if (probe > kSmemLimit) continue;
    clusters = resident_clusters(ks, threads, probe);
    if (clusters < 1) continue;
    clusters = clusters < tiles ? clusters : tiles;
    max_tiles = (tiles + clusters - 1) / clusters;
    if (ft_smem(S, stages, max_tiles) <= kSmemLimit) break;
  }
  if (stages < 2 || clusters < 1) return RQ_ERR_SHAPE;
  const size_t smem = ft_smem(S, stages, max_tiles);
  FtMaps maps;
  for (int i = 0; i < RQ_MAX_GROUP; ++i) {
    const int j = i < count ? i : 0;
    const CUtensorMap* map = weight_map(ws[j], Ns[j], K, S);
    if (map == nullptr) return RQ_ERR_CUDA;
    maps.m[i] = *map;
  }

  FtArgs a;
  a.x = x;
  a.M = M;
  a.K = K;
  a.nseg = count;
  for (int i = 0; i <= RQ_MAX_GROUP; ++i) a.tile_start[i] = tile_start[i <= count ? i : count];
  for (int i = 0; i < RQ_MAX_GROUP; ++i) {
    a.seg_n[i] = i < count ? Ns[i] : 0;
    a.seg_y[i] = i < count ? ys[i] : nullptr;
  }
  a.nsb = nsb;
  a.S = S;
  a.tiles = tiles;
  a.clusters = clusters;
  a.stages = stages;
  a.max_tiles = max_tiles;
  const int sigma = (4 * S) & 31;  // row stride in words, mod 32 banks
  a.perm = (sigma == 4 || sigma == 12 || sigma == 20 || sigma == 28) ? 1 : 0;
  a.wait_limit_ns = kWaitLimitNs;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(clusters * ks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  if (std::getenv("RQ_GEMV_LOG") != nullptr)
    std::fprintf(stderr, "rq_gemv: q4k_ft M=%d N=%d K=%d grid=%d\n", M, tiles * kTileRows, K,
                 clusters * ks);
  if (M <= 4) return cuda_status(cudaLaunchKernelEx(&cfg, q4k_gemv_ft_kernel<true>, maps, a));
  return cuda_status(cudaLaunchKernelEx(&cfg, q4k_gemv_ft_kernel<false>, maps, a));
}

rq_status launch_q4k_gemv_mma(const uint8_t* w, const float* x, float* y, int M, int N, int K,
                              cudaStream_t st) {
  return launch_q4k_gemv_mma_group(1, &w, &N, &y, x, M, K, st);
}

rq_status read_and_clear_gemv_mma_error() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_ft_error, sizeof(v)) != cudaSuccess) return RQ_ERR_CUDA;
  if (v == 0) return RQ_OK;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_ft_error, &zero, sizeof(zero)) != cudaSuccess) return RQ_ERR_CUDA;
  return RQ_ERR_TIMEOUT;
}

}  // namespace rq
