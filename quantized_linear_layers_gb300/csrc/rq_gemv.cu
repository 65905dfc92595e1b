// rq_gemv.cu -- decode GEMV on GGUF Q4_K / Q6_K weights, M = 1..8 tokens.
//
// realizar 0.8.4, q6k_gemv_indexed.rs (q4k_gemv_into and its variants,
// q6k_gemv_indexed_async) and cublas_prefill/mod.rs (cublas_gemm_threshold:
// the batched GEMV reads Q4_K directly at 0.5625 B/weight).  The kernel
// bodies are not on the pages; this design is written for sm_103a:
//
//  * Persistent grid (SM count x resident CTAs).  Each warp owns groups of R
//    consecutive weight rows; within a group, lane l handles the 64-weight
//    quant groups u = l, l+32, ... of every row (one 16-byte header load and
//    two 16-byte quant loads per row, all coalesced across the warp).  The
//    next item's loads are issued before the current one is decoded, so two
//    items of weight bytes are in flight per warp.
//  * x is read through L1 (16-byte loads) once per item and reused by all R
//    rows.
//  * Every weight is decoded on its own: Q4_K w = fl(q * (d sc) - dmin m)
//    (one FMA, a single rounding of the exact value), Q6_K w = (q - 32) *
//    (d scale) (exact in fp32).  Each lane sums the 64 products of an item in
//    fp32 and adds that partial to its total, so every rounding is relative
//    to sum_k |x_k w_k| (well inside the 1e-4 bound); an output that comes
//    out non-finite (overflow, non-finite x) is recomputed exactly in fp64.
//  * fp32 accumulation, one warp-shuffle reduction per row.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <map>
#include <utility>

#include "rq_device.cuh"
#include "rq_gemv_exact.cuh"
#include "rq_internal.h"

namespace rq {

// Counts outputs recomputed on the exact path (diagnostics and tests).
__device__ unsigned long long g_gemv_exact_outputs;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Byte j of v (a value below 2^8) as a float, without a conversion: the
// byte goes into the mantissa of 2^23.
__device__ __forceinline__ float byte_j_f(uint32_t v, int j) {
  return __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440u | (uint32_t)j)) - 8388608.0f;
}

// ------------------------------------------------------------------ Q4_K --

struct Q4Item {
  uint4 h;   // d, dmin (fp16 pair) and the 12 packed scale/min bytes
  uint4 a;   // quant bytes 0..15 of the 64-weight group
  uint4 b;   // quant bytes 16..31
};

template <int R>
__device__ __forceinline__ void q4_load(Q4Item (&it)[R], const uint8_t* __restrict__ W,
                                        size_t rowbytes, int row0, int N, int u,
                                        bool valid) {
  const int sb = u >> 2, g = u & 3;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (valid && row0 + r < N) {
      const uint8_t* p = W + (size_t)(row0 + r) * rowbytes + (size_t)sb * kQ4KBytes;
      it[r].h = ldg_nc_v4(p);
      it[r].a = ldg_nc_v4(p + 16 + 32 * g);
      it[r].b = ldg_nc_v4(p + 32 + 32 * g);
    } else {
      it[r].h = make_uint4(0, 0, 0, 0);
      it[r].a = it[r].h;
      it[r].b = it[r].h;
    }
  }
}

__device__ __forceinline__ uint32_t q4_word(const Q4Item& it, int w) {
  switch (w) {
    case 0: return it.a.x; case 1: return it.a.y;
    case 2: return it.a.z; case 3: return it.a.w;
    case 4: return it.b.x; case 5: return it.b.y;
    case 6: return it.b.z; default: return it.b.w;
  }
}

// Accumulate the contribution of 64-weight group u of R rows into acc.
template <int M, int R>
__device__ __forceinline__ void q4_compute(const Q4Item (&it)[R], int u,
                                           const float* __restrict__ x, int K,
                                           float (&acc)[R][M]) {
  const int sb = u >> 2, g = u & 3;
  const int k0 = sb * kQK + 64 * g;
  const int sh = (g & 1) * 16;     // byte pair of sub-blocks 2g, 2g+1
  const bool upper = g >= 2;       // sub-blocks 4..7 use the split packing
  float Alo[R], Ahi[R], Blo[R], Bhi[R];  // d sc and dmin m of sub-blocks 2g, 2g+1
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t A = it[r].h.y, B = it[r].h.z, C = it[r].h.w;
    const uint32_t a16 = A >> sh, b16 = B >> sh, c16 = C >> sh;
    // 6-bit scales (scp) and mins (mp) of sub-blocks 2g (low byte), 2g+1
    const uint32_t scp = upper ? ((c16 & 0x0F0Fu) | ((a16 >> 2) & 0x3030u)) : (a16 & 0x3F3Fu);
    const uint32_t mp = upper ? (((c16 >> 4) & 0x0F0Fu) | ((b16 >> 2) & 0x3030u)) : (b16 & 0x3F3Fu);
    const float2 dd = half_pair(it[r].h.x);  // .x = d, .y = dmin
    Alo[r] = dd.x * byte_j_f(scp, 0);
    Ahi[r] = dd.x * byte_j_f(scp, 1);
    Blo[r] = dd.y * byte_j_f(mp, 0);
    Bhi[r] = dd.y * byte_j_f(mp, 1);
  }
  float T[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) T[r][m] = 0.f;

#pragma unroll
  for (int w = 0; w < 8; ++w) {
    float4 xl[M], xh[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float* xr = x + (size_t)m * K + k0 + 4 * w;
      xl[m] = __ldg(reinterpret_cast<const float4*>(xr));
      xh[m] = __ldg(reinterpret_cast<const float4*>(xr + 32));
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t v = q4_word(it[r], w);
      const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;
      float wl[4], wh[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wl[j] = fmaf(byte_j_f(lo, j), Alo[r], -Blo[r]);
        wh[j] = fmaf(byte_j_f(hi, j), Ahi[r], -Bhi[r]);
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float t = T[r][m];
        t = fmaf(xl[m].x, wl[0], t); t = fmaf(xl[m].y, wl[1], t);
        t = fmaf(xl[m].z, wl[2], t); t = fmaf(xl[m].w, wl[3], t);
        t = fmaf(xh[m].x, wh[0], t); t = fmaf(xh[m].y, wh[1], t);
        t = fmaf(xh[m].z, wh[2], t); t = fmaf(xh[m].w, wh[3], t);
        T[r][m] = t;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] += T[r][m];
}

template <int M, int R>
__global__ void __launch_bounds__(kThreads)
q4k_gemv_kernel(const uint8_t* __restrict__ W, const float* __restrict__ x,
                float* __restrict__ y, int N, int K) {
  const int nsb = K >> 8, U = nsb * 4;
  const size_t rowbytes = (size_t)nsb * kQ4KBytes;
  const int lane = threadIdx.x & 31;
  const int gwarp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const int ngroups = (N + R - 1) / R;
  const int iters = (U + 31) >> 5;

  int rg = gwarp, it = 0;
  const bool active = rg < ngroups;
  Q4Item cur[R];
  if (active) q4_load<R>(cur, W, rowbytes, rg * R, N, lane, lane < U);
  pdl_wait();  // x and y only after the previous launch has completed
  pdl_trigger();
  if (!active) return;

  float acc[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

  while (true) {
    int nrg = rg, nit = it + 1;
    if (nit == iters) { nit = 0; nrg += nwarps; }
    const bool has_next = nrg < ngroups;
    Q4Item nxt[R];
    if (has_next) {
      const int nu = nit * 32 + lane;
      q4_load<R>(nxt, W, rowbytes, nrg * R, N, nu, nu < U);
    }
    const int u = it * 32 + lane;
    if (u < U) q4_compute<M, R>(cur, u, x, K, acc);
    if (nit == 0) {  // row group rg complete
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = warp_sum(acc[r][m]);  // the same in every lane
          acc[r][m] = 0.f;
          const int row = rg * R + r;
          if (row < N) {
            if (!isfinite(v)) {
              v = (float)q4k_row_exact(W + (size_t)row * rowbytes, x + (size_t)m * K, K, lane);
              if (lane == 0) atomicAdd(&g_gemv_exact_outputs, 1ull);
            }
            if (lane == 0) y[(size_t)m * N + row] = v;
          }
        }
    }
    if (!has_next) break;
#pragma unroll
    for (int r = 0; r < R; ++r) cur[r] = nxt[r];
    rg = nrg;
    it = nit;
  }
}

// ------------------------------------------------------------------ Q6_K --
//
// Unit = (super-block sb, half h, l-quad lq): the 32 weights
// 128h + 32i + 8lq + j (i = 0..3, j = 0..7), built from 8 bytes of ql at
// 64h + 8lq, 8 bytes of ql at 64h + 32 + 8lq and 8 bytes of qh at 32h + 8lq,
// with scales sc[8h + lq/2 + 2i].  Super-blocks are 210 bytes, so fields are
// only 2-byte aligned; each 8-byte quant field is read as three aligned 32-bit
// words and funnel-shifted (the third word ends at most at byte 196 of the
// block, so it never leaves the block); the scales are read as 16-bit pairs.

struct Q6Item {
  uint32_t qa[2], qb[2], qh[2];  // ql(64h+8lq..), ql(64h+32+8lq..), qh(32h+8lq..)
  uint32_t sc[2];                // scales 8h .. 8h+7
  uint32_t d;                    // fp16 d in the low half
};

__device__ __forceinline__ void ld8_unaligned(const uint8_t* p, uint32_t (&out)[2]) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint8_t* base = reinterpret_cast<const uint8_t*>(a & ~uintptr_t(3));
  const uint32_t shift = (uint32_t)(a & 3) * 8;  // 0 or 16
  const uint32_t w0 = ldg_nc_u32(base), w1 = ldg_nc_u32(base + 4), w2 = ldg_nc_u32(base + 8);
  out[0] = __funnelshift_r(w0, w1, shift);
  out[1] = __funnelshift_r(w1, w2, shift);
}

template <int R>
__device__ __forceinline__ void q6_load(Q6Item (&it)[R], const uint8_t* __restrict__ W,
                                        size_t rowbytes, int row0, int N, int u,
                                        bool valid) {
  const int sb = u >> 3, h = (u >> 2) & 1, lq = u & 3;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (valid && row0 + r < N) {
      const uint8_t* p = W + (size_t)(row0 + r) * rowbytes + (size_t)sb * kQ6KBytes;
      ld8_unaligned(p + 64 * h + 8 * lq, it[r].qa);
      ld8_unaligned(p + 64 * h + 32 + 8 * lq, it[r].qb);
      ld8_unaligned(p + 128 + 32 * h + 8 * lq, it[r].qh);
      const uint8_t* ps = p + 192 + 8 * h;  // 8 scale bytes, 2-byte aligned
      it[r].sc[0] = ldg_nc_u16(ps) | (ldg_nc_u16(ps + 2) << 16);
      it[r].sc[1] = ldg_nc_u16(ps + 4) | (ldg_nc_u16(ps + 6) << 16);
      it[r].d = ldg_nc_u16(p + 208);
    } else {
      it[r].qa[0] = it[r].qa[1] = it[r].qb[0] = it[r].qb[1] = 0;
      it[r].qh[0] = it[r].qh[1] = it[r].sc[0] = it[r].sc[1] = 0;
      it[r].d = 0;
    }
  }
}

__device__ __forceinline__ float sbyte(uint32_t w2[2], int i) {
  const uint32_t word = i < 4 ? w2[0] : w2[1];
  return (float)(int)(int8_t)((word >> (8 * (i & 3))) & 0xFFu);
}

template <int M, int R>
__device__ __forceinline__ void q6_compute(Q6Item (&it)[R], int u,
                                           const float* __restrict__ x, int K,
                                           float (&acc)[R][M]) {
  const int sb = u >> 3, h = (u >> 2) & 1, lq = u & 3;
  const int kbase = sb * kQK + 128 * h + 8 * lq;  // + 32 i + j
  float T[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) T[r][m] = 0.f;
  float dsc[R][4];  // d * scale of quarter i (exact)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float d = __half2float(__ushort_as_half((unsigned short)(it[r].d & 0xFFFFu)));
#pragma unroll
    for (int i = 0; i < 4; ++i) dsc[r][i] = d * sbyte(it[r].sc, lq / 2 + 2 * i);
  }

#pragma unroll
  for (int half = 0; half < 2; ++half) {      // bytes j = 4*half .. 4*half+3
#pragma unroll
    for (int i = 0; i < 4; ++i) {             // quarter i: weights 32i + j
      float4 xv[M];
#pragma unroll
      for (int m = 0; m < M; ++m)
        xv[m] = __ldg(reinterpret_cast<const float4*>(x + (size_t)m * K + kbase + 32 * i + 4 * half));
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t la = it[r].qa[half], lb = it[r].qb[half], hb = it[r].qh[half];
        uint32_t q;
        if (i == 0) q = (la & 0x0F0F0F0Fu) | ((hb << 4) & 0x30303030u);
        else if (i == 1) q = (lb & 0x0F0F0F0Fu) | ((hb << 2) & 0x30303030u);
        else if (i == 2) q = ((la >> 4) & 0x0F0F0F0Fu) | (hb & 0x30303030u);
        else q = ((lb >> 4) & 0x0F0F0F0Fu) | ((hb >> 2) & 0x30303030u);
        // w = (q - 32) * d * scale, exact in fp32
        float w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = (byte_j_f(q, j) - 32.0f) * dsc[r][i];
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float t = T[r][m];
          t = fmaf(xv[m].x, w[0], t); t = fmaf(xv[m].y, w[1], t);
          t = fmaf(xv[m].z, w[2], t); t = fmaf(xv[m].w, w[3], t);
          T[r][m] = t;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] += T[r][m];
}

template <int M, int R>
__global__ void __launch_bounds__(kThreads)
q6k_gemv_kernel(const uint8_t* __restrict__ W, const float* __restrict__ x,
                float* __restrict__ y, int N, int K) {
  const int nsb = K >> 8, U = nsb * 8;
  const size_t rowbytes = (size_t)nsb * kQ6KBytes;
  const int lane = threadIdx.x & 31;
  const int gwarp = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const int ngroups = (N + R - 1) / R;
  const int iters = (U + 31) >> 5;

  int rg = gwarp, it = 0;
  const bool active = rg < ngroups;
  Q6Item cur[R];
  if (active) q6_load<R>(cur, W, rowbytes, rg * R, N, lane, lane < U);
  pdl_wait();  // x and y only after the previous launch has completed
  pdl_trigger();
  if (!active) return;

  float acc[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

  while (true) {
    int nrg = rg, nit = it + 1;
    if (nit == iters) { nit = 0; nrg += nwarps; }
    const bool has_next = nrg < ngroups;
    Q6Item nxt[R];
    if (has_next) {
      const int nu = nit * 32 + lane;
      q6_load<R>(nxt, W, rowbytes, nrg * R, N, nu, nu < U);
    }
    const int u = it * 32 + lane;
    if (u < U) q6_compute<M, R>(cur, u, x, K, acc);
    if (nit == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
          float v = warp_sum(acc[r][m]);  // the same in every lane
          acc[r][m] = 0.f;
          const int row = rg * R + r;
          if (row < N) {
            if (!isfinite(v)) {
              v = (float)q6k_row_exact(W + (size_t)row * rowbytes, x + (size_t)m * K, K, lane);
              if (lane == 0) atomicAdd(&g_gemv_exact_outputs, 1ull);
            }
            if (lane == 0) y[(size_t)m * N + row] = v;
          }
        }
    }
    if (!has_next) break;
#pragma unroll
    for (int r = 0; r < R; ++r) cur[r] = nxt[r];
    rg = nrg;
    it = nit;
  }
}

// ------------------------------------------------- Q4_K, one token ---------
//
// M = 1 is the decode hot path.  Each lane owns one 64-weight quant group u
// of every row and keeps x[64u .. 64u+63] in registers for the whole kernel,
// so x costs no memory traffic per weight.  At the start the lane splits each
// 32-value half of its x into three int8 planes, x = s (x1 + x2/128 +
// x3/16384) to within max|x| / (127 * 32768); the 4-bit quants, masked to one
// nibble per byte, then enter 4-way byte dot products (dp4a) against the
// planes, three per four weights, and the sub-block sums are put back
// together in fp32.  This is not an activation quantization: the planes
// reproduce x to ~2^-22 of its sub-block maximum, far inside the GEMV
// tolerance.
// A team of ceil(K/64/32) warps covers K; a CTA runs `teams` teams and one
// producer warp.  Each CTA owns a contiguous block of rows (the row blocks of
// all CTAs differ by at most one row); the producer streams the block into a
// shared-memory ring, `rows_per_stage` consecutive rows (one contiguous
// cp.async.bulk copy) per stage, and the teams take the stage's rows in turn.
// Per row a lane reads its 48 bytes (header + 32 quant bytes) from shared
// memory -- conflict-free 16-byte loads -- decodes and accumulates; a warp
// shuffle reduction and one shared atomic per warp and row complete the dot
// product.  Every mbarrier wait is bounded.

__device__ unsigned int g_gemv_error;  // bit 0: a pipeline wait timed out

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

struct M1Args {
  // One-token Q4_K with rows split between two CTAs of a single weight: a
  // 3-D view [N rows][K/256 super-blocks][144 B] of it whose box is one
  // stage (rows_per_stage rows x this CTA's super-blocks); tma = 1 loads
  // each stage with one copy of it.
  CUtensorMap map;
  int tma;
  uint32_t stage_stride;  // bytes between stages in the ring (128-byte multiple)
  const uint8_t* W;
  const float* x;
  float* y;
  int N, K;
  int team_warps;      // warps per team: ceil(K / 64 / 32)
  int teams;           // teams per CTA
  int rows_per_stage;  // 2 * teams
  int stages;
  uint32_t ring_bytes;  // stages * rows_per_stage * rowbytes
  uint64_t wait_limit_ns;
  int row_align;        // Q6_K: rows per 16-byte-aligned group of rows
  int M;                // tokens (the multi-token Q6_K kernel)
  int max_rows;         // most rows any CTA owns (sizes the row accumulators)
  int evict_first;      // weight copies ask L2 to evict their lines first
  // One-token Q4_K: 2 = clusters of two CTAs share a block of rows, CTA
  // rank h taking super-blocks [h*nsb/2, (h+1)*nsb/2) of each row (rank 0
  // adds rank 1's partial sums and writes y); 1 = one CTA per row block.
  int ksplit;
  // One-token Q4_K: the rows are the concatenation of nseg weights that
  // share x (rows [seg_start[i], seg_start[i+1]) are rows of seg_w[i] and
  // go to seg_y[i]); a single weight is one segment.
  int nseg;
  int seg_start[RQ_MAX_GROUP + 1];
  const uint8_t* seg_w[RQ_MAX_GROUP];
  float* seg_y[RQ_MAX_GROUP];
};

__device__ __forceinline__ int m1_seg(const M1Args& a, int row) {
  int i = 0;
  while (i + 1 < a.nseg && row >= a.seg_start[i + 1]) ++i;
  return i;
}

__device__ __forceinline__ uint32_t m1_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void m1_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Store v into the shared memory of CTA `rank` of the cluster, at the offset
// of `local` in this CTA (a posted store: no round trip).
__device__ __forceinline__ void m1_st_peer(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Exact int -> float for |v| < 2^22 on the FP32 pipe (no conversion
// instruction): v is added into the mantissa of 1.5 * 2^23.
__device__ __forceinline__ float i2f_small(int v) {
  return __int_as_float(v + 0x4B400000) - 12582912.0f;
}

// Byte b (0 or 1) of a 16-bit pair as a float (the byte goes into the
// mantissa of 2^23).
__device__ __forceinline__ float byte_to_float(uint32_t pair, int b) {
  return __uint_as_float(__byte_perm(pair, 0x4B000000u, b ? 0x7441u : 0x7440u)) - 8388608.0f;
}

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}


// x of one 32-weight sub-block as three int8 planes: with s = max|x| / 127,
// x = s * (x1 + x2 / 128 + x3 / 16384) + e, |e| <= max|x| / (127 * 32768).
// t = x / s is rounded once (fp32 multiply); x1 = rint(t) and the residuals
// t - x1 (|.| <= 1/2) and their x128 scalings are exact, so the only errors
// are that rounding and the final residual.  Each plane holds values in
// [-127, 127] resp. [-64, 64] packed four per register (byte j = element j).
struct XSplit {
  int p1[8], p2[8], p3[8];  // planes, 4 int8 per register
  float scale;              // s
  float sum;                // sum of the 32 x values (fp32)
  float ea, eb;             // error-bound constants of the sub-block (q4k_cert)
};

// sum_l x_l * q_l for the 32 quants of one nibble plane (byte j of word w =
// quant 4w + j), from the three integer plane products.
struct Dot3 {
  int a1, a2, a3;
};

__device__ __forceinline__ float dot3_value(const Dot3& d, float scale) {
  const float v = fmaf(i2f_small(d.a3), 1.0f / 16384.0f,
                       fmaf(i2f_small(d.a2), 1.0f / 128.0f, i2f_small(d.a1)));
  return v * scale;
}

// The same for the one-token Q4_K kernel, with the plane products combined
// in 32-bit integers first and rounded to fp32 once (relative error 2^-24):
// 2^14 (x1 + x2/2^7 + x3/2^14) for the low nibbles (exact: |a1| <= 32*127*15,
// so the sum stays below 2^30); the high nibbles enter in place as 16 q, so
// every product is a multiple of 16 and 2^14 (x1 + ...) / 16 = a1*2^10 +
// a2*2^3 + a3/2^4 is exact too.  Both are 2^14 times the plane sum; the
// 2^-14 rides in the row coefficients (q4_coeffs).
__device__ __forceinline__ float dot3_lo_int(const Dot3& d, float scale) {
  return __int2float_rn(d.a1 * 16384 + d.a2 * 128 + d.a3) * scale;
}
__device__ __forceinline__ float dot3_hi_int(const Dot3& d, float scale) {
  return __int2float_rn(d.a1 * 1024 + d.a2 * 8 + (d.a3 >> 4)) * scale;
}

// Group coefficients from a header for sub-blocks 2g, 2g+1, with the 2^-14
// of dot3_lo_int / dot3_hi_int: (d sc_lo 2^-14, d sc_hi 2^-14, dmin m_lo,
// dmin m_hi); no underflow (d >= 2^-24 and sc >= 1 when it is non-zero).
// The 6-bit scales and mins of all four byte positions are assembled at
// once (byte k of scw is the scale of sub-block k, k + 4 for the upper
// lanes; mw likewise for the mins), and the lane's two are moved into the
// mantissa of 2^23 by a byte permute with the selectors sel0 / sel1
// (0x7440 | byte index of sub-block 2g resp. 2g + 1 within its word).
__device__ __forceinline__ float4 q4_coeffs(const uint4& h, uint32_t sel0, uint32_t sel1,
                                            bool upper) {
  const uint32_t scw = upper ? ((h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u))
                             : (h.y & 0x3F3F3F3Fu);
  const uint32_t mw = upper ? (((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u))
                            : (h.z & 0x3F3F3F3Fu);
  const float2 dd = half_pair(h.x);
  const float d14 = dd.x * (1.0f / 16384.0f);
  const float s0 = __uint_as_float(__byte_perm(scw, 0x4B000000u, sel0)) - 8388608.0f;
  const float s1 = __uint_as_float(__byte_perm(scw, 0x4B000000u, sel1)) - 8388608.0f;
  const float m0 = __uint_as_float(__byte_perm(mw, 0x4B000000u, sel0)) - 8388608.0f;
  const float m1 = __uint_as_float(__byte_perm(mw, 0x4B000000u, sel1)) - 8388608.0f;
  return make_float4(d14 * s0, d14 * s1, dd.y * m0, dd.y * m1);
}

// Error bound of one lane's 64-weight dot product (q4k_cert).  For
// sub-block j of the lane (32 values v, plane scale s = max|v|/127, sum of
// the third-plane residuals rs = sum |t - planes| * 16384 <= 16, sa =
// sum |v|) the computed contribution differs from the exact
// sum_k v_k (d sc_j q_k - dmin m_j) by at most
//   d sc_j * A_j + dmin m_j * B_j,
//   A_j = 15 s rs / 16384      (the planes' residuals, q <= 15)
//       + 135 u sa             (relative rounding of s*t against v (3u), of
//                               the plane sum's conversion and scaling (2u)
//                               and of the four-step FMA chain (4u), each
//                               against at most 15 sa),
//   B_j = 13 u sa              (the fp32 sum of v (9u) and the chain (4u)),
// u = 2^-24; the constants below add a margin (150 u, 16 u, factor 1 + 2^-7).
// The lane contributes D = sum_j (d sc_j A_j + dmin m_j B_j) - tau |p|.
__device__ __forceinline__ void q4k_cert_consts(float s, float rs, float sa, float mx,
                                                float& ea, float& eb) {
  constexpr float kU = 0x1p-24f, kMargin = 1.0f + 0x1p-7f;
  ea = fmaf(15.0f * s, rs * (1.0f / 16384.0f), 150.0f * kU * sa) * kMargin;
  eb = 16.0f * kU * sa * kMargin;
  // planes not valid (tiny maximum) or x not finite (sa is then Inf or NaN):
  // exact path
  if ((mx > 0.0f && mx < kCertTinyMax) || !(sa < INFINITY)) ea = eb = INFINITY;
}

// Two rows' 64-weight dot products (integer path), interleaved, with their
// certificate terms: returns (p0, p1, D0, D1).
__device__ __forceinline__ float4 q4_group_dot2i(const uint8_t* r0, const uint8_t* r1,
                                                 int off_h, int off_a, uint32_t sel0,
                                                 uint32_t sel1, bool upper,
                                                 const XSplit& xl, const XSplit& xh) {
  const uint4 h0 = lds128(r0 + off_h), h1 = lds128(r1 + off_h);
  const uint4 a0 = lds128(r0 + off_a), a1 = lds128(r1 + off_a);
  const uint4 b0 = lds128(r0 + off_a + 16), b1 = lds128(r1 + off_a + 16);
  const uint32_t q0[8] = {a0.x, a0.y, a0.z, a0.w, b0.x, b0.y, b0.z, b0.w};
  const uint32_t q1[8] = {a1.x, a1.y, a1.z, a1.w, b1.x, b1.y, b1.z, b1.w};
  Dot3 l0 = {0, 0, 0}, g0 = {0, 0, 0}, l1 = {0, 0, 0}, g1 = {0, 0, 0};
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    // high nibbles stay in place: unsigned bytes 16 q against signed x
    const int lo0 = (int)(q0[w] & 0x0F0F0F0Fu), lo1 = (int)(q1[w] & 0x0F0F0F0Fu);
    const uint32_t hi0 = q0[w] & 0xF0F0F0F0u, hi1 = q1[w] & 0xF0F0F0F0u;
    l0.a1 = __dp4a(lo0, xl.p1[w], l0.a1);
    l1.a1 = __dp4a(lo1, xl.p1[w], l1.a1);
    l0.a2 = __dp4a(lo0, xl.p2[w], l0.a2);
    l1.a2 = __dp4a(lo1, xl.p2[w], l1.a2);
    l0.a3 = __dp4a(lo0, xl.p3[w], l0.a3);
    l1.a3 = __dp4a(lo1, xl.p3[w], l1.a3);
    g0.a1 = dp4a_us(hi0, xh.p1[w], g0.a1);
    g1.a1 = dp4a_us(hi1, xh.p1[w], g1.a1);
    g0.a2 = dp4a_us(hi0, xh.p2[w], g0.a2);
    g1.a2 = dp4a_us(hi1, xh.p2[w], g1.a2);
    g0.a3 = dp4a_us(hi0, xh.p3[w], g0.a3);
    g1.a3 = dp4a_us(hi1, xh.p3[w], g1.a3);
  }
  const float4 c0 = q4_coeffs(h0, sel0, sel1, upper), c1 = q4_coeffs(h1, sel0, sel1, upper);
  const float dl0 = dot3_lo_int(l0, xl.scale), dh0 = dot3_hi_int(g0, xh.scale);
  const float dl1 = dot3_lo_int(l1, xl.scale), dh1 = dot3_hi_int(g1, xh.scale);
  float p0 = c0.x * dl0;
  p0 = fmaf(c0.y, dh0, p0);
  p0 = fmaf(-c0.z, xl.sum, p0);
  p0 = fmaf(-c0.w, xh.sum, p0);
  float p1 = c1.x * dl1;
  p1 = fmaf(c1.y, dh1, p1);
  p1 = fmaf(-c1.z, xl.sum, p1);
  p1 = fmaf(-c1.w, xh.sum, p1);
  // ea carries the 2^14 of the coefficients' d sc 2^-14
  float e0 = c0.x * xl.ea;
  e0 = fmaf(c0.y, xh.ea, e0);
  e0 = fmaf(c0.z, xl.eb, e0);
  e0 = fmaf(c0.w, xh.eb, e0);
  float e1 = c1.x * xl.ea;
  e1 = fmaf(c1.y, xh.ea, e1);
  e1 = fmaf(c1.z, xl.eb, e1);
  e1 = fmaf(c1.w, xh.eb, e1);
  return make_float4(p0, p1, fmaf(-kCertTau, fabsf(p0), e0), fmaf(-kCertTau, fabsf(p1), e1));
}

// Round to the nearest integer with the fp32 magic constant 1.5 * 2^23
// (valid for |t| < 2^22): returns the rounded value as a float and as an int.
__device__ __forceinline__ float round_magic(float t, int& i) {
  const float f = t + 12582912.0f;
  i = __float_as_int(f) - 0x4B400000;
  return f - 12582912.0f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Shared-memory layout of the x planes: per 64-weight unit u, 208 bytes:
// plane p (0..2) half h (0 = low nibbles, 1 = high) byte l at p*64 + h*32 + l;
// the 16 padding bytes make 16-byte reads of consecutive units conflict-free.
constexpr int kPlaneStride = 208;

template <int RPT>
__device__ __forceinline__ void q4k_m1_body(const M1Args& a, const int bid, const int nblk) {
  static_assert(RPT == 2 || RPT == 4 || RPT == 8, "rows per team per stage");
  constexpr int SPB = 8 / RPT;  // stages per 8-row reduction batch
  extern __shared__ __align__(128) uint8_t smem_m1[];
  // this CTA's share of each row: super-blocks [h*nsb, (h+1)*nsb) of a
  // row of ksplit*nsb
  const int h = a.ksplit == 2 ? (int)m1_cluster_rank() : 0;
  const int nsb = (a.K >> 8) / a.ksplit, U = nsb * 4, nsub = nsb * 8;
  const int rowbytes = nsb * kQ4KBytes;            // bytes of a row this CTA reads
  const int rowstride = rowbytes * a.ksplit;       // bytes of a whole row
  const float* xh = a.x + (size_t)h * nsb * 256;
  const int rps = a.rows_per_stage;  // teams * RPT
  const uint32_t stage_bytes = (uint32_t)(rps * rowbytes);
  uint8_t* ring = smem_m1;
  uint8_t* planes = ring + a.ring_bytes;                              // U * 208
  const int nsub2 = (nsub + 1) & ~1;  // keeps the barriers 8-byte aligned
  float* xscale = reinterpret_cast<float*>(planes + U * kPlaneStride);  // nsub2
  float* xsum = xscale + nsub2;                                        // nsub2
  float* xa = xsum + nsub2;                                            // nsub2
  float* xb = xa + nsub2;                                              // nsub2
  uint64_t* bars = reinterpret_cast<uint64_t*>(xb + nsub2);
  float* acc = reinterpret_cast<float*>(bars + 2 * a.stages);          // max_rows
  float* dacc = acc + a.max_rows;                                      // max_rows
  int* flist = reinterpret_cast<int*>(dacc + a.max_rows);              // max_rows
  int* nfail = flist + a.max_rows;                                     // 4 words
  float* racc = reinterpret_cast<float*>(nfail + 4);                   // max_rows (rank 0: rank 1's
  float* rdacc = racc + a.max_rows;                                    // max_rows  sums, certificates)
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + a.stages);

  const int compute_warps = a.teams * a.team_warps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cb = bid / a.ksplit, ncb = nblk / a.ksplit;  // row block of the cluster
  const int r0 = (int)((int64_t)cb * a.N / ncb);
  const int r1 = (int)((int64_t)(cb + 1) * a.N / ncb);
  const int rows = r1 - r0;
  const int iters = (rows + rps - 1) / rps;
  // Only the first stage is requested before the previous launch has
  // completed; the rest of the ring after the x planes are built, so that
  // the x loads do not queue behind it (measured on GB300: decode pass
  // 1.122 -> 1.094 ms; the whole ring before the wait 1.122, the rest right
  // after it 1.130)
  const int first = iters < 1 ? iters : 1;

  for (int i = threadIdx.x; i < rows; i += blockDim.x) acc[i] = dacc[i] = 0.f;
  if (threadIdx.x == 0) {
    *nfail = 0;
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, compute_warps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  uint32_t issued = 0, parity_bits = 0;
  bool prod_ok = true;
  auto produce = [&](int it) {
    const int s = it % a.stages;
    const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, a.wait_limit_ns, &g_gemv_error)) {
      prod_ok = false;
      return;
    }
    const int nr = min(rps, rows - it * rps);
    if (a.tma) {
      // the whole box, rows past N read as zero (and count as bytes)
      mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
      if (a.evict_first)
        tma_load_3d_hint(smem_u32(ring + s * a.stage_stride), &a.map, full0 + 8 * s, 0, h * nsb,
                         r0 + it * rps, l2_policy_evict_first());
      else
        tma_load_3d(smem_u32(ring + s * a.stage_stride), &a.map, full0 + 8 * s, 0, h * nsb,
                    r0 + it * rps);
    } else {
      mbar_arrive_expect_tx(full0 + 8 * s, (uint32_t)(nr * rowbytes));
      // one copy per segment the stage's rows fall in (per row when the rows
      // are split between the CTAs of a cluster)
      for (int v = r0 + it * rps, done = 0; done < nr;) {
        const int sg = m1_seg(a, v);
        const int take = a.ksplit == 1 ? min(nr - done, a.seg_start[sg + 1] - v) : 1;
        const uint32_t dst = smem_u32(ring + s * a.stage_stride + (size_t)done * rowbytes);
        const uint8_t* src =
            a.seg_w[sg] + (size_t)(v - a.seg_start[sg]) * rowstride + (size_t)h * rowbytes;
        if (a.evict_first)
          bulk_g2s_hint(dst, src, (uint32_t)(take * rowbytes), full0 + 8 * s,
                        l2_policy_evict_first());
        else
          bulk_g2s(dst, src, (uint32_t)(take * rowbytes), full0 + 8 * s);
        v += take;
        done += take;
      }
    }
    issued |= 1u << s;
    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
  };
  const bool producer = warp == compute_warps && lane == 0;
  // the first stage's weight copy is in flight while the previous launch
  // finishes and x is prepared
  if (producer)
    for (int it = 0; it < first && prod_ok; ++it) produce(it);
  pdl_wait();  // x and y only after the previous launch has completed
  pdl_trigger();

  // ------------------------------------------------ x planes (all compute warps)
  // Four lanes per 32-value sub-block, eight values each: coalesced 16-byte
  // loads, a two-level shuffle for the sub-block's max and sum, and 8-byte
  // stores of each plane's bytes.
  if (warp < compute_warps) {
    const int q = lane & 3;
    // the next iteration's x is loaded before this one is converted, so the
    // loads of consecutive iterations overlap
    const int step32 = compute_warps * 8;
    float4 na = make_float4(0.f, 0.f, 0.f, 0.f), nb = na;
    int sb32 = warp * 8 + (lane >> 2);
    if (sb32 < nsub) {
      const float4* px = reinterpret_cast<const float4*>(xh + 32 * sb32 + 8 * q);
      na = __ldg(px);
      nb = __ldg(px + 1);
    }
    for (; sb32 < nsub; sb32 += step32) {
      const float4 va = na, vb = nb;
      if (sb32 + step32 < nsub) {
        const float4* px = reinterpret_cast<const float4*>(xh + 32 * (sb32 + step32) + 8 * q);
        na = __ldg(px);
        nb = __ldg(px + 1);
      }
      const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      float mx = 0.f, sm = 0.f, sa = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx = fmaxf(mx, fabsf(v[i]));
        sm += v[i];
        sa += fabsf(v[i]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
      sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
      const float inv = mx > 0.f ? 127.0f / mx : 0.0f;
      uint32_t b1[2] = {0, 0}, b2[2] = {0, 0}, b3[2] = {0, 0};
      float rs = 0.f;  // third-plane residuals, in units of s / 16384
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float t = fminf(fmaxf(v[i] * inv, -127.0f), 127.0f);
        int i1, i2, i3;
        const float f1 = round_magic(t, i1);
        const float u2 = (t - f1) * 128.0f;
        const float f2 = round_magic(u2, i2);
        const float u3 = (u2 - f2) * 128.0f;
        rs += fabsf(u3 - round_magic(u3, i3));
        const int sh8 = 8 * (i & 3);
        b1[i >> 2] |= ((uint32_t)i1 & 0xFFu) << sh8;
        b2[i >> 2] |= ((uint32_t)i2 & 0xFFu) << sh8;
        b3[i >> 2] |= ((uint32_t)i3 & 0xFFu) << sh8;
      }
      sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 1);
      sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 2);
      rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
      rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
      uint8_t* pl = planes + (sb32 >> 1) * kPlaneStride + (sb32 & 1) * 32 + 8 * q;
      *reinterpret_cast<uint2*>(pl) = make_uint2(b1[0], b1[1]);
      *reinterpret_cast<uint2*>(pl + 64) = make_uint2(b2[0], b2[1]);
      *reinterpret_cast<uint2*>(pl + 128) = make_uint2(b3[0], b3[1]);
      if (q == 0) {
        const float sc = mx > 0.f ? mx / 127.0f : 1.0f;
        float ea, eb;
        q4k_cert_consts(sc, rs, sa, mx, ea, eb);
        xscale[sb32] = sc;
        xsum[sb32] = sm;
        xa[sb32] = ea * 16384.0f;
        xb[sb32] = eb;
      }
    }
  }
  __syncthreads();

  if (producer) {
    for (int it = first; it < iters && prod_ok; ++it) produce(it);
    // every issued copy has landed before the CTA can exit
    for (int s = 0; s < a.stages; ++s)
      if (issued & (1u << s))
        mbar_wait(full0 + 8 * s, (parity_bits >> s) & 1u, a.wait_limit_ns, &g_gemv_error);
  } else if (warp < compute_warps) {
    // ------------------------------------------------------------ compute --
    const int team = warp / a.team_warps, wt = warp - team * a.team_warps;
    const int u = wt * 32 + lane;
    const bool active = u < U;
    const int sb = u >> 2, g = u & 3;
    // byte permute selectors of the lane's two sub-blocks' scale bytes
    const uint32_t sel0 = 0x7440u | (uint32_t)((g & 1) * 2), sel1 = sel0 + 1u;
    const bool upper = g >= 2;
    XSplit xsl, xsh;
    if (active) {
      const uint8_t* pu = planes + u * kPlaneStride;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        XSplit& xs = h ? xsh : xsl;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 v1 = lds128(pu + 0 + 32 * h + 16 * c);
          const uint4 v2 = lds128(pu + 64 + 32 * h + 16 * c);
          const uint4 v3 = lds128(pu + 128 + 32 * h + 16 * c);
          xs.p1[4 * c] = v1.x; xs.p1[4 * c + 1] = v1.y; xs.p1[4 * c + 2] = v1.z; xs.p1[4 * c + 3] = v1.w;
          xs.p2[4 * c] = v2.x; xs.p2[4 * c + 1] = v2.y; xs.p2[4 * c + 2] = v2.z; xs.p2[4 * c + 3] = v2.w;
          xs.p3[4 * c] = v3.x; xs.p3[4 * c + 1] = v3.y; xs.p3[4 * c + 2] = v3.z; xs.p3[4 * c + 3] = v3.w;
        }
        xs.scale = xscale[2 * u + h];
        xs.sum = xsum[2 * u + h];
        xs.ea = xa[2 * u + h];
        xs.eb = xb[2 * u + h];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xsl.p1[i] = xsl.p2[i] = xsl.p3[i] = xsh.p1[i] = xsh.p2[i] = xsh.p3[i] = 0;
      }
      xsl.scale = xsh.scale = 1.f;
      xsl.sum = xsh.sum = 0.f;
      xsl.ea = xsh.ea = xsl.eb = xsh.eb = 0.f;
    }
    const int off_h = sb * kQ4KBytes, off_a = off_h + 16 + 32 * g;
    bool ok = true;
    int cs = 0;          // ring slot of the next iteration
    uint32_t cph = 0u;   // and the parity of its phase
    for (int it0 = 0; it0 < iters && ok; it0 += SPB) {
      // slots 0..7: the row sums of 8 rows, 8..15: their certificate terms
      float pa[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pa[i] = 0.f;
#pragma unroll
      for (int q = 0; q < SPB; ++q) {
        const int it = it0 + q;
        if (it < iters && ok) {
          const int s = cs;
          const uint32_t ph = cph;
          if (++cs == a.stages) {
            cs = 0;
            cph ^= 1u;
          }
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_fast(full0 + 8 * s, ph, a.wait_limit_ns, &g_gemv_error));
          if (ok) {
            const int nr = min(rps, rows - it * rps);
            const uint8_t* stage = ring + s * a.stage_stride + (size_t)team * RPT * rowbytes;
            if (nr == rps) {
              // a full stage: every row of the team is there
              if (active) {
#pragma unroll
                for (int j = 0; j < RPT; j += 2) {
                  const float4 p2 = q4_group_dot2i(stage + j * rowbytes, stage + (j + 1) * rowbytes,
                                                   off_h, off_a, sel0, sel1, upper, xsl, xsh);
                  pa[q * RPT + j] = p2.x;
                  pa[q * RPT + j + 1] = p2.y;
                  pa[8 + q * RPT + j] = p2.z;
                  pa[8 + q * RPT + j + 1] = p2.w;
                }
              }
            } else {
#pragma unroll
              for (int j = 0; j < RPT; j += 2) {
                const int ra = team * RPT + j;
                if (active && ra < nr) {
                  const bool two = ra + 1 < nr;
                  const float4 p2 = q4_group_dot2i(stage + j * rowbytes,
                                                   stage + (two ? j + 1 : j) * rowbytes, off_h,
                                                   off_a, sel0, sel1, upper, xsl, xsh);
                  pa[q * RPT + j] = p2.x;
                  pa[q * RPT + j + 1] = two ? p2.y : 0.f;
                  pa[8 + q * RPT + j] = p2.z;
                  pa[8 + q * RPT + j + 1] = two ? p2.w : 0.f;
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
          }
        }
      }
      // slot (lane >> 1) & 15: kind (sum / certificate) and row slot of this
      // warp's 8 rows (stage it0 + slot / RPT, team row slot % RPT)
      const float tot = reduce16(pa, lane);
      const int slot = (lane >> 1) & 7;
      const int it = it0 + slot / RPT;
      if ((lane & 1) == 0 && it < iters) {
        const int rr = team * RPT + slot % RPT;
        if (rr < min(rps, rows - it * rps)) atomicAdd((lane & 16 ? dacc : acc) + it * rps + rr, tot);
      }
    }
  }
  __syncthreads();
  // Outputs whose certificate holds are stored; the others are listed and
  // recomputed exactly, one warp per output.  Rows split between the CTAs of
  // a cluster: rank 1 posts its partial sums and certificates into rank 0's
  // receive buffers, and rank 0 adds them after the cluster barrier.
  if (a.ksplit == 2) {
    if (h == 1)
      for (int i = threadIdx.x; i < rows; i += blockDim.x) {
        m1_st_peer(racc + i, 0, acc[i]);
        m1_st_peer(rdacc + i, 0, dacc[i]);
      }
    m1_cluster_sync();  // rank 1's stores are visible to rank 0
    if (h != 0) return;
  }
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    float y = acc[i], D = dacc[i];
    if (a.ksplit == 2) {
      y += racc[i];
      D += rdacc[i];
    }
    if (cert_fails(D)) {
      flist[atomicAdd(nfail, 1)] = i;
    } else {
      const int sg = m1_seg(a, r0 + i);
      a.seg_y[sg][r0 + i - a.seg_start[sg]] = y;
    }
  }
  __syncthreads();
  const int nwarps = blockDim.x >> 5;
  for (int f = warp; f < *nfail; f += nwarps) {
    const int row = r0 + flist[f];
    const int sg = m1_seg(a, row);
    const float y = (float)q4k_row_exact(a.seg_w[sg] + (size_t)(row - a.seg_start[sg]) * rowstride,
                                         a.x, a.K, lane);
    if (lane == 0) {
      a.seg_y[sg][row - a.seg_start[sg]] = y;
      atomicAdd(&g_gemv_exact_outputs, 1ull);
    }
  }
}

// MAXT: the most threads a launch of the instance has (17 warps: 96
// registers a thread; 16 warps: 128).
template <int RPT, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) q4k_gemv_m1_kernel(const __grid_constant__ M1Args a) {
  q4k_m1_body<RPT>(a, blockIdx.x, gridDim.x);
}

// ------------------------------------------------- Q6_K, one token ---------
//
// Same structure as the one-token Q4_K kernel (bulk-copy ring of row stages,
// teams of warps, x as three int8 planes in registers, dp4a inner products,
// 8-row transpose reductions, shared atomics per row).  A lane owns the
// 64 weights 128hh + 32i + 16lq + j (i = 0..3, j = 0..15) of super-block sb
// (unit u = 4 sb + 2 hh + lq): 16 bytes of ql at 64hh + 16lq (i = 0, 2),
// 16 at 64hh + 32 + 16lq (i = 1, 3) and 16 of qh at 128 + 32hh + 16lq,
// with the scale of 16-weight sub-block 8hh + 2i + lq for quarter i.  The
// 6-bit quant q (0..63) enters dp4a as a non-negative int8 and the offset
// is applied once per sub-block: sum x (q - 32) = sum x q - 32 sum x.
// Super-blocks are 210 bytes, so fields are only 2-byte aligned in shared
// memory: each 16-byte field is read as five aligned words and
// funnel-shifted.  Rows are 16-byte aligned only in groups of `row_align`,
// so each CTA's row block and every stage start on such a group; the bytes
// of a final stage past the last 16-byte boundary are copied by the
// producer with plain loads.

struct XSplit16 {
  int p1[4], p2[4], p3[4];  // planes of one 16-weight sub-block
  float sc14;               // s / 16384: one unit of the combined plane value
  int pc;                   // sum over the sub-block of 16384 p1 + 128 p2 + p3
  float ec;                 // error-bound constant of the sub-block (q6k_cert)
};

// Error bound of one lane's 64 Q6_K weights (q6k_cert).  The offset -32 is
// applied in integers: for quarter i the lane forms
//   I_i = sum_k q_k (16384 p1 + 128 p2 + p3)_k - 32 pc_i = 16384 sum_k (q_k - 32) t_k
// exactly (|.| < 2^31), so every later fp32 rounding is relative to
// sum_k |q_k - 32| |x_k| and thus to sum_k |x_k w_k|.  The only other error
// is that of the planes: |t_k - x_k / s| <= r_k / 16384 with the third-plane
// residual r_k <= 1/2, so quarter i contributes at most
//   |d scale_i| * 32 s_i sum_k r_k / 16384 = |d scale_i| * ec_i
// (|q - 32| <= 32; the constant adds a factor 1 + 2^-7).
// `finite`: every x of the sub-block is finite.
__device__ __forceinline__ float q6k_cert_const(float s, float rs, float mx, bool finite) {
  // planes not valid (tiny maximum) or x not finite: exact path
  if ((mx > 0.0f && mx < kCertTinyMax) || !finite) return INFINITY;
  return 32.0f * s * rs * (1.0f / 16384.0f) * (1.0f + 0x1p-7f);
}

// 16 bytes at a 2-byte aligned shared-memory address (the word after the
// field is read and discarded; it lies inside the CTA's shared memory).
__device__ __forceinline__ void lds16u(const uint8_t* p, uint32_t (&w)[4]) {
  const uint32_t mis = smem_u32(p) & 3u;
  const uint32_t* b = reinterpret_cast<const uint32_t*>(p - mis);
  const uint32_t sh = mis * 8u;
  const uint32_t v0 = b[0], v1 = b[1], v2 = b[2], v3 = b[3], v4 = b[4];
  w[0] = __funnelshift_r(v0, v1, sh);
  w[1] = __funnelshift_r(v1, v2, sh);
  w[2] = __funnelshift_r(v2, v3, sh);
  w[3] = __funnelshift_r(v3, v4, sh);
}

// One row's dot product over a lane's unit, with its certificate term:
// returns (p, D).  blk: the super-block in shared memory.
__device__ __forceinline__ float2 q6_unit_dot(const uint8_t* blk, int hh, int lq,
                                              const XSplit16 (&xs)[4]) {
  uint32_t qa[4], qb[4], qh[4], sc[4];
  lds16u(blk + 64 * hh + 16 * lq, qa);
  lds16u(blk + 64 * hh + 32 + 16 * lq, qb);
  lds16u(blk + 128 + 32 * hh + 16 * lq, qh);
  lds16u(blk + 192, sc);  // the 16 int8 scales
  const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 208)));
  Dot3 t[4] = {{0, 0, 0}, {0, 0, 0}, {0, 0, 0}, {0, 0, 0}};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t h = qh[w];
    const int q0 = (int)((qa[w] & 0x0F0F0F0Fu) | ((h << 4) & 0x30303030u));
    const int q1 = (int)((qb[w] & 0x0F0F0F0Fu) | ((h << 2) & 0x30303030u));
    const int q2 = (int)(((qa[w] >> 4) & 0x0F0F0F0Fu) | (h & 0x30303030u));
    const int q3 = (int)(((qb[w] >> 4) & 0x0F0F0F0Fu) | ((h >> 2) & 0x30303030u));
    t[0].a1 = __dp4a(q0, xs[0].p1[w], t[0].a1);
    t[1].a1 = __dp4a(q1, xs[1].p1[w], t[1].a1);
    t[2].a1 = __dp4a(q2, xs[2].p1[w], t[2].a1);
    t[3].a1 = __dp4a(q3, xs[3].p1[w], t[3].a1);
    t[0].a2 = __dp4a(q0, xs[0].p2[w], t[0].a2);
    t[1].a2 = __dp4a(q1, xs[1].p2[w], t[1].a2);
    t[2].a2 = __dp4a(q2, xs[2].p2[w], t[2].a2);
    t[3].a2 = __dp4a(q3, xs[3].p2[w], t[3].a2);
    t[0].a3 = __dp4a(q0, xs[0].p3[w], t[0].a3);
    t[1].a3 = __dp4a(q1, xs[1].p3[w], t[1].a3);
    t[2].a3 = __dp4a(q2, xs[2].p3[w], t[2].a3);
    t[3].a3 = __dp4a(q3, xs[3].p3[w], t[3].a3);
  }
  // scale of sub-block 8hh + 2i + lq: byte 8hh + lq + 2i of the 16
  const uint32_t sw0 = hh ? sc[2] : sc[0], sw1 = hh ? sc[3] : sc[1];
  float r = 0.f, e = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t word = i < 2 ? sw0 : sw1;
    const int bsel = lq + 2 * (i & 1);
    const float s8 = i2f_small((int)(word << (24 - 8 * bsel)) >> 24);  // signed byte
    const int I = t[i].a1 * 16384 + t[i].a2 * 128 + t[i].a3 - 32 * xs[i].pc;
    r = fmaf(s8, __int2float_rn(I) * xs[i].sc14, r);
    e = fmaf(fabsf(s8), xs[i].ec, e);
  }
  const float p = d * r;
  return make_float2(p, fmaf(-kCertTau, fabsf(p), fabsf(d) * e));
}

// Shared-memory layout of the Q6_K x planes: per unit u, 208 bytes: plane p
// (0..2), quarter i (0..3), byte j (0..15) at p*64 + i*16 + j.

template <int RPT>
__device__ __forceinline__ void q6k_m1_body(const M1Args& a, const int bid, const int nblk) {
  static_assert(RPT == 2 || RPT == 4 || RPT == 8, "rows per team per stage");
  constexpr int SPB = 8 / RPT;
  extern __shared__ __align__(128) uint8_t smem_q6[];
  const int nsb = a.K >> 8, U = nsb * 4, nsub16 = a.K >> 4;
  const int rowbytes = nsb * kQ6KBytes;
  const int rps = a.rows_per_stage;
  const uint32_t stage_bytes = (uint32_t)(rps * rowbytes);
  uint8_t* ring = smem_q6;
  uint8_t* planes = ring + a.ring_bytes;                              // U * 208
  float* xsc14 = reinterpret_cast<float*>(planes + U * kPlaneStride);  // nsub16
  int* xpc = reinterpret_cast<int*>(xsc14 + nsub16);                   // nsub16
  float* xec = reinterpret_cast<float*>(xpc + nsub16);                 // nsub16
  uint64_t* bars = reinterpret_cast<uint64_t*>(xec + nsub16 + (nsub16 & 1));
  float* acc = reinterpret_cast<float*>(bars + 2 * a.stages);          // max_rows
  float* dacc = acc + a.max_rows;                                      // max_rows
  int* flist = reinterpret_cast<int*>(dacc + a.max_rows);              // max_rows
  int* nfail = flist + a.max_rows;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + a.stages);

  const int compute_warps = a.teams * a.team_warps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ra = a.row_align;
  const int ngrp = (a.N + ra - 1) / ra;
  const int r0 = min(a.N, (int)((int64_t)bid * ngrp / nblk) * ra);
  const int r1 = min(a.N, (int)((int64_t)(bid + 1) * ngrp / nblk) * ra);
  const int rows = r1 - r0;
  const int iters = (rows + rps - 1) / rps;
  const int first = iters < a.stages ? iters : a.stages;

  for (int i = threadIdx.x; i < rows; i += blockDim.x) acc[i] = dacc[i] = 0.f;
  if (threadIdx.x == 0) {
    *nfail = 0;
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, compute_warps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  uint32_t issued = 0, parity_bits = 0;
  bool prod_ok = true;
  auto produce = [&](int it) {
    const int s = it % a.stages;
    const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, a.wait_limit_ns, &g_gemv_error)) {
      prod_ok = false;
      return;
    }
    const int nr = min(rps, rows - it * rps);
    const uint32_t bytes = (uint32_t)(nr * rowbytes);
    const uint32_t bulk = bytes & ~15u;
    const uint8_t* src = a.W + (size_t)(r0 + it * rps) * rowbytes;
    uint8_t* dst = ring + s * stage_bytes;
    // the last stage of the matrix may end off a 16-byte boundary
    for (uint32_t b = bulk; b < bytes; b += 2)
      *reinterpret_cast<unsigned short*>(dst + b) = (unsigned short)ldg_nc_u16(src + b);
    mbar_arrive_expect_tx(full0 + 8 * s, bulk);
    if (bulk != 0) {
      if (a.evict_first)
        bulk_g2s_hint(smem_u32(dst), src, bulk, full0 + 8 * s, l2_policy_evict_first());
      else
        bulk_g2s(smem_u32(dst), src, bulk, full0 + 8 * s);
    }
    issued |= 1u << s;
    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
  };
  const bool producer = warp == compute_warps && lane == 0;
  if (producer)
    for (int it = 0; it < first && prod_ok; ++it) produce(it);
  pdl_wait();  // x and y only after the previous launch has completed
  pdl_trigger();

  // ------------------------------------------------ x planes (all compute warps)
  // Two lanes per 16-value sub-block, eight values each.
  if (warp < compute_warps) {
    const int half = lane & 1;
    for (int s16 = warp * 16 + (lane >> 1); s16 < nsub16; s16 += compute_warps * 16) {
      const float4* px = reinterpret_cast<const float4*>(a.x + 16 * s16 + 8 * half);
      const float4 va = __ldg(px), vb = __ldg(px + 1);
      const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      float mx = 0.f;
      int nonfin = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx = fmaxf(mx, fabsf(v[i]));
        nonfin |= !isfinite(v[i]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      nonfin |= __shfl_xor_sync(0xFFFFFFFFu, nonfin, 1);
      const float inv = mx > 0.f ? 127.0f / mx : 0.0f;
      uint32_t b1[2] = {0, 0}, b2[2] = {0, 0}, b3[2] = {0, 0};
      int pc = 0;
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float t = fminf(fmaxf(v[i] * inv, -127.0f), 127.0f);
        int i1, i2, i3;
        const float f1 = round_magic(t, i1);
        const float u2 = (t - f1) * 128.0f;
        const float f2 = round_magic(u2, i2);
        const float u3 = (u2 - f2) * 128.0f;
        rs += fabsf(u3 - round_magic(u3, i3));
        pc += i1 * 16384 + i2 * 128 + i3;
        const int sh8 = 8 * (i & 3);
        b1[i >> 2] |= ((uint32_t)i1 & 0xFFu) << sh8;
        b2[i >> 2] |= ((uint32_t)i2 & 0xFFu) << sh8;
        b3[i >> 2] |= ((uint32_t)i3 & 0xFFu) << sh8;
      }
      pc += __shfl_xor_sync(0xFFFFFFFFu, pc, 1);
      rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
      // sub-block s16 = 16 sb + 8 hh + 2 i + lq belongs to unit 4 sb + 2 hh + lq
      const int t16 = s16 & 15;
      const int u = 4 * (s16 >> 4) + 2 * (t16 >> 3) + (t16 & 1), qi = (t16 >> 1) & 3;
      uint8_t* pl = planes + u * kPlaneStride + qi * 16 + 8 * half;
      *reinterpret_cast<uint2*>(pl) = make_uint2(b1[0], b1[1]);
      *reinterpret_cast<uint2*>(pl + 64) = make_uint2(b2[0], b2[1]);
      *reinterpret_cast<uint2*>(pl + 128) = make_uint2(b3[0], b3[1]);
      if (half == 0) {
        const float sc = mx > 0.f ? mx / 127.0f : 1.0f;
        xsc14[4 * u + qi] = sc * (1.0f / 16384.0f);
        xpc[4 * u + qi] = pc;
        xec[4 * u + qi] = q6k_cert_const(sc, rs, mx, nonfin == 0);
      }
    }
  }
  __syncthreads();

  if (producer) {
    for (int it = first; it < iters && prod_ok; ++it) produce(it);
    for (int s = 0; s < a.stages; ++s)
      if (issued & (1u << s))
        mbar_wait(full0 + 8 * s, (parity_bits >> s) & 1u, a.wait_limit_ns, &g_gemv_error);
  } else if (warp < compute_warps) {
    // ------------------------------------------------------------ compute --
    const int team = warp / a.team_warps, wt = warp - team * a.team_warps;
    const int u = wt * 32 + lane;
    const bool active = u < U;
    const int sb = u >> 2, hh = (u >> 1) & 1, lq = u & 1;
    XSplit16 xs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (active) {
        const uint8_t* pu = planes + u * kPlaneStride + 16 * i;
        const uint4 v1 = lds128(pu), v2 = lds128(pu + 64), v3 = lds128(pu + 128);
        xs[i].p1[0] = v1.x; xs[i].p1[1] = v1.y; xs[i].p1[2] = v1.z; xs[i].p1[3] = v1.w;
        xs[i].p2[0] = v2.x; xs[i].p2[1] = v2.y; xs[i].p2[2] = v2.z; xs[i].p2[3] = v2.w;
        xs[i].p3[0] = v3.x; xs[i].p3[1] = v3.y; xs[i].p3[2] = v3.z; xs[i].p3[3] = v3.w;
        xs[i].sc14 = xsc14[4 * u + i];
        xs[i].pc = xpc[4 * u + i];
        xs[i].ec = xec[4 * u + i];
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) xs[i].p1[w] = xs[i].p2[w] = xs[i].p3[w] = 0;
        xs[i].sc14 = 0.f;
        xs[i].pc = 0;
        xs[i].ec = 0.f;
      }
    }
    const int off = sb * kQ6KBytes;
    bool ok = true;
    int cs = 0;          // ring slot of the next iteration
    uint32_t cph = 0u;   // and the parity of its phase
    for (int it0 = 0; it0 < iters && ok; it0 += SPB) {
      float pa[16];  // slots 0..7: row sums, 8..15: their certificate terms
#pragma unroll
      for (int i = 0; i < 16; ++i) pa[i] = 0.f;
#pragma unroll
      for (int qq = 0; qq < SPB; ++qq) {
        const int it = it0 + qq;
        if (it < iters && ok) {
          const int s = cs;
          const uint32_t ph = cph;
          if (++cs == a.stages) {
            cs = 0;
            cph ^= 1u;
          }
          ok = __all_sync(0xFFFFFFFFu, mbar_wait_fast(full0 + 8 * s, ph, a.wait_limit_ns, &g_gemv_error));
          if (ok) {
            const int nr = min(rps, rows - it * rps);
            const uint8_t* stage = ring + s * stage_bytes + (size_t)team * RPT * rowbytes;
#pragma unroll
            for (int j = 0; j < RPT; ++j)
              if (active && team * RPT + j < nr) {
                const float2 pd = q6_unit_dot(stage + j * rowbytes + off, hh, lq, xs);
                pa[qq * RPT + j] = pd.x;
                pa[8 + qq * RPT + j] = pd.y;
              }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
          }
        }
      }
      const float tot = reduce16(pa, lane);
      const int slot = (lane >> 1) & 7;
      const int it = it0 + slot / RPT;
      if ((lane & 1) == 0 && it < iters) {
        const int rr = team * RPT + slot % RPT;
        if (rr < min(rps, rows - it * rps)) atomicAdd((lane & 16 ? dacc : acc) + it * rps + rr, tot);
      }
    }
  }
  __syncthreads();
  // certified outputs are stored, the others recomputed exactly (one warp each)
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    if (cert_fails(dacc[i])) flist[atomicAdd(nfail, 1)] = i;
    else a.y[r0 + i] = acc[i];
  }
  __syncthreads();
  const int nwarps = blockDim.x >> 5;
  for (int f = warp; f < *nfail; f += nwarps) {
    const int row = r0 + flist[f];
    const float y = (float)q6k_row_exact(a.W + (size_t)row * rowbytes, a.x, a.K, lane);
    if (lane == 0) {
      a.y[row] = y;
      atomicAdd(&g_gemv_exact_outputs, 1ull);
    }
  }
}

template <int RPT>
__global__ void __launch_bounds__(544, 1) q6k_gemv_m1_kernel(const __grid_constant__ M1Args a) {
  q6k_m1_body<RPT>(a, blockIdx.x, gridDim.x);
}

// One launch for a token's Q4_K members and one Q6_K member that share x
// (the decoder's q, k and v): CTAs [0, g4) run the Q4_K body over its
// members' rows, the others the Q6_K body, each with its own arguments and
// its own layout of the (shared) dynamic shared memory.  The other
// one-token Q4_K launches run it too, with g4 = the grid (every CTA on the
// Q4_K side), so that a decode pass launches this one kernel throughout.
template <int R4, int R6>
__global__ void __launch_bounds__(544, 1) gemv_m1_dual_kernel(const __grid_constant__ M1Args a4,
                                                              const __grid_constant__ M1Args a6,
                                                              int g4) {
  if ((int)blockIdx.x < g4)
    q4k_m1_body<R4>(a4, blockIdx.x, g4);
  else
    q6k_m1_body<R6>(a6, blockIdx.x - g4, gridDim.x - g4);
}

// ------------------------------------------------- Q6_K, 2..8 tokens ------
//
// The one-token Q6_K kernel's ring, teams and unit ownership, with the x
// planes of all M tokens in shared memory instead of registers.  Per row a
// lane unpacks its 64 quants once, then for each token reads that token's
// planes for its unit (conflict-free 16-byte loads) and takes the dp4a
// products; the M per-token sums of a row are reduced across the warp at
// once with the 8-slot transpose pattern (slot = token).

__global__ void __launch_bounds__(544, 1) q6k_gemv_mt_kernel(const __grid_constant__ M1Args a) {
  extern __shared__ __align__(128) uint8_t smem_q6t[];
  const int M = a.M;
  // with ksplit CTAs per cluster, CTA rank h computes super-blocks
  // [h*nsb, (h+1)*nsb) of every row (whole rows are staged; rank 0 adds the
  // others' sums through distributed shared memory)
  const int ks = a.ksplit;
  const int h = ks > 1 ? (int)m1_cluster_rank() : 0;
  const int nsb = (a.K >> 8) / ks, U = nsb * 4, nsub16 = nsb * 16;
  const int sb0 = h * nsb;
  const int rowbytes = (a.K >> 8) * kQ6KBytes;
  const int rps = a.rows_per_stage;
  const uint32_t stage_bytes = (uint32_t)(rps * rowbytes);
  uint8_t* ring = smem_q6t;
  uint8_t* planes = ring + a.ring_bytes;                                    // M * U * 208
  float* xsc14 = reinterpret_cast<float*>(planes + (size_t)M * U * kPlaneStride);  // M * nsub16
  int* xpc = reinterpret_cast<int*>(xsc14 + M * nsub16);                    // M * nsub16
  float* xec = reinterpret_cast<float*>(xpc + M * nsub16);                  // M * nsub16
  uint64_t* bars = reinterpret_cast<uint64_t*>(xec + M * nsub16);
  float* acc = reinterpret_cast<float*>(bars + 2 * a.stages);               // max_rows * M
  float* dacc = acc + a.max_rows * M;                                       // max_rows * M
  int* flist = reinterpret_cast<int*>(dacc + a.max_rows * M);               // max_rows * M
  int* nfail = flist + a.max_rows * M;                                      // 4 words
  float* racc = reinterpret_cast<float*>(nfail + 4);                        // max_rows * M
  float* rdacc = racc + a.max_rows * M;                                     // max_rows * M
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + a.stages);

  const int compute_warps = a.teams * a.team_warps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ra = a.row_align;
  const int ngrp = (a.N + ra - 1) / ra;
  const int cb = (int)blockIdx.x / ks, ncb = (int)gridDim.x / ks;  // row block of the cluster
  const int r0 = min(a.N, (int)((int64_t)cb * ngrp / ncb) * ra);
  const int r1 = min(a.N, (int)((int64_t)(cb + 1) * ngrp / ncb) * ra);
  const int rows = r1 - r0;
  const int iters = (rows + rps - 1) / rps;
  const int first = iters < a.stages ? iters : a.stages;

  for (int i = threadIdx.x; i < rows * M; i += blockDim.x) acc[i] = dacc[i] = 0.f;
  if (threadIdx.x == 0) {
    *nfail = 0;
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, compute_warps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  uint32_t issued = 0, parity_bits = 0;
  bool prod_ok = true;
  auto produce = [&](int it) {
    const int s = it % a.stages;
    const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
    if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, a.wait_limit_ns, &g_gemv_error)) {
      prod_ok = false;
      return;
    }
    const int nr = min(rps, rows - it * rps);
    const uint32_t bytes = (uint32_t)(nr * rowbytes);
    const uint32_t bulk = bytes & ~15u;
    const uint8_t* src = a.W + (size_t)(r0 + it * rps) * rowbytes;
    uint8_t* dst = ring + s * stage_bytes;
    for (uint32_t b = bulk; b < bytes; b += 2)
      *reinterpret_cast<unsigned short*>(dst + b) = (unsigned short)ldg_nc_u16(src + b);
    mbar_arrive_expect_tx(full0 + 8 * s, bulk);
    if (bulk != 0) {
      if (a.evict_first)
        bulk_g2s_hint(smem_u32(dst), src, bulk, full0 + 8 * s, l2_policy_evict_first());
      else
        bulk_g2s(smem_u32(dst), src, bulk, full0 + 8 * s);
    }
    issued |= 1u << s;
    parity_bits = (parity_bits & ~(1u << s)) | (ph << s);
  };
  const bool producer = warp == compute_warps && lane == 0;
  if (producer)
    for (int it = 0; it < first && prod_ok; ++it) produce(it);
  pdl_wait();  // x and y only after the previous launch has completed
  pdl_trigger();

  // x planes of every token: two lanes per 16-value sub-block
  if (warp < compute_warps) {
    const int half = lane & 1;
    for (int idx = warp * 16 + (lane >> 1); idx < M * nsub16; idx += compute_warps * 16) {
      const int m = idx / nsub16, s16 = idx - m * nsub16;
      const float4* px =
          reinterpret_cast<const float4*>(a.x + (size_t)m * a.K + 256 * sb0 + 16 * s16 + 8 * half);
      const float4 va = __ldg(px), vb = __ldg(px + 1);
      const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      float mx = 0.f;
      int nonfin = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx = fmaxf(mx, fabsf(v[i]));
        nonfin |= !isfinite(v[i]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      nonfin |= __shfl_xor_sync(0xFFFFFFFFu, nonfin, 1);
      const float inv = mx > 0.f ? 127.0f / mx : 0.0f;
      uint32_t b1[2] = {0, 0}, b2[2] = {0, 0}, b3[2] = {0, 0};
      int pc = 0;
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float t = fminf(fmaxf(v[i] * inv, -127.0f), 127.0f);
        int i1, i2, i3;
        const float f1 = round_magic(t, i1);
        const float u2 = (t - f1) * 128.0f;
        const float f2 = round_magic(u2, i2);
        const float u3 = (u2 - f2) * 128.0f;
        rs += fabsf(u3 - round_magic(u3, i3));
        pc += i1 * 16384 + i2 * 128 + i3;
        const int sh8 = 8 * (i & 3);
        b1[i >> 2] |= ((uint32_t)i1 & 0xFFu) << sh8;
        b2[i >> 2] |= ((uint32_t)i2 & 0xFFu) << sh8;
        b3[i >> 2] |= ((uint32_t)i3 & 0xFFu) << sh8;
      }
      pc += __shfl_xor_sync(0xFFFFFFFFu, pc, 1);
      rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
      const int t16 = s16 & 15;
      const int u = 4 * (s16 >> 4) + 2 * (t16 >> 3) + (t16 & 1), qi = (t16 >> 1) & 3;
      uint8_t* pl = planes + ((size_t)m * U + u) * kPlaneStride + qi * 16 + 8 * half;
      *reinterpret_cast<uint2*>(pl) = make_uint2(b1[0], b1[1]);
      *reinterpret_cast<uint2*>(pl + 64) = make_uint2(b2[0], b2[1]);
      *reinterpret_cast<uint2*>(pl + 128) = make_uint2(b3[0], b3[1]);
      if (half == 0) {
        const float sc = mx > 0.f ? mx / 127.0f : 1.0f;
        const int at = m * nsub16 + 4 * u + qi;
        xsc14[at] = sc * (1.0f / 16384.0f);
        xpc[at] = pc;
        xec[at] = q6k_cert_const(sc, rs, mx, nonfin == 0);
      }
    }
  }
  __syncthreads();

  if (producer) {
    for (int it = first; it < iters && prod_ok; ++it) produce(it);
    for (int s = 0; s < a.stages; ++s)
      if (issued & (1u << s))
        mbar_wait(full0 + 8 * s, (parity_bits >> s) & 1u, a.wait_limit_ns, &g_gemv_error);
  } else if (warp < compute_warps) {
    const int team = warp / a.team_warps, wt = warp - team * a.team_warps;
    const int rpt = rps / a.teams;
    const int u = wt * 32 + lane;
    const bool active = u < U;
    const int sb = u >> 2, hh = (u >> 1) & 1, lq = u & 1;
    const int off = (sb0 + sb) * kQ6KBytes;
    bool ok = true;
    int cs = 0;          // ring slot of the next iteration
    uint32_t cph = 0u;   // and the parity of its phase
    for (int it = 0; it < iters && ok; ++it) {
      const int s = cs;
      const uint32_t ph = cph;
      if (++cs == a.stages) {
        cs = 0;
        cph ^= 1u;
      }
      ok = __all_sync(0xFFFFFFFFu, mbar_wait_fast(full0 + 8 * s, ph, a.wait_limit_ns, &g_gemv_error));
      if (!ok) break;
      const int nr = min(rps, rows - it * rps);
      const uint8_t* stage = ring + s * stage_bytes;
      for (int j = 0; j < rpt; ++j) {
        const int rr = team * rpt + j;
        float pa[16];  // slots 0..7: the token sums, 8..15: their certificate terms
#pragma unroll
        for (int m = 0; m < 16; ++m) pa[m] = 0.f;
        if (active && rr < nr) {
          const uint8_t* blk = stage + (size_t)rr * rowbytes + off;
          uint32_t qa[4], qb[4], qh[4], sc[4];
          lds16u(blk + 64 * hh + 16 * lq, qa);
          lds16u(blk + 64 * hh + 32 + 16 * lq, qb);
          lds16u(blk + 128 + 32 * hh + 16 * lq, qh);
          lds16u(blk + 192, sc);
          const float d = __half2float(
              __ushort_as_half(*reinterpret_cast<const unsigned short*>(blk + 208)));
          int q[4][4];  // quarter i, word w
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t h = qh[w];
            q[0][w] = (int)((qa[w] & 0x0F0F0F0Fu) | ((h << 4) & 0x30303030u));
            q[1][w] = (int)((qb[w] & 0x0F0F0F0Fu) | ((h << 2) & 0x30303030u));
            q[2][w] = (int)(((qa[w] >> 4) & 0x0F0F0F0Fu) | (h & 0x30303030u));
            q[3][w] = (int)(((qb[w] >> 4) & 0x0F0F0F0Fu) | ((h >> 2) & 0x30303030u));
          }
          const uint32_t sw0 = hh ? sc[2] : sc[0], sw1 = hh ? sc[3] : sc[1];
          float s8[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t word = i < 2 ? sw0 : sw1;
            const int bsel = lq + 2 * (i & 1);
            s8[i] = i2f_small((int)(word << (24 - 8 * bsel)) >> 24);
          }
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            if (m < M) {
              const uint8_t* pu = planes + ((size_t)m * U + u) * kPlaneStride;
              const float4 xsc = *reinterpret_cast<const float4*>(xsc14 + m * nsub16 + 4 * u);
              const int4 xp = *reinterpret_cast<const int4*>(xpc + m * nsub16 + 4 * u);
              const float4 xe = *reinterpret_cast<const float4*>(xec + m * nsub16 + 4 * u);
              const float sc14[4] = {xsc.x, xsc.y, xsc.z, xsc.w};
              const int pcs[4] = {xp.x, xp.y, xp.z, xp.w};
              const float ecs[4] = {xe.x, xe.y, xe.z, xe.w};
              float r = 0.f, e = 0.f;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 v1 = lds128(pu + 16 * i), v2 = lds128(pu + 64 + 16 * i);
                const uint4 v3 = lds128(pu + 128 + 16 * i);
                const int p1[4] = {(int)v1.x, (int)v1.y, (int)v1.z, (int)v1.w};
                const int p2[4] = {(int)v2.x, (int)v2.y, (int)v2.z, (int)v2.w};
                const int p3[4] = {(int)v3.x, (int)v3.y, (int)v3.z, (int)v3.w};
                Dot3 t = {0, 0, 0};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  t.a1 = __dp4a(q[i][w], p1[w], t.a1);
                  t.a2 = __dp4a(q[i][w], p2[w], t.a2);
                  t.a3 = __dp4a(q[i][w], p3[w], t.a3);
                }
                // offset -32 in integers, as in the one-token kernel (q6k_cert)
                const int I = t.a1 * 16384 + t.a2 * 128 + t.a3 - 32 * pcs[i];
                r = fmaf(s8[i], __int2float_rn(I) * sc14[i], r);
                e = fmaf(fabsf(s8[i]), ecs[i], e);
              }
              const float pm = d * r;
              pa[m] = pm;
              pa[8 + m] = fmaf(-kCertTau, fabsf(pm), fabsf(d) * e);
            }
          }
        }
        // slot (lane >> 1) & 15: kind (sum / certificate) and token
        const float tot = reduce16(pa, lane);
        const int slot = (lane >> 1) & 7;
        if ((lane & 1) == 0 && slot < M && rr < nr)
          atomicAdd((lane & 16 ? dacc : acc) + (it * rps + rr) * M + slot, tot);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
  }
  __syncthreads();
  // two CTAs per row block: rank 1 posts its sums and certificates into rank
  // 0's receive buffers before the cluster barrier
  if (ks > 1) {
    if (h == 1)
      for (int i = threadIdx.x; i < rows * M; i += blockDim.x) {
        m1_st_peer(racc + i, 0, acc[i]);
        m1_st_peer(rdacc + i, 0, dacc[i]);
      }
    m1_cluster_sync();  // rank 1's stores are visible to rank 0
    if (h != 0) return;
  }
  for (int i = threadIdx.x; i < rows * M; i += blockDim.x) {
    const int row = i / M, m = i - row * M;
    float v = acc[i], D = dacc[i];
    if (ks > 1) {
      v += racc[i];
      D += rdacc[i];
    }
    if (cert_fails(D)) flist[atomicAdd(nfail, 1)] = i;
    else a.y[(size_t)m * a.N + r0 + row] = v;
  }
  __syncthreads();
  // outputs whose certificate fails: exact recomputation, one warp each
  const int nwarps = blockDim.x >> 5;
  for (int f = warp; f < *nfail; f += nwarps) {
    const int row = flist[f] / M, m = flist[f] - row * M;
    const float y = (float)q6k_row_exact(a.W + (size_t)(r0 + row) * rowbytes,
                                         a.x + (size_t)m * a.K, a.K, lane);
    if (lane == 0) {
      a.y[(size_t)m * a.N + r0 + row] = y;
      atomicAdd(&g_gemv_exact_outputs, 1ull);
    }
  }
}

// ---------------------------------------------------------------- launch --

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D view [N rows][K/256 super-blocks][144 B] of a Q4_K weight with a box of
// `rows` rows x `sbs` super-blocks; rows past N read as zero.
bool q4k_stage_map(CUtensorMap* map, const uint8_t* w, int N, int K, int sbs, int rows) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const int nsb = K / kQK;
  const cuuint64_t dims[3] = {(cuuint64_t)kQ4KBytes, (cuuint64_t)nsb, (cuuint64_t)N};
  const cuuint64_t strides[2] = {(cuuint64_t)kQ4KBytes, (cuuint64_t)nsb * kQ4KBytes};
  const cuuint32_t box[3] = {(cuuint32_t)kQ4KBytes, (cuuint32_t)sbs, (cuuint32_t)rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(w), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Resident CTAs per SM for a kernel at a dynamic shared-memory size; the
// occupancy query is cached per (kernel, smem) since it costs host time.
template <typename KernelT>
int blocks_per_sm(KernelT kernel, size_t smem) {
  static std::map<std::pair<const void*, size_t>, int> cache;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  cache.emplace(key, per_sm);
  return per_sm;
}

template <typename KernelT>
int persistent_grid(KernelT kernel, size_t smem, int ngroups) {
  const int per_sm = blocks_per_sm(kernel, smem);
  const int want = (ngroups + kWarps - 1) / kWarps;
  const int cap = device_sm_count() * per_sm;
  return want < cap ? (want < 1 ? 1 : want) : cap;
}

// RQ_GEMV_LOG: one line per GEMV launch on stderr naming the kernel chosen
// (tuning runs and the tests that pin the choice for the decoder shapes).
void gemv_log(const char* kernel, int M, int N, int K, int grid) {
  if (std::getenv("RQ_GEMV_LOG") != nullptr)
    std::fprintf(stderr, "rq_gemv: %s M=%d N=%d K=%d grid=%d\n", kernel, M, N, K, grid);
}

template <int M, int R>
rq_status run_q4k(const uint8_t* w, const float* x, float* y, int N, int K,
                  cudaStream_t st) {
  auto kern = q4k_gemv_kernel<M, R>;
  const int grid = persistent_grid(kern, 0, (N + R - 1) / R);
  // launched without programmatic serialization: measured on GB300, this
  // small persistent grid launched early slows its neighbours down
  gemv_log("q4k_generic", M, N, K, grid);
  kern<<<grid, kThreads, 0, st>>>(w, x, y, N, K);
  return launch_status();
}

template <int M, int R>
rq_status run_q6k(const uint8_t* w, const float* x, float* y, int N, int K,
                  cudaStream_t st) {
  auto kern = q6k_gemv_kernel<M, R>;
  const int grid = persistent_grid(kern, 0, (N + R - 1) / R);
  // launched without programmatic serialization: measured on GB300, this
  // small persistent grid launched early slows its neighbours down
  gemv_log("q6k_generic", M, N, K, grid);
  kern<<<grid, kThreads, 0, st>>>(w, x, y, N, K);
  return launch_status();
}

// Launch shape of a one-token kernel: its arguments, dynamic shared memory,
// threads, grid and rows per team per stage.
struct M1Plan {
  M1Args a;
  size_t smem;
  int threads;
  int grid;
  int rpt;
};

int m1_knob(const char* name, int dflt, int lo, int hi) {
  const char* e = std::getenv(name);
  const int v = e ? std::atoi(e) : dflt;
  return v < lo ? lo : (v > hi ? hi : v);
}

template <typename Kern>
rq_status m1_allow_smem(Kern kern, size_t smem, size_t& set) {
  if (smem <= set) return RQ_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return RQ_ERR_CUDA;
  set = smem;
  return RQ_OK;
}

// One-token Q4_K shape: team_warps = ceil(K/64/32), up to 16 compute warps
// per CTA, one CTA per SM (or `grid` CTAs when positive), shared memory split
// between the x planes and a ring of weight stages.  The RQ_GEMV_*
// environment variables override the shape for tuning runs.
rq_status plan_q4k_m1(int nseg, const int* starts, const uint8_t* const* ws, float* const* ys,
                      const float* x, int K, int grid, bool allow_ksplit, M1Plan* p) {
  const int N = starts[nseg];
  const int sms = device_sm_count();
  // rows longer than 8 warps' worth of 64-weight groups are split between
  // the two CTAs of a cluster (more warps per SM for the long rows of a
  // down projection); RQ_GEMV_KSPLIT=0 / 1 forces it off / on (on needs an
  // even number of super-blocks per row)
  const int nsb_full = K / kQK;
  int ksplit = ((nsb_full * 4 + 31) / 32 > 8) ? 2 : 1;
  if (const char* e = std::getenv("RQ_GEMV_KSPLIT")) ksplit = std::atoi(e) != 0 ? 2 : 1;
  if (!allow_ksplit || nsb_full % 2 != 0 || sms < 2) ksplit = 1;
  if (grid <= 0) grid = ksplit * (N < sms / ksplit ? N : sms / ksplit);
  if (grid > ksplit * N) grid = ksplit * N;
  const int max_rows = (N + grid / ksplit - 1) / (grid / ksplit);
  // defaults from launch-shape sweeps on GB300: few rows per CTA favour
  // smaller teams and stages; long rows favour a shallower ring
  const bool few_rows = max_rows <= 8;
  const int warps_per_cta = m1_knob("RQ_GEMV_WARPS", few_rows ? 8 : 16, 1, 16);
  int rpt = m1_knob("RQ_GEMV_RPT", few_rows ? 2 : 4, 2, 8);
  rpt = rpt >= 8 ? 8 : (rpt >= 4 ? 4 : 2);
  const int Kc = K / ksplit;  // the part of a row one CTA reads
  const int ring_kb = m1_knob("RQ_GEMV_RING_KB", Kc >= 8192 ? 100 : 150, 16, 200);
  const int max_stages = m1_knob("RQ_GEMV_STAGES", 8, 2, 16);
  const int U = Kc / 64, nsub = Kc / 32;
  M1Args& a = p->a;
  a.W = ws[0];
  a.x = x;
  a.y = ys[0];
  a.N = N;
  a.K = K;
  a.nseg = nseg;
  for (int i = 0; i <= RQ_MAX_GROUP; ++i) a.seg_start[i] = starts[i <= nseg ? i : nseg];
  for (int i = 0; i < RQ_MAX_GROUP; ++i) {
    a.seg_w[i] = i < nseg ? ws[i] : nullptr;
    a.seg_y[i] = i < nseg ? ys[i] : nullptr;
  }
  a.row_align = 1;
  a.M = 1;
  a.ksplit = ksplit;
  a.team_warps = (U + 31) / 32;
  if (a.team_warps > 16) return RQ_ERR_SHAPE;
  a.teams = a.team_warps >= warps_per_cta ? 1 : warps_per_cta / a.team_warps;
  {
    // no more teams than a CTA's rows keep busy in one stage (measured on
    // GB300: o 3584 x 3584, 24 rows a CTA, 6 teams instead of 8: 4.95 ->
    // 4.73 us; RQ_GEMV_TEAM_CAP=0 keeps every team)
    const int busy = (max_rows + rpt - 1) / rpt;
    if (m1_knob("RQ_GEMV_TEAM_CAP", 1, 0, 1) == 1 && a.teams > busy) a.teams = busy;
  }
  a.rows_per_stage = rpt * a.teams;
  const int rowbytes = (Kc / kQK) * kQ4KBytes;
  const int stage_bytes = a.rows_per_stage * rowbytes;
  // split rows of a single weight: one 3-D copy per stage (RQ_GEMV_TMA3D=0:
  // one bulk copy per half-row instead); TMA destinations 128-byte aligned
  a.tma = (ksplit == 2 && nseg == 1 && m1_knob("RQ_GEMV_TMA3D", 1, 0, 1) == 1 &&
           a.rows_per_stage <= 256 && Kc / kQK <= 256) ? 1 : 0;
  if (a.tma && !q4k_stage_map(&a.map, ws[0], N, K, Kc / kQK, a.rows_per_stage)) a.tma = 0;
  a.stage_stride = a.tma ? (uint32_t)((stage_bytes + 127) & ~127) : (uint32_t)stage_bytes;
  const size_t nsub2 = (size_t)((nsub + 1) & ~1);
  // planes; per sub-block: scale, sum, two error-bound constants; barriers;
  // per row: sum, certificate, exact-path list; the list's count
  const size_t fixed = (size_t)U * kPlaneStride + 16 * nsub2 + 16 * (size_t)max_stages +
                       20 * (size_t)max_rows + 16;
  const size_t limit = 227 * 1024;
  if (fixed + 2 * (size_t)a.stage_stride > limit) return RQ_ERR_SHAPE;
  size_t ring = (size_t)ring_kb * 1024;
  if (ring > limit - fixed) ring = limit - fixed;
  int stages = (int)(ring / a.stage_stride);
  stages = stages > max_stages ? max_stages : (stages < 2 ? 2 : stages);
  // no more stages than a CTA has iterations
  const int iters_max = (max_rows + a.rows_per_stage - 1) / a.rows_per_stage;
  if (stages > iters_max) stages = iters_max < 1 ? 1 : iters_max;
  a.stages = stages;
  a.ring_bytes = (uint32_t)stages * a.stage_stride;
  a.wait_limit_ns = kWaitLimitNs;
  a.max_rows = max_rows;
  // weights are read once per pass: their copies go to L2 with priority
  // evict_first, which keeps x, y and the kernel's code there (measured on
  // GB300: decode pass 1.198 -> 1.181 ms; RQ_GEMV_EVICT_FIRST=0 turns it off)
  a.evict_first = m1_knob("RQ_GEMV_EVICT_FIRST", 1, 0, 1);
  p->smem = a.ring_bytes + (size_t)U * kPlaneStride + 16 * nsub2 + 16 * (size_t)stages +
            20 * (size_t)max_rows + 16;
  p->threads = (a.teams * a.team_warps + 1) * 32;
  p->grid = grid;
  p->rpt = rpt;
  return RQ_OK;
}

// Dynamic shared memory the mixed-launch kernel instances have been allowed
// (index (R4 == 4 ? 2 : 0) + (R6 == 4 ? 1 : 0)), shared by its launchers.
size_t g_dual_smem_set[4] = {48 * 1024, 48 * 1024, 48 * 1024, 48 * 1024};

rq_status run_q4k_m1(int nseg, const int* starts, const uint8_t* const* ws, float* const* ys,
                     const float* x, int K, cudaStream_t st) {
  M1Plan p;
  const rq_status s = plan_q4k_m1(nseg, starts, ws, ys, x, K, 0, true, &p);
  if (s != RQ_OK) return s;
  // One-token Q4_K launches with 2 or 4 rows per team per stage run the
  // kernel of the mixed q/k/v launch, every CTA on its Q4_K side: a decode
  // pass then launches a single kernel, whose code stays in the SMs'
  // instruction caches from one launch to the next (measured on GB300: the
  // 28-layer decode pass 1.323 ms with three kernels, 1.256 with two, 1.197
  // with one; RQ_GEMV_ONE_KERNEL=0 keeps the separate instances).
  if ((p.rpt == 4 || p.rpt == 2) && m1_knob("RQ_GEMV_ONE_KERNEL", 1, 0, 1) == 1) {
    auto dk = p.rpt == 4 ? gemv_m1_dual_kernel<4, 4> : gemv_m1_dual_kernel<2, 2>;
    const rq_status sd = m1_allow_smem(dk, p.smem, g_dual_smem_set[p.rpt == 4 ? 3 : 0]);
    if (sd != RQ_OK) return sd;
    gemv_log(p.a.ksplit == 1 ? "q4k_m1 (mixed kernel)" : "q4k_m1_ksplit (mixed kernel)", 1, p.a.N,
             K, p.grid);
    if (p.a.ksplit == 1)
      return launch_kernel(dk, p.grid, p.threads, p.smem, st, p.a, p.a, p.grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, dk, p.a, p.a, p.grid));
  }
  // launches of up to 16 warps take the instance compiled for 512 threads
  // (128 registers a thread, where 17 warps allow 96)
  const bool w16 = p.threads <= 512 && m1_knob("RQ_GEMV_W16", 1, 0, 1) == 1;
  auto kern = p.rpt == 8 ? (w16 ? q4k_gemv_m1_kernel<8, 512> : q4k_gemv_m1_kernel<8, 544>)
            : p.rpt == 4 ? (w16 ? q4k_gemv_m1_kernel<4, 512> : q4k_gemv_m1_kernel<4, 544>)
                         : (w16 ? q4k_gemv_m1_kernel<2, 512> : q4k_gemv_m1_kernel<2, 544>);
  static size_t smem_set[6] = {48 * 1024, 48 * 1024, 48 * 1024, 48 * 1024, 48 * 1024, 48 * 1024};
  const rq_status sa = m1_allow_smem(
      kern, p.smem, smem_set[(p.rpt == 8 ? 2 : (p.rpt == 4 ? 1 : 0)) + (w16 ? 3 : 0)]);
  if (sa != RQ_OK) return sa;
  gemv_log(p.a.ksplit == 1 ? "q4k_m1" : "q4k_m1_ksplit", 1, p.a.N, K, p.grid);
  if (p.a.ksplit == 1) return launch_kernel(kern, p.grid, p.threads, p.smem, st, p.a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, p.a));
}

// One-token (M = 1) or multi-token (M = 2..8) Q6_K shape: as for Q4_K, plus
// the row alignment of the bulk copies (rows are 16-byte aligned in groups of
// 16 / gcd(rowbytes, 16)); `grid` CTAs when positive.
rq_status plan_q6k_m1(const uint8_t* w, const float* x, float* y, int M, int N, int K, int grid,
                      M1Plan* p) {
  if ((reinterpret_cast<uintptr_t>(w) & 15) != 0) return RQ_ERR_SHAPE;
  const int nsb = K / kQK;
  const int rowbytes = nsb * kQ6KBytes;
  int g = 1;
  while (g < 16 && rowbytes % (2 * g) == 0) g *= 2;  // gcd(rowbytes, 16)
  const int ra = 16 / g;
  const int sms = device_sm_count();
  const int ngrp = (N + ra - 1) / ra;
  // launches of 6..8 tokens with fewer row groups than SMs split each row's
  // super-blocks between the two CTAs of a cluster (each CTA builds the x
  // planes of its half only; measured on the 512 x 3584 shape: 10.6 -> 9.9 us
  // at 8 tokens, no gain at 4, a loss at 2); RQ_GEMV_Q6_KSPLIT=0 / 1 forces
  // it off / on for 2..8 tokens
  int ks = (M >= 6 && ngrp < sms) ? 2 : 1;
  if (const char* e = std::getenv("RQ_GEMV_Q6_KSPLIT")) ks = std::atoi(e) != 0 ? 2 : 1;
  if (M == 1 || nsb % 2 != 0 || sms < 2) ks = 1;
  const int U = nsb / ks * 4, nsub16 = nsb / ks * 16;
  if (grid <= 0) grid = ks * (ngrp < sms / ks ? ngrp : sms / ks);
  if (grid > ks * ngrp) grid = ks * ngrp;
  const int max_rows = (ngrp + grid / ks - 1) / (grid / ks) * ra;
  // (a few-token launch keeps 16 warps: its x prologue scales with M)
  const bool few_rows = max_rows <= 8;
  const int warps_per_cta = m1_knob("RQ_GEMV_WARPS", few_rows && M == 1 ? 8 : 16, 1, 16);
  int rpt = m1_knob("RQ_GEMV_RPT", few_rows ? 2 : 4, 2, 8);
  rpt = rpt >= 8 ? 8 : (rpt >= 4 ? 4 : 2);
  // split rows: one row per team per stage, so that all warps (which build
  // the x planes) fit next to a ring of whole rows
  if (ks > 1) rpt = 1;
  const int ring_kb = m1_knob("RQ_GEMV_RING_KB", 150, 16, 200);
  const int max_stages = m1_knob("RQ_GEMV_STAGES", 8, 2, 16);
  M1Args& a = p->a;
  a.W = w;
  a.x = x;
  a.y = y;
  a.N = N;
  a.K = K;
  a.row_align = ra;
  a.M = M;
  a.ksplit = ks;
  a.tma = 0;
  a.nseg = 1;
  a.seg_start[0] = 0;
  for (int i = 1; i <= RQ_MAX_GROUP; ++i) a.seg_start[i] = N;
  for (int i = 0; i < RQ_MAX_GROUP; ++i) {
    a.seg_w[i] = w;
    a.seg_y[i] = y;
  }
  a.team_warps = (U + 31) / 32;
  a.teams = a.team_warps >= warps_per_cta ? 1 : warps_per_cta / a.team_warps;
  a.rows_per_stage = rpt * a.teams;
  if (a.rows_per_stage % ra != 0) return RQ_ERR_SHAPE;
  const int stage_bytes = a.rows_per_stage * rowbytes;
  // planes; per token and sub-block: scale, offset sum, error-bound constant;
  // barriers; per output: sum, certificate, exact-path list; the list's count
  const size_t fixed = (size_t)M * U * kPlaneStride + 12 * (size_t)M * nsub16 +
                       16 * (size_t)max_stages + 20 * (size_t)M * max_rows + 16;
  const size_t limit = 227 * 1024;
  if (fixed + 2 * (size_t)stage_bytes > limit) return RQ_ERR_SHAPE;
  size_t ring = (size_t)ring_kb * 1024;
  if (ring > limit - fixed) ring = limit - fixed;
  int stages = (int)(ring / stage_bytes);
  stages = stages > max_stages ? max_stages : (stages < 2 ? 2 : stages);
  // no more stages than a CTA has iterations
  const int iters_max = (max_rows + a.rows_per_stage - 1) / a.rows_per_stage;
  if (stages > iters_max) stages = iters_max < 1 ? 1 : iters_max;
  a.stages = stages;
  a.ring_bytes = (uint32_t)(stages * stage_bytes);
  a.stage_stride = (uint32_t)stage_bytes;
  a.wait_limit_ns = kWaitLimitNs;
  a.max_rows = max_rows;
  // weights are read once per pass: their copies go to L2 with priority
  // evict_first, which keeps x, y and the kernel's code there (measured on
  // GB300: decode pass 1.198 -> 1.181 ms; RQ_GEMV_EVICT_FIRST=0 turns it off)
  a.evict_first = m1_knob("RQ_GEMV_EVICT_FIRST", 1, 0, 1);
  p->smem = a.ring_bytes + (size_t)M * U * kPlaneStride + 12 * (size_t)M * nsub16 +
            16 * (size_t)stages + 20 * (size_t)M * max_rows + 16;
  p->threads = (a.teams * a.team_warps + 1) * 32;
  p->grid = grid;
  p->rpt = rpt;
  return RQ_OK;
}

rq_status run_q6k_m1(const uint8_t* w, const float* x, float* y, int M, int N, int K,
                     cudaStream_t st) {
  M1Plan p;
  const rq_status s = plan_q6k_m1(w, x, y, M, N, K, 0, &p);
  if (s != RQ_OK) return s;
  auto kern = M > 1 ? q6k_gemv_mt_kernel
                    : (p.rpt == 8 ? q6k_gemv_m1_kernel<8>
                                  : (p.rpt == 4 ? q6k_gemv_m1_kernel<4> : q6k_gemv_m1_kernel<2>));
  static size_t smem_set[4] = {48 * 1024, 48 * 1024, 48 * 1024, 48 * 1024};
  const rq_status sa =
      m1_allow_smem(kern, p.smem, smem_set[M > 1 ? 3 : (p.rpt == 8 ? 2 : (p.rpt == 4 ? 1 : 0))]);
  if (sa != RQ_OK) return sa;
  gemv_log(M > 1 ? (p.a.ksplit > 1 ? "q6k_mt_ksplit" : "q6k_mt") : "q6k_m1", M, N, K, p.grid);
  if (p.a.ksplit == 1) return launch_kernel(kern, p.grid, p.threads, p.smem, st, p.a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.a.ksplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, p.a));
}

}  // namespace

rq_status read_and_clear_gemv_error() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v)) != cudaSuccess) return RQ_ERR_CUDA;
  if (v == 0) return RQ_OK;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero)) != cudaSuccess) return RQ_ERR_CUDA;
  return RQ_ERR_TIMEOUT;
}

rq_status read_and_clear_gemv_exact_outputs(int64_t* out) {
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_exact_outputs, sizeof(v)) != cudaSuccess)
    return RQ_ERR_CUDA;
  const unsigned long long zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_gemv_exact_outputs, &zero, sizeof(zero)) != cudaSuccess)
    return RQ_ERR_CUDA;
  if (out != nullptr) *out = (int64_t)v;
  return RQ_OK;
}

rq_status launch_q4k_gemv(const uint8_t* w, const float* x, float* y, int M,
                          int N, int K, cudaStream_t st) {
  if (M < 1 || M > 8) return RQ_ERR_SHAPE;
  // the one-token kernel keeps 64 x values per lane in registers; its team
  // of ceil(K/2048) warps plus the producer warp fit 544 threads.  Several
  // tokens take one launch each (the weight is read once per token).
  if (K <= 32 * 2048 && std::getenv("RQ_GEMV_GENERIC") == nullptr) {
    const int starts[2] = {0, N};
    for (int m = 0; m < M; ++m) {
      float* ym = y + (size_t)m * N;
      // RQ_ERR_SHAPE: the shape does not fit the kernel or its shared
      // memory and nothing was launched, so the generic kernel takes it
      const rq_status s1 = run_q4k_m1(1, starts, &w, &ym, x + (size_t)m * K, K, st);
      if (s1 == RQ_ERR_SHAPE && m == 0) break;
      if (s1 != RQ_OK) return s1;
      if (m == M - 1) return RQ_OK;
    }
  }
  switch (M) {
    case 1: return run_q4k<1, 2>(w, x, y, N, K, st);
    case 2: return run_q4k<2, 2>(w, x, y, N, K, st);
    case 3: return run_q4k<3, 2>(w, x, y, N, K, st);
    case 4: return run_q4k<4, 2>(w, x, y, N, K, st);
    case 5: return run_q4k<5, 1>(w, x, y, N, K, st);
    case 6: return run_q4k<6, 1>(w, x, y, N, K, st);
    case 7: return run_q4k<7, 1>(w, x, y, N, K, st);
    default: return run_q4k<8, 1>(w, x, y, N, K, st);
  }
}

rq_status launch_q4k_gemv_group(int count, const int* starts, const uint8_t* const* ws,
                                float* const* ys, const float* x, int K, cudaStream_t st) {
  if (count < 1 || count > RQ_MAX_GROUP || K > 32 * 2048) return RQ_ERR_SHAPE;
  return run_q4k_m1(count, starts, ws, ys, x, K, st);
}

rq_status launch_gemv_m1_dual(int count, const int* starts, const uint8_t* const* ws,
                              float* const* ys, const uint8_t* w6, float* y6, int n6,
                              const float* x, int K, cudaStream_t st) {
  if (count < 1 || count > RQ_MAX_GROUP || K > 16 * 2048 || n6 < 1) return RQ_ERR_SHAPE;
  const int sms = device_sm_count();
  // CTAs in proportion to the work: a Q6_K weight costs about 1.5 times the
  // instructions of a Q4_K weight in these kernels
  const double c4 = (double)starts[count], c6 = 1.5 * n6;
  int g6 = (int)(sms * c6 / (c4 + c6) + 0.5);
  g6 = m1_knob("RQ_GEMV_DUAL_G6", g6, 1, sms - 1);
  M1Plan p4, p6;
  rq_status s = plan_q4k_m1(count, starts, ws, ys, x, K, sms - g6, false, &p4);
  if (s != RQ_OK) return s;
  s = plan_q6k_m1(w6, x, y6, 1, n6, K, g6, &p6);
  if (s != RQ_OK) return s;
  if ((p4.rpt != 2 && p4.rpt != 4) || (p6.rpt != 2 && p6.rpt != 4)) return RQ_ERR_SHAPE;
  auto kern = p4.rpt == 4 ? (p6.rpt == 4 ? gemv_m1_dual_kernel<4, 4> : gemv_m1_dual_kernel<4, 2>)
                          : (p6.rpt == 4 ? gemv_m1_dual_kernel<2, 4> : gemv_m1_dual_kernel<2, 2>);
  const size_t smem = p4.smem > p6.smem ? p4.smem : p6.smem;
  const int threads = p4.threads > p6.threads ? p4.threads : p6.threads;
  s = m1_allow_smem(kern, smem, g_dual_smem_set[(p4.rpt == 4 ? 2 : 0) + (p6.rpt == 4 ? 1 : 0)]);
  if (s != RQ_OK) return s;
  gemv_log("dual_q4k_q6k_m1", 1, starts[count] + n6, K, p4.grid + p6.grid);
  return launch_kernel(kern, p4.grid + p6.grid, threads, smem, st, p4.a, p6.a, p4.grid);
}

rq_status launch_q6k_gemv(const uint8_t* w, const float* x, float* y, int M,
                          int N, int K, cudaStream_t st) {
  switch (M) {
    case 1:
      if (K <= 16 * 2048 && std::getenv("RQ_GEMV_Q6_GENERIC") == nullptr) {
        // RQ_ERR_SHAPE: the one-token kernel does not take this shape or
        // alignment and nothing was launched
        const rq_status s1 = run_q6k_m1(w, x, y, 1, N, K, st);
        if (s1 != RQ_ERR_SHAPE) return s1;
      }
      return run_q6k<1, 2>(w, x, y, N, K, st);
    default:
      break;
  }
  if (M >= 2 && M <= 8 && K <= 16 * 2048 && std::getenv("RQ_GEMV_Q6_GENERIC") == nullptr) {
    // the multi-token variant (x planes of all tokens in shared memory);
    // RQ_ERR_SHAPE: they do not fit and nothing was launched
    const rq_status s2 = run_q6k_m1(w, x, y, M, N, K, st);
    if (s2 != RQ_ERR_SHAPE) return s2;
  }
  switch (M) {
    case 2: return run_q6k<2, 2>(w, x, y, N, K, st);
    case 3: return run_q6k<3, 1>(w, x, y, N, K, st);
    case 4: return run_q6k<4, 1>(w, x, y, N, K, st);
    case 5: return run_q6k<5, 1>(w, x, y, N, K, st);
    case 6: return run_q6k<6, 1>(w, x, y, N, K, st);
    case 7: return run_q6k<7, 1>(w, x, y, N, K, st);
    case 8: return run_q6k<8, 1>(w, x, y, N, K, st);
    default: return RQ_ERR_SHAPE;
  }
}

}  // namespace rq
