// rq_gemm.cu -- FP8 E4M3 prefill GEMM on sm_103a tensor cores.
//
// realizar 0.8.4, cublas_prefill/gemm.rs, cublas_prefill_fp8_gemm: the GEMM
// multiplies raw E4M3 codes, and the activation scale act_absmax/448 and the
// weight scale w_absmax/448 are applied afterwards from device memory (no host
// sync).  The pages call cuBLASLt into an f16 buffer and rescale in a second
// kernel; here both scales are applied to the fp32 accumulator in the GEMM's
// own epilogue, and the GEMM is hand-written:
//
//   Y[m, n] = (sum_k e4m3(X[m, k]) * e4m3(W[n, k])) * x_deq * w_deq
//
// Roles (192 threads, one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: 128 x 128 B tiles of W and BN x 128 B tiles of
//               X (SWIZZLE_128B) into a shared-memory ring (8 stages by
//               default, fewer where they do not fit; RQ_GEMM_STAGES sets
//               another depth for tuning);
//   warp 1      allocates TMEM, and one thread issues tcgen05.mma
//               (kind::f8f6f4, E4M3 x E4M3 -> f32, M = 128, N = BN, K = 32)
//               into one of two TMEM accumulators (2 x BN columns);
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)...), scale, masked coalesced f32 stores.
// The tile's MMA M dimension is the weight rows (N of the problem) and its
// MMA N dimension is the tokens, so M padded to 16 is a valid MMA width.
// Every mbarrier wait is bounded by a time limit; on expiry the kernel
// records RQ_ERR_TIMEOUT in a device word, drains its own copies and MMAs,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>

#include "rq_device.cuh"
#include "rq_internal.h"

namespace rq {

__device__ unsigned int g_rq_device_error;  // bit 0: a pipeline wait timed out

namespace {

constexpr int kBM = 128;               // weight rows per tile (MMA M)
constexpr int kBK = 128;               // K bytes per stage = one swizzle row
constexpr int kStages = 4;             // default ring depth, split-K kernel
// Default ring depth of the one-CTA kernel (capped by what fits).  Measured
// on GB300 at 16 tokens (graph-replayed, weights from HBM): the 37888 x 3584
// gate/up group 26.1 us with 4 stages, 24.3 with 6 to 10.  The split-K
// kernel keeps 4: 8 stages made its long splits (the 3584 x 18944 down
// projection) faster alone (16 tokens 16.7 -> 15.9 us) but the 28-layer
// stack at 32 tokens slower (2.34 -> 2.49 ms per pass), its larger shared
// memory keeping the next launch from starting beside it.
constexpr int kStagesSingle = 8;
constexpr int kMaxStages = 16;
constexpr int kMaxBN = 256;
constexpr int kMaxSegs = RQ_MAX_GROUP;  // members of a grouped launch
constexpr int kThreads = 192;
// pair kernel: producer, MMA issuer and 8 epilogue warps (two per TMEM lane
// quarter, each storing half of the tile's token columns)
constexpr int kThreadsPair = 320;
constexpr int kABytes = kBM * kBK;           // 16 KB
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory a CTA may opt into

// --------------------------------------------------------- PTX wrappers --

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map,
                                            uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// start address >> 4 (bits 0-13), leading byte offset 16 B (unused for this
// layout, bits 16-29), stride byte offset 1024 B between 8-row groups
// (bits 32-45), descriptor version 1 (bit 46), swizzle mode 2 = 128 B
// (bits 61-63).  Tile bases are 1024-byte aligned, so the base offset is 0;
// the K step inside the 128-byte row advances the start address by 32 B.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f8f6f4: D = f32 (bits 4-5 = 1), A = B = E4M3
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(int mma_m, int mma_n) {
  return (1u << 4) | ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(mma_m >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
        "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
        "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------- kernel ----

// Output rows [start[i], start[i+1]) of the (concatenated) weight belong to
// member i of a group of linear layers that share the input: its own output
// y[i] ([M x (start[i+1] - start[i])], row-major) and its own weight scale.
// A single GEMM is one segment.
struct OutSegs {
  int count;
  int start[kMaxSegs + 1];
  float* y[kMaxSegs];
  const float* w_deq[kMaxSegs];
};

// Segment of output row n (a short scan: at most kMaxSegs segments).
__device__ __forceinline__ int seg_of(const OutSegs& o, int n) {
  int i = 0;
  while (i + 1 < o.count && n >= o.start[i + 1]) ++i;
  return i;
}

struct GemmArgs {
  const float* x_deq;
  OutSegs out;
  int M, N, K;
  int bn;          // tokens per tile: multiple of 16, <= 256
  int tiles_n;     // ceil(N / 128)
  int tiles_m;     // ceil(M_pad / bn)
  int stages;      // stages of the shared-memory ring
  int w_early;     // 1: the weight was written before the previous launch began
  uint32_t tmem_cols;
  uint64_t wait_limit_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nst = args.stages;                         // stages of the ring
  const uint32_t b_stride = (uint32_t)args.bn * kBK;   // token tile bytes per stage
  uint8_t* sA = smem;                                  // nst x 16 KB
  uint8_t* sB = smem + nst * kABytes;                  // nst x BN x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + nst * b_stride);
  // bars: full[nst], empty[nst], tfull[2], tempty[2], done[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * nst + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + nst);
  const uint32_t tfull0 = smem_u32(bars + 2 * nst);
  const uint32_t tempty0 = smem_u32(bars + 2 * nst + 2);
  const uint32_t done_bar = smem_u32(bars + 2 * nst + 4);
  const int bn = args.bn;
  const int kblocks = args.K / kBK;
  const int ntiles = args.tiles_n * args.tiles_m;
  const uint32_t stage_tx = (uint32_t)(kABytes + bn * kBK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 4);
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(args.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Nothing another launch may write is read before the previous launch has
  // completed, except, with w_early, the weight tiles of the first stages.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int early = 0;  // leading stages whose weight tile went out before the wait
      if (args.w_early) {
        for (int t = blockIdx.x; t < ntiles && early < nst; t += gridDim.x) {
          const int tn = t / args.tiles_m;
          for (int kb = 0; kb < kblocks && early < nst; ++kb, ++early) {
            const uint32_t fb = full0 + 8 * early;
            mbar_arrive_expect_tx(fb, stage_tx);
            tma_load_2d(smem_u32(sA + early * kABytes), &tmap_w, fb, kb * kBK, tn * kBM);
          }
        }
      }
      pdl_wait();
      pdl_trigger();
      int stage = 0, unit = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued, parity
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int tn = t / args.tiles_m, tm = t - tn * args.tiles_m;
        for (int kb = 0; kb < kblocks; ++kb, ++unit) {
          const uint32_t fb = full0 + 8 * stage;
          if (unit >= early) {
            if (!mbar_wait_fast(empty0 + 8 * stage, phase ^ 1, args.wait_limit_ns,
                           &g_rq_device_error)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(fb, stage_tx);
            tma_load_2d(smem_u32(sA + stage * kABytes), &tmap_w, fb, kb * kBK, tn * kBM);
          }
          tma_load_2d(smem_u32(sB + stage * b_stride), &tmap_x, fb, kb * kBK, tm * bn);
          issued_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == nst) { stage = 0; phase ^= 1; }
        }
      }
      // Drain: every issued copy has landed before the CTA can exit.
      for (int s = 0; s < nst; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_fast(full0 + 8 * s, (last_parity >> s) & 1u, args.wait_limit_ns,
                    &g_rq_device_error);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = instr_desc(kBM, bn);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        if (!mbar_wait_fast(tempty0 + 8 * acc, acc_phase ^ 1, args.wait_limit_ns, &g_rq_device_error)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * bn);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_fast(full0 + 8 * stage, phase, args.wait_limit_ns, &g_rq_device_error)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * kABytes);
          const uint32_t b_addr = smem_u32(sB + stage * b_stride);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8(d_tmem, smem_desc(a_addr + 32 * kk), smem_desc(b_addr + 32 * kk), idesc,
                   (kb | kk) != 0);
          mma_commit(empty0 + 8 * stage);  // frees the stage when these MMAs finish
          if (++stage == nst) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);  // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // Drain: all issued MMAs have completed before TMEM is released.
      mma_commit(done_bar);
      mbar_wait_fast(done_bar, 0, args.wait_limit_ns, &g_rq_device_error);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31
    const float scale_x = *args.x_deq;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const int tn = t / args.tiles_m, tm = t - tn * args.tiles_m;
      // every lane polls; the outcome is made warp-uniform before the
      // .sync.aligned TMEM loads below
      const bool ready =
          mbar_wait_fast(tfull0 + 8 * acc, acc_phase, args.wait_limit_ns, &g_rq_device_error);
      if (!__all_sync(0xFFFFFFFFu, ready)) break;
      tc_fence_after();
      const int n = tn * kBM + quad * 32 + lane;
      const int m0 = tm * bn;
      const int sg = seg_of(args.out, n);
      const int ns = args.out.start[sg + 1] - args.out.start[sg];
      float* yr = args.out.y[sg] + (n - args.out.start[sg]);
      const float scale_w = n < args.N ? *args.out.w_deq[sg] : 0.f;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * bn);
      for (int c = 0; c < bn; c += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
        if (n < args.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c + j;
            if (m < args.M) yr[(size_t)m * ns] = (__uint_as_float(v[j]) * scale_x) * scale_w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(args.tmem_cols)
                 : "memory");
  }
}

// ------------------------------------------------------ 2-CTA variant ----
//
// A cluster of two CTAs (a "pair") computes a 256 x BN output tile with
// tcgen05.mma.cta_group::2 (M = 256): CTA r of the pair holds weight rows
// 128r .. 128r+127 of the tile (A) and token rows r*BN/2 .. of the tile (B),
// so each SM streams half of the B tile the 1-CTA kernel needs and the
// tensor cores read half the shared-memory operand bytes per MAC.  Only the
// leader (rank 0) issues MMAs; both CTAs' TMA loads complete on the leader's
// "full" barriers, the leader's commits arrive on both CTAs' "empty" and
// "tmem full" barriers (multicast), and both CTAs' epilogue warps arrive on
// the leader's "tmem empty" barriers.  Each CTA's TMEM holds its 128 rows of
// the accumulator.  All waits are bounded as in the 1-CTA kernel.

constexpr int kStages2 = 6;  // default ring depth, pair kernel
constexpr int kBHalfMax = kMaxBN / 2 * kBK;  // 16 KB: this CTA's half of B
// the most shared memory the pair kernel takes by default (occupancy query)
constexpr int kSmemBytes2 = kStages2 * (kABytes + kBHalfMax) + 1024 + 1024;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Remote arrive without release semantics: a release at cluster scope would
// make the arriving thread wait for all its earlier global stores.  Callers
// order what must be ordered (tcgen05 reads) with tcgen05 fences.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// TMA load into this CTA's shared memory, completing on the pair leader's
// barrier (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t leader_bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(leader_bar)
      : "memory");
}

__device__ __forceinline__ void mma_f8_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at this shared offset in both CTAs of the pair
// when this thread's earlier tcgen05 operations complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"((unsigned short)3)
      : "memory");
}

// Arrive on this CTA's own barrier when this thread's earlier tcgen05
// operations complete (pair granularity).
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsPair, 1)
fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_x, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nst = args.stages;
  const uint32_t b_stride = (uint32_t)(args.bn / 2) * kBK;  // this CTA's half of the token tile
  uint8_t* sA = smem;                            // nst x 16 KB
  uint8_t* sB = smem + nst * kABytes;            // nst x BN/2 x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + nst * b_stride);
  // bars: full[nst], empty[nst], tfull[2], tempty[2], done[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * nst + 5);

  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + nst);
  const uint32_t tfull0 = smem_u32(bars + 2 * nst);
  const uint32_t tempty0 = smem_u32(bars + 2 * nst + 2);
  const uint32_t done_bar = smem_u32(bars + 2 * nst + 4);
  const int bn = args.bn, half = bn / 2;
  const int kblocks = args.K / kBK;
  const int ntiles = args.tiles_n * args.tiles_m;  // tiles_n counts 256-row tiles
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const uint32_t stage_tx = (uint32_t)(kABytes + half * kBK);  // bytes per CTA per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);   // the leader's expect_tx for both CTAs' bytes
      mbar_init(empty0 + 8 * s, 1);  // the leader's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 16);  // 8 epilogue warps x 2 CTAs (leader's is used)
    }
    mbar_init(done_bar, 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(args.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Nothing another launch may write is read before the previous launch has
  // completed, except, with w_early, the weight tiles of the first stages.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    // ---------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int early = 0;  // leading stages whose weight tile went out before the wait
      if (args.w_early) {
        for (int t = pair; t < ntiles && early < nst; t += npairs) {
          const int wrow = t / args.tiles_m * 256 + (int)rank * kBM;
          for (int kb = 0; kb < kblocks && early < nst; ++kb, ++early) {
            // the leader arms its barrier for both CTAs' bytes; the peer's
            // copies may land first (the transaction count may run negative)
            if (leader) mbar_arrive_expect_tx(full0 + 8 * early, 2 * stage_tx);
            tma_load_2d_pair(smem_u32(sA + early * kABytes), &tmap_w,
                             peer_addr(full0 + 8 * early, 0), kb * kBK, wrow);
          }
        }
      }
      pdl_wait();
      pdl_trigger();
      int stage = 0, unit = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < ntiles && ok; t += npairs) {
        const int tn = t / args.tiles_m, tm = t - tn * args.tiles_m;
        const int wrow = tn * 256 + (int)rank * kBM;
        const int trow = tm * bn + (int)rank * half;
        for (int kb = 0; kb < kblocks; ++kb, ++unit) {
          const uint32_t lead_full = peer_addr(full0 + 8 * stage, 0);
          if (unit >= early) {
            if (!mbar_wait_fast(empty0 + 8 * stage, phase ^ 1, args.wait_limit_ns,
                           &g_rq_device_error)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * stage_tx);
            tma_load_2d_pair(smem_u32(sA + stage * kABytes), &tmap_w, lead_full, kb * kBK, wrow);
          }
          tma_load_2d_pair(smem_u32(sB + stage * b_stride), &tmap_x, lead_full, kb * kBK, trow);
          if (++stage == nst) { stage = 0; phase ^= 1; }
        }
      }
      // Drain: this CTA's last copies have landed once the leader's MMAs
      // that consume them have freed the stages (seen on our own "empty").
      for (int i = 0; i < nst && ok; ++i) {
        if (!mbar_wait_fast(empty0 + 8 * stage, phase ^ 1, args.wait_limit_ns, &g_rq_device_error))
          break;
        if (++stage == nst) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (leader)
    if (leader && lane == 0) {
      const uint32_t idesc = instr_desc(256, bn);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < ntiles && ok; t += npairs) {
        if (!mbar_wait_fast(tempty0 + 8 * acc, acc_phase ^ 1, args.wait_limit_ns, &g_rq_device_error))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * bn);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_fast(full0 + 8 * stage, phase, args.wait_limit_ns, &g_rq_device_error)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * kABytes);
          const uint32_t b_addr = smem_u32(sB + stage * b_stride);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8_pair(d_tmem, smem_desc(a_addr + 32 * kk), smem_desc(b_addr + 32 * kk), idesc,
                        (kb | kk) != 0);
          mma_commit_pair(empty0 + 8 * stage);
          if (++stage == nst) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair(tfull0 + 8 * acc);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      mma_commit_pair_local(done_bar);
      mbar_wait_fast(done_bar, 0, args.wait_limit_ns, &g_rq_device_error);
    }
  } else {
    // --------------------------------------------------- epilogue (both)
    const int quad = warp & 3;                       // TMEM lanes 32*quad .. +31
    const int c_lo = ((warp - 2) >> 2) * (bn >> 1);  // this warp's half of the columns
    const int c_hi = c_lo + (bn >> 1);
    const float scale_x = *args.x_deq;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < ntiles; t += npairs) {
      const int tn = t / args.tiles_m, tm = t - tn * args.tiles_m;
      const bool ready =
          mbar_wait_fast(tfull0 + 8 * acc, acc_phase, args.wait_limit_ns, &g_rq_device_error);
      if (!__all_sync(0xFFFFFFFFu, ready)) break;
      tc_fence_after();
      const int n = tn * 256 + (int)rank * kBM + quad * 32 + lane;
      const int m0 = tm * bn;
      const int sg = seg_of(args.out, n);
      const int ns = args.out.start[sg + 1] - args.out.start[sg];
      float* yr = args.out.y[sg] + (n - args.out.start[sg]);
      const float scale_w = n < args.N ? *args.out.w_deq[sg] : 0.f;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * bn);
      for (int c = c_lo; c < c_hi; c += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
        if (n < args.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c + j;
            if (m < args.M) yr[(size_t)m * ns] = (__uint_as_float(v[j]) * scale_x) * scale_w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(tempty0 + 8 * acc);
        else
          mbar_arrive_cluster_relaxed(peer_addr(tempty0 + 8 * acc, 0));
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its peer may still touch its memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(args.tmem_cols)
                 : "memory");
  }
}

// ------------------------------------------------------ split-K variant --
//
// For shapes with too few 128 x BN output tiles to fill the SMs (small N,
// or a few hundred tokens and below): a cluster of S CTAs shares one output
// tile, CTA rank s accumulating K blocks [s*kb/S, (s+1)*kb/S) in its own
// TMEM.  The epilogue writes the partial tile into the CTA's stage buffers
// (idle once the last MMA has completed); after a cluster barrier each CTA
// sums 1/S of the tile's token columns over the S partials through
// distributed shared memory, in rank order, scales and stores y.  One tile
// per cluster (not persistent), no atomics, no zeroing of y.

struct SplitArgs {
  const float* x_deq;
  OutSegs out;
  int M, N, K;
  int bn, tiles_m, splits;
  int stages;  // stages of the shared-memory ring (their bytes also hold the partial tile)
  int w_early;  // 1: the weight was written before the previous launch began
  uint32_t tmem_cols;
  uint64_t wait_limit_ns;
};

// 16 bytes at a shared::cluster address (ordered after the cluster barrier
// by the barrier's own memory clobber; no clobber here, so that several
// loads are in flight before the first is used).
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

constexpr int kMaxSplits = 8;

__global__ void __launch_bounds__(kThreads, 1)
fp8_gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmap_w,
                       const __grid_constant__ CUtensorMap tmap_x, const SplitArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nst = args.stages;
  const uint32_t b_stride = (uint32_t)args.bn * kBK;
  uint8_t* sA = smem;                                  // nst x 16 KB
  uint8_t* sB = smem + nst * kABytes;                  // nst x BN x 128 B
  float* part = reinterpret_cast<float*>(smem);        // [bn][128] after the mainloop
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + nst * b_stride);
  // bars: full[nst], empty[nst], tfull[1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * nst + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + nst);
  const uint32_t tfull = smem_u32(bars + 2 * nst);
  const int S = args.splits;
  const uint32_t rank = cluster_rank();
  const int t = (int)blockIdx.x / S;
  const int tn = t / args.tiles_m, tm = t - tn * args.tiles_m;
  const int bn = args.bn;
  const int kblocks = args.K / kBK;
  const int kb0 = (int)((int64_t)rank * kblocks / S);
  const int kb1 = (int)((int64_t)(rank + 1) * kblocks / S);
  const uint32_t stage_tx = (uint32_t)(kABytes + bn * kBK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(args.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Nothing another launch may write is read before the previous launch has
  // completed, except, with w_early, the weight tiles of the first stages.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      const int early = args.w_early ? min(nst, kb1 - kb0) : 0;
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(full0 + 8 * i, stage_tx);
        tma_load_2d(smem_u32(sA + i * kABytes), &tmap_w, full0 + 8 * i, (kb0 + i) * kBK,
                    tn * kBM);
      }
      pdl_wait();
      pdl_trigger();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t fb = full0 + 8 * stage;
        if (kb - kb0 >= early) {
          if (!mbar_wait_fast(empty0 + 8 * stage, phase ^ 1, args.wait_limit_ns, &g_rq_device_error))
            break;
          mbar_arrive_expect_tx(fb, stage_tx);
          tma_load_2d(smem_u32(sA + stage * kABytes), &tmap_w, fb, kb * kBK, tn * kBM);
        }
        tma_load_2d(smem_u32(sB + stage * b_stride), &tmap_x, fb, kb * kBK, tm * bn);
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == nst) { stage = 0; phase ^= 1; }
      }
      for (int s = 0; s < nst; ++s)
        if (issued_mask & (1u << s))
          mbar_wait_fast(full0 + 8 * s, (last_parity >> s) & 1u, args.wait_limit_ns,
                    &g_rq_device_error);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = instr_desc(kBM, bn);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_fast(full0 + 8 * stage, phase, args.wait_limit_ns, &g_rq_device_error)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sA + stage * kABytes);
        const uint32_t b_addr = smem_u32(sB + stage * b_stride);
#pragma unroll
        for (int kk = 0; kk < kBK / 32; ++kk)
          mma_f8(tmem_base, smem_desc(a_addr + 32 * kk), smem_desc(b_addr + 32 * kk), idesc,
                 (kb != kb0 || kk != 0) ? 1u : 0u);
        mma_commit(empty0 + 8 * stage);
        if (++stage == nst) { stage = 0; phase ^= 1; }
      }
      // completes when every MMA above has: the partial is in TMEM and no
      // MMA reads the stage buffers any more
      mma_commit(tfull);
    }
  } else {
    // ------------------------------------ epilogue: partial tile to smem --
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const bool ready = mbar_wait_fast(tfull, 0, args.wait_limit_ns, &g_rq_device_error);
    if (__all_sync(0xFFFFFFFFu, ready)) {
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16);
      for (int c = 0; c < bn; c += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + (uint32_t)c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) part[(c + j) * kBM + row] = __uint_as_float(v[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every partial of the cluster is in shared memory

  const float scale_x = *args.x_deq;
  float seg_scale[kMaxSegs];  // x scale times each member's weight scale
#pragma unroll
  for (int i = 0; i < kMaxSegs; ++i)
    seg_scale[i] = i < args.out.count ? scale_x * *args.out.w_deq[i] : 0.f;
  uint32_t base[kMaxSplits];  // the partial's address in each CTA of the cluster
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q) {
    base[q] = 0;
    if (q < S)
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                   : "=r"(base[q])
                   : "r"(smem_u32(part)), "r"((uint32_t)q));
  }
  // this CTA's share of the tile: token columns [c0, c1).  Thread t keeps
  // rows 4*(t % 32) .. +3 (blockDim is a multiple of 32), so the members,
  // output pointers and scales of its rows are found once.
  const int c0 = (int)((int64_t)rank * bn / S), c1 = (int)((int64_t)(rank + 1) * bn / S);
  const int r = (threadIdx.x & 31) * 4;
  const int n = tn * kBM + r;
  float* yrow[4];
  int ystride[4];
  float rscale[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int ne = n + e;
    const int sg = seg_of(args.out, ne < args.N ? ne : args.N - 1);
    ystride[e] = args.out.start[sg + 1] - args.out.start[sg];
    yrow[e] = ne < args.N ? args.out.y[sg] + (ne - args.out.start[sg]) : nullptr;
    float sc = seg_scale[0];
#pragma unroll
    for (int i = 1; i < kMaxSegs; ++i)
      if (sg == i) sc = seg_scale[i];
    rscale[e] = sc;
  }
  const uint32_t roff = (uint32_t)(r * 4);
  for (int c = c0 + (int)(threadIdx.x >> 5); c < c1; c += (int)(blockDim.x >> 5)) {
    const uint32_t off = (uint32_t)(c * kBM * 4) + roff;
    float4 v[kMaxSplits];
#pragma unroll
    for (int q = 0; q < kMaxSplits; ++q)
      if (q < S) v[q] = ld_cluster_f4(base[q] + off);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kMaxSplits; ++q)
      if (q < S) {  // rank order
        sum.x += v[q].x;
        sum.y += v[q].y;
        sum.z += v[q].z;
        sum.w += v[q].w;
      }
    const int m = tm * bn + c;
    if (m < args.M) {
      const float o[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (yrow[e] != nullptr) yrow[e][(size_t)m * ystride[e]] = o[e] * rscale[e];
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(args.tmem_cols)
                 : "memory");
  }
}

// A block that waits on an mbarrier nothing completes (timeout test hook).
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    mbar_wait_fast(b, 0, limit_ns, &g_rq_device_error);
  }
}

// ----------------------------------------------------------- host side --

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D map over a row-major [rows x K] byte matrix, box = box_rows x 128 B,
// 128-byte swizzle, out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint32_t tmem_columns(int bn) {
  uint32_t need = (uint32_t)(2 * bn), c = 32;
  while (c < need) c <<= 1;
  return c;
}

// Ring depth for a token tile of b_stride bytes per stage: `dflt`, or
// RQ_GEMM_STAGES (tuning runs), within what fits next to the barriers and
// the alignment slack; at least min_bytes of stage buffers (the split-K
// kernel keeps its partial tile there).
int gemm_stages(int b_stride, int dflt, int min_bytes) {
  const char* env = std::getenv("RQ_GEMM_STAGES");
  int s = env ? std::atoi(env) : dflt;
  const int per = kABytes + b_stride;
  const int fit = (kSmemLimit - 2048) / per;
  while (s * per < min_bytes) ++s;
  if (s > fit) s = fit;
  if (s > kMaxStages) s = kMaxStages;
  return s < 2 ? 2 : s;
}

size_t gemm_smem_bytes(int stages, int b_stride) {
  return 1024 /*alignment slack*/ + (size_t)stages * (kABytes + b_stride) + 1024 /*barriers*/;
}

// Tokens per tile.  Every CTA is resident at once (one per SM), so a launch
// takes ceil(tiles / SMs) rounds.  The kernels stream their operands from L2
// at a rate that caps them (about 100 GB/s per SM on GB300), so a round
// costs about the operand rows a CTA loads per K block: 128 weight rows plus
// the tile's BN tokens (BN/2 in the pair kernel).  Candidates are multiples
// of 16 up to 256; the cheapest estimate wins, ties going to the wider tile.
// RQ_GEMM_BN (a multiple of 16, 16..256) forces a width, for tuning
// measurements.
int choose_bn(int m_pad, int N, int sms) {
  const char* env = std::getenv("RQ_GEMM_BN");
  const int v = env ? std::atoi(env) : 0;
  const int forced = (v >= 16 && v <= kMaxBN && v % 16 == 0) ? v : 0;
  if (forced) return forced < m_pad ? forced : m_pad;
  if (m_pad <= kMaxBN) return m_pad;
  const long tiles_n = (N + kBM - 1) / kBM;
  int best = kMaxBN;
  long best_cost = -1;
  for (int bn = kMaxBN; bn >= 64; bn -= 16) {
    const long tiles = tiles_n * ((m_pad + bn - 1) / bn);
    const long rounds = (tiles + sms - 1) / sms;
    const long cost = rounds * (kBM + bn);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Cost estimates of the two kernels in the units above.
int pair_cost(int m_pad, int N, int pairs, int bn) {
  const long tiles = (long)((N + 255) / 256) * ((m_pad + bn - 1) / bn);
  return (int)(((tiles + pairs - 1) / pairs) * (kBM + bn / 2));
}
int single_cost(int m_pad, int N, int sms, int bn) {
  const long tiles = (long)((N + kBM - 1) / kBM) * ((m_pad + bn - 1) / bn);
  return (int)(((tiles + sms - 1) / sms) * (kBM + bn));
}

// Tokens per tile for the pair kernel: multiples of 32 (each CTA holds half),
// same round-based cost model over the SM pairs.
int choose_bn_pair(int m_pad, int N, int pairs) {
  const char* env = std::getenv("RQ_GEMM_BN");
  const int v = env ? std::atoi(env) : 0;
  const int m32 = (m_pad + 31) / 32 * 32;
  if (v >= 32 && v <= kMaxBN && v % 32 == 0) return v < m32 ? v : m32;
  if (m32 <= kMaxBN) return m32;
  const long tiles_n = (N + 255) / 256;
  int best = kMaxBN;
  long best_cost = -1;
  for (int bn = kMaxBN; bn >= 64; bn -= 32) {
    const long tiles = tiles_n * ((m_pad + bn - 1) / bn);
    const long rounds = (tiles + pairs - 1) / pairs;
    const long cost = rounds * (kBM + bn / 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Number of CTA pairs of the pair kernel that fit on the GPU at once.
int resident_pairs(int sms) {
  static int cached = 0;
  if (cached == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2));
    cfg.blockDim = dim3(kThreadsPair);
    cfg.dynamicSmemBytes = kSmemBytes2;
    int n = 0;
    cudaFuncSetAttribute(fp8_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemLimit);
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    cached = n;
  }
  return cached;
}

// The pair kernel halves the token rows each CTA loads, so it wins unless
// its 256-row tiles leave more of the last round idle; the two are compared
// with the same cost estimate.  RQ_GEMM_PAIR=0 / 1 forces the one-CTA / pair
// kernel.
bool use_pair_kernel(int m_pad, int N, int sms, int pairs, int bn_pair, int bn_single) {
  if (N <= kBM) return false;
  const char* env = std::getenv("RQ_GEMM_PAIR");
  if (env != nullptr) return std::atoi(env) != 0;
  return pair_cost(m_pad, N, pairs, bn_pair) < single_cost(m_pad, N, sms, bn_single);
}

}  // namespace

// K splits for the split-K kernel (1: not used).  Used when the widest
// tiles leave more than half of the SMs idle; each split keeps at least four
// K blocks.  RQ_GEMM_SPLIT forces a split count (1 = never), for tuning.
static int choose_splits(int m_pad, int N, int K, int sms, int* bn_out) {
  const int bn = m_pad < kMaxBN ? m_pad : kMaxBN;
  *bn_out = bn;
  const int tiles = ((N + kBM - 1) / kBM) * ((m_pad + bn - 1) / bn);
  const int kblocks = K / kBK;
  int S = 1;
  const char* env = std::getenv("RQ_GEMM_SPLIT");
  if (env != nullptr) {
    S = std::atoi(env);
  } else if (2 * tiles <= sms) {
    S = sms / tiles;
    if (S > kblocks / 4) S = kblocks / 4;
    if (S > kMaxSplits) S = kMaxSplits;
    if (S >= 2) {
      // Both kernels stream their operands at a rate set by the rows they
      // load per K block (128 weight rows + the tile's tokens); the split
      // kernel adds the exchange of a 128 x BN partial tile, worth about
      // 2400 row-blocks at BN = 256 (fitted to GB300 timings).
      const int rbn = choose_bn(m_pad, N, sms);
      const long rtiles = (long)((N + kBM - 1) / kBM) * ((m_pad + rbn - 1) / rbn);
      const long rounds = (rtiles + sms - 1) / sms;
      const long reg_cost = rounds * (kBM + rbn) * kblocks;
      const long split_cost = (long)(kBM + bn) * ((kblocks + S - 1) / S) + 2400L * bn / 256;
      if (split_cost >= reg_cost) S = 1;
    }
  }
  if (S > kMaxSplits) S = kMaxSplits;
  if (S > kblocks) S = kblocks;
  return S < 2 ? 1 : S;
}

static rq_status launch_fp8_gemm_splitk(const uint8_t* x_fp8, const float* x_deq,
                                        const uint8_t* w_fp8, const OutSegs& out, int M, int N,
                                        int K, int bn, int S, bool w_early, cudaStream_t st) {
  const int m_pad = (M + 15) / 16 * 16;
  CUtensorMap tw, tx;
  if (!make_map(&tw, w_fp8, N, K, kBM) || !make_map(&tx, x_fp8, m_pad, K, bn))
    return RQ_ERR_CUDA;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fp8_gemm_splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit) != cudaSuccess)
      return RQ_ERR_CUDA;
    attr_done = true;
  }
  SplitArgs a;
  a.stages = gemm_stages(bn * kBK, kStages, bn * kBM * 4);
  a.w_early = w_early ? 1 : 0;
  a.x_deq = x_deq;
  a.out = out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bn = bn;
  a.tiles_m = (m_pad + bn - 1) / bn;
  a.splits = S;
  a.tmem_cols = tmem_columns(bn / 2);
  a.wait_limit_ns = kWaitLimitNs;
  const int tiles = ((N + kBM - 1) / kBM) * a.tiles_m;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  if (std::getenv("RQ_GEMM_LOG") != nullptr)
    std::fprintf(stderr, "rq_gemm: split-k M=%d N=%d K=%d bn=%d tiles=%d splits=%d stages=%d\n",
                 M, N, K, bn, tiles, S, a.stages);
  cfg.gridDim = dim3(tiles * S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(a.stages, bn * kBK);
  cfg.stream = st;
  cfg.attrs = attr;
  // Wide token tiles on clusters of 3 or more are launched without
  // programmatic serialization: measured on GB300, their early launch made
  // the 28-layer stack slower (128 tokens: 3.03 -> 2.83 ms per pass without
  // it; 256 tokens: 3.84 -> 3.43 ms), while narrow tiles gain from it.
  const bool pdl = pdl_enabled() && !(bn >= 128 && S >= 3);
  cfg.numAttrs = pdl ? 2 : 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, fp8_gemm_splitk_kernel, tw, tx, a));
}

rq_status launch_fp8_gemm_group(const uint8_t* x_fp8, const float* x_deq,
                                const uint8_t* w_fp8, int count, const int* starts,
                                float* const* ys, const float* const* w_deqs, int M, int K,
                                cudaStream_t st, bool w_early) {
  if (count < 1 || count > kMaxSegs) return RQ_ERR_SHAPE;
  // RQ_GEMM_EARLY=0: no weight loads before the wait (A/B measurements)
  if (const char* e = std::getenv("RQ_GEMM_EARLY")) w_early = w_early && std::atoi(e) != 0;
  OutSegs out;
  out.count = count;
  for (int i = 0; i <= count; ++i) out.start[i] = starts[i];
  for (int i = 0; i < count; ++i) {
    out.y[i] = ys[i];
    out.w_deq[i] = w_deqs[i];
  }
  for (int i = count; i < kMaxSegs; ++i) {
    out.start[i + 1] = starts[count];
    out.y[i] = nullptr;
    out.w_deq[i] = nullptr;
  }
  const int N = starts[count];
  const int m_pad = (M + 15) / 16 * 16;
  const int sms = device_sm_count();
  int bn_split = 0;
  const int S = choose_splits(m_pad, N, K, sms, &bn_split);
  if (S > 1)
    return launch_fp8_gemm_splitk(x_fp8, x_deq, w_fp8, out, M, N, K, bn_split, S, w_early, st);
  const int pairs = sms >= 2 ? resident_pairs(sms) : 0;
  const int bn_pair = sms >= 2 ? choose_bn_pair(m_pad, N, pairs) : 0;
  const int bn_single = choose_bn(m_pad, N, sms);
  const bool pair = sms >= 2 && use_pair_kernel(m_pad, N, sms, pairs, bn_pair, bn_single);
  const int bn = pair ? bn_pair : bn_single;
  CUtensorMap tw, tx;
  if (!make_map(&tw, w_fp8, N, K, kBM) || !make_map(&tx, x_fp8, m_pad, K, pair ? bn / 2 : bn))
    return RQ_ERR_CUDA;
  GemmArgs a;
  a.x_deq = x_deq;
  a.out = out;
  a.M = M;
  a.N = N;
  a.K = K;
  a.bn = bn;
  a.tiles_n = pair ? (N + 255) / 256 : (N + kBM - 1) / kBM;
  a.tiles_m = (m_pad + bn - 1) / bn;
  a.tmem_cols = tmem_columns(bn);
  a.wait_limit_ns = kWaitLimitNs;
  a.w_early = w_early ? 1 : 0;
  const int tiles = a.tiles_n * a.tiles_m;
  if (pair) {
    static bool attr2 = false;
    if (!attr2) {
      if (cudaFuncSetAttribute(fp8_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemLimit) != cudaSuccess)
        return RQ_ERR_CUDA;
      attr2 = true;
    }
    const int b_stride = bn / 2 * kBK;
    a.stages = gemm_stages(b_stride, kStages2, 0);
    // A persistent grid must be resident at once: not every SM can be
    // paired inside its GPC, so the grid is the number of pairs that fit.
    const int max_pairs = resident_pairs(sms);
    const int grid = 2 * (tiles < max_pairs ? tiles : max_pairs);
    if (std::getenv("RQ_GEMM_LOG") != nullptr)
      std::fprintf(stderr, "rq_gemm: pair M=%d N=%d K=%d bn=%d tiles=%d grid=%d stages=%d\n", M,
                   N, K, bn, tiles, grid, a.stages);
    return launch_kernel(fp8_gemm_pair_kernel, grid, kThreadsPair,
                         gemm_smem_bytes(a.stages, b_stride), st, tw, tx, a);
  }
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit) != cudaSuccess)
      return RQ_ERR_CUDA;
    attr_done = true;
  }
  a.stages = gemm_stages(bn * kBK, kStagesSingle, 0);
  const int grid = tiles < sms ? tiles : sms;
  if (std::getenv("RQ_GEMM_LOG") != nullptr)
    std::fprintf(stderr, "rq_gemm: single M=%d N=%d K=%d bn=%d tiles=%d grid=%d stages=%d\n", M,
                 N, K, bn, tiles, grid, a.stages);
  return launch_kernel(fp8_gemm_kernel, grid, kThreads, gemm_smem_bytes(a.stages, bn * kBK), st,
                       tw, tx, a);
}

rq_status launch_fp8_gemm(const uint8_t* x_fp8, const float* x_deq,
                          const uint8_t* w_fp8, const float* w_deq, float* y,
                          int M, int N, int K, cudaStream_t st, bool w_early) {
  const int starts[2] = {0, N};
  return launch_fp8_gemm_group(x_fp8, x_deq, w_fp8, 1, starts, &y, &w_deq, M, K, st, w_early);
}

rq_status read_and_clear_device_error(cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return RQ_ERR_CUDA;
  const rq_status gemv = read_and_clear_gemv_error();
  if (gemv == RQ_ERR_CUDA) return gemv;
  const rq_status quant = read_and_clear_quant_error();
  if (quant == RQ_ERR_CUDA) return quant;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_rq_device_error, sizeof(v)) != cudaSuccess)
    return RQ_ERR_CUDA;
  if (v == 0) return gemv != RQ_OK ? gemv : quant;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_rq_device_error, &zero, sizeof(zero)) != cudaSuccess)
    return RQ_ERR_CUDA;
  return RQ_ERR_TIMEOUT;
}

rq_status launch_debug_wait_timeout(int64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>((uint64_t)limit_ns);
  return launch_status();
}

}  // namespace rq
