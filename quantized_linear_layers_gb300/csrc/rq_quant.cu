// rq_quant.cu -- per-tensor absmax and scaled FP32 -> E4M3 quantization.
//
// realizar 0.8.4, cublas_prefill/mod.rs: ABSMAX_REDUCE_PTX (block max of |x|
// folded into a pre-zeroed word with an unsigned atomic max, valid because
// non-negative float bit patterns order like their values) and
// F32_TO_E4M3_DEVICE_SCALED_PTX (scale read from device memory, thread 0
// writes absmax/448).  Both are HBM-bound streaming kernels: 16-byte loads,
// grid sized to a multiple of the SM count, grid-stride loops.
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
  if (vec)
    absmax_kernel<true><<<grid, kThreads, 0, st>>>(x, n, absmax_bits);
  else
    absmax_kernel<false><<<grid, kThreads, 0, st>>>(x, n, absmax_bits);
  return launch_status();
}

rq_status launch_quant(const float* x, int64_t n, int64_t n_out,
                       const uint32_t* absmax_bits, uint8_t* out,
                       float* dequant_out, cudaStream_t st) {
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(out) & 3) == 0;
  const int grid = grid_for(vec ? (n_out + 3) / 4 : n_out);
  if (vec)
    quant_kernel<true><<<grid, kThreads, 0, st>>>(x, n, n_out, absmax_bits, out,
                                                  dequant_out);
  else
    quant_kernel<false><<<grid, kThreads, 0, st>>>(x, n, n_out, absmax_bits,
                                                   out, dequant_out);
  return launch_status();
}

}  // namespace rq
