// rq_internal.h -- host-side interfaces between the librq translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/rq.h"

namespace rq {

// Map a CUDA error (or a pending launch error) to a status.
inline rq_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}
inline rq_status launch_status() { return cuda_status(cudaGetLastError()); }

int device_sm_count();

// Programmatic dependent launch of the library's kernels (on unless the
// environment sets RQ_PDL=0 when the library first launches).
bool pdl_enabled();

// Launch with programmatic stream serialization (when enabled), so that the
// kernel can be scheduled while its predecessor in the stream finishes.
template <typename... KArgs, typename... Args>
rq_status launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cuda_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

// rq_quant.cu ---------------------------------------------------------------
// Zero *absmax_bits on the stream, then reduce max|x| into it.
rq_status launch_absmax(const float* x, int64_t n, uint32_t* absmax_bits,
                        cudaStream_t st);
// Encode n elements of x with the device absmax, zero-fill out[n..n_out),
// write the dequant scale (if non-null).
rq_status launch_quant(const float* x, int64_t n, int64_t n_out,
                       const uint32_t* absmax_bits, uint8_t* out,
                       float* dequant_out, cudaStream_t st);

// Absmax + encode in one cooperative wave: x held in registers when it fits
// one wave of them (up to 512 x 24 float4 per CTA), else up to 220 KB per
// CTA of x staged in shared memory and the rest, at the front of x and at
// most 16 MB -- 128 MB for tensors of 2^24 elements or more -- streamed by
// all CTAs and read twice.
// Needs x 16-byte and out 4-byte aligned; RQ_ERR_SHAPE (nothing launched) if
// the wave does not fit the GPU.  `state` is one 64-bit device word and
// `slots` `nslots` of them (at least the SM count), all zero before the
// first launch and used by this kernel only, on one stream at a time.
// absmax_out / dequant_out may be null.
bool act_quant_fused_fits(const float* x, int64_t n, const uint8_t* out);
rq_status launch_act_quant_fused(const float* x, int64_t n, int64_t n_out,
                                 uint8_t* out, uint32_t* absmax_out,
                                 float* dequant_out, unsigned long long* state,
                                 unsigned long long* slots, int nslots, cudaStream_t st);
// Two kernels, no zeroing: per-CTA partial maxima into `slots` (at least
// act_quant_slots() words), then the encoding, which reduces the slots and
// walks x backwards (what the first pass read last may still be in L2).
int act_quant_slots();
rq_status launch_act_quant_two_pass(const float* x, int64_t n, int64_t n_out, uint8_t* out,
                                    uint32_t* slots, uint32_t* absmax_out,
                                    float* dequant_out, cudaStream_t st);
// Absmax + encode in one launch of one thread-block cluster (x read twice,
// the second time from L2): for small activations.  Needs x 16-byte and out
// 4-byte aligned (else RQ_ERR_SHAPE, nothing launched); absmax_out /
// dequant_out may be null.
rq_status launch_act_quant_cluster(const float* x, int64_t n, int64_t n_out, uint8_t* out,
                                   uint32_t* absmax_out, float* dequant_out,
                                   cudaStream_t st);
// Read and clear the one-pass kernel's device error word (after a sync).
rq_status read_and_clear_quant_error();

// rq_gemv.cu ----------------------------------------------------------------
rq_status launch_q4k_gemv(const uint8_t* w, const float* x, float* y, int M,
                          int N, int K, cudaStream_t st);
rq_status launch_q6k_gemv(const uint8_t* w, const float* x, float* y, int M,
                          int N, int K, cudaStream_t st);
// One-token Q4_K GEMV over the rows of several weights that share x
// (member i: rows [starts[i], starts[i+1]) of ws[i] into ys[i]); one launch.
// RQ_ERR_SHAPE (nothing launched) when the shape does not fit the kernel.
rq_status launch_q4k_gemv_group(int count, const int* starts, const uint8_t* const* ws,
                                float* const* ys, const float* x, int K, cudaStream_t st);
// One launch for the one-token GEMVs of Q4_K members (as above) and one Q6_K
// weight w6 ([n6 x K], into y6) that share x.  RQ_ERR_SHAPE (nothing
// launched) when the shapes do not fit the kernel.
rq_status launch_gemv_m1_dual(int count, const int* starts, const uint8_t* const* ws,
                              float* const* ys, const uint8_t* w6, float* y6, int n6,
                              const float* x, int K, cudaStream_t st);
// Read and clear the GEMV kernels' device error word (after a sync).
rq_status read_and_clear_gemv_error();
// Read (into *out, if non-null) and clear the count of GEMV outputs that took
// the exact fp64 path (after a sync).
rq_status read_and_clear_gemv_exact_outputs(int64_t* out);

// rq_wcache.cu --------------------------------------------------------------
// Decode the packed weight (fixed fp32 order) and reduce its absmax into
// *absmax_bits (which the caller zeroed on the stream).
rq_status launch_dequant_absmax(int qtype, const uint8_t* w, int N, int K,
                                uint32_t* absmax_bits, cudaStream_t st);
// Decode again and encode with 448/absmax'; write the dequant scale.
rq_status launch_dequant_encode(int qtype, const uint8_t* w, int N, int K,
                                const uint32_t* absmax_bits, uint8_t* out,
                                float* dequant_out, cudaStream_t st);

// rq_gemm.cu ----------------------------------------------------------------
// w_early: the weight was written before the launch preceding this one began
// (a cached weight built by an earlier call); the kernel may then start
// loading its first weight tiles before that launch has completed.
rq_status launch_fp8_gemm(const uint8_t* x_fp8, const float* x_deq,
                          const uint8_t* w_fp8, const float* w_deq, float* y,
                          int M, int N, int K, cudaStream_t st, bool w_early = false);
// One GEMM over weights concatenated by rows: member i owns rows
// [starts[i], starts[i+1]), its scale w_deqs[i] and its output ys[i]
// ([M x (starts[i+1] - starts[i])]).  count <= RQ_MAX_GROUP.
rq_status launch_fp8_gemm_group(const uint8_t* x_fp8, const float* x_deq,
                                const uint8_t* w_fp8, int count, const int* starts,
                                float* const* ys, const float* const* w_deqs, int M, int K,
                                cudaStream_t st, bool w_early = false);
rq_status read_and_clear_device_error(cudaStream_t st);
rq_status launch_debug_wait_timeout(int64_t limit_ns, cudaStream_t st);

}  // namespace rq
