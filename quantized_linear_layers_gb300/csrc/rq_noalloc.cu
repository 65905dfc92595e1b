// rq_noalloc.cu -- FP8 linear layer for callers that must not allocate.
//
// Some callers cannot call cudaMalloc on their serving path: code running
// inside a host framework that owns and pre-reserves all device memory (for
// example an inference engine's plugin or operator callback), or a process
// that runs under a fixed device-memory budget where a new allocation would
// fail or stall the device.  rq_fp8_linear_noalloc serves them: it runs the
// same activation absmax, E4M3 quantization and FP8 GEMM kernels as the FP8
// route of rq_linear, but keeps the activation's E4M3 copy and its two device
// scalars in the fixed array below instead of context-owned allocations.
#include <mutex>

#include "rq_internal.h"

namespace rq {
namespace {

// Scratch layout: absmax word at byte 0, activation dequant scale at byte
// 128, activation E4M3 bytes (M_pad x K) from byte 256.  The GPU holds this
// array until the process exits (it may be reserved only when the module is
// loaded, which lazy loading defers to the first call).
constexpr size_t kActOffset = 256;
constexpr size_t kScratchBytes = kActOffset + RQ_NOALLOC_MAX_ACT_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// Device address of the array, looked up on the first call with the device
// current (in host code the array's name is only a host-side stand-in).  The
// library serves one device per process; the table is indexed by device only
// so that the lookup never returns another device's address.
uint8_t* scratch_address() {
  static std::mutex mu;
  static uint8_t* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<uint8_t*>(p);
  }
  return addr[dev];
}

bool is_aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace
}  // namespace rq

extern "C" rq_status rq_fp8_linear_noalloc(const float* x, const uint8_t* w_fp8,
                                           const float* w_dequant, float* y, int M,
                                           int N, int K, rq_stream_t stream) {
  using namespace rq;
  if (x == nullptr || w_fp8 == nullptr || w_dequant == nullptr || y == nullptr)
    return RQ_ERR_NULL;
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return RQ_ERR_SHAPE;
  if (!is_aligned(x, 16) || !is_aligned(w_fp8, 16) || !is_aligned(w_dequant, 4) ||
      !is_aligned(y, 4))
    return RQ_ERR_SHAPE;
  const int64_t m_pad = ((int64_t)M + 15) / 16 * 16;
  const int64_t act_bytes = m_pad * (int64_t)K;
  if (act_bytes > (int64_t)RQ_NOALLOC_MAX_ACT_BYTES) return RQ_ERR_SHAPE;
  uint8_t* base = scratch_address();
  if (base == nullptr) return RQ_ERR_CUDA;
  uint32_t* absmax_word = reinterpret_cast<uint32_t*>(base);
  float* act_deq = reinterpret_cast<float*>(base + 128);
  uint8_t* act = base + kActOffset;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the absmax word is zeroed and the pad rows rewritten on every call, so
  // nothing left in the array by an earlier call reaches this one's result
  rq_status s = launch_absmax(x, (int64_t)M * K, absmax_word, st);
  if (s == RQ_OK) s = launch_quant(x, (int64_t)M * K, act_bytes, absmax_word, act, act_deq, st);
  if (s == RQ_OK) s = launch_fp8_gemm(act, act_deq, w_fp8, w_dequant, y, M, N, K, st);
  return s;
}
