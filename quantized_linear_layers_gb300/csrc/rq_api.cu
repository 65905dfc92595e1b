// rq_api.cu -- the C ABI of librq.so: validation, context, caches, routing.
//
// Host-side counterpart of realizar 0.8.4 cublas_prefill/gemm.rs
// (get_or_cache_fp8_weight, cublas_prefill_fp8_gemm with its activation
// reuse, cublas_prefill_gemm's FP8 branch), cublas_prefill/mod.rs
// (cublas_gemm_threshold, gpu_absmax_device) and q6k_gemv_indexed.rs
// (null-pointer guard before any launch).  Every argument is checked here,
// before anything is launched; kernels never trap.
#include <cstdlib>
#include <cstring>
#include <map>
#include <tuple>
#include <vector>

#include "rq_internal.h"

namespace rq {

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("RQ_PDL");
    return e == nullptr || std::atoi(e) != 0;
  }();
  return on;
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace rq

using namespace rq;

namespace {

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

struct WeightKey {
  const void* w;
  int qtype, N, K;
  bool operator<(const WeightKey& o) const {
    return std::tie(w, qtype, N, K) < std::tie(o.w, o.qtype, o.N, o.K);
  }
};

struct WeightEntry {
  uint8_t* fp8 = nullptr;  // [N x K] E4M3, followed (256-aligned) by the scale
  float* deq = nullptr;
  size_t bytes = 0;
};

// FP8 weights of a group of linears that share an input, concatenated by
// rows: member i's rows start at starts[i]; its dequant scale is deq[i].
struct GroupEntry {
  uint8_t* fp8 = nullptr;
  float* deq = nullptr;
  int starts[RQ_MAX_GROUP + 1] = {0};
  size_t bytes = 0;
};

rq_status check_quant_shape(int qtype, int N, int K) {
  if (qtype != RQ_Q4K && qtype != RQ_Q6K) return RQ_ERR_QTYPE;
  if (N < 1 || K < 256 || K % 256 != 0) return RQ_ERR_SHAPE;
  return RQ_OK;
}

}  // namespace

struct TraceSlot {
  cudaEvent_t start = nullptr, stop = nullptr;
  int kind = 0;
  int kernels = 1;  // kernels launched between the two events
};

struct rq_ctx {
  int device = 0;
  // kernel tracing
  bool trace_on = false;
  unsigned int trace_mask = (1u << RQ_TRACE_KINDS) - 1u;  // kinds that are traced
  int trace_cap = 0, trace_used = 0;
  std::vector<TraceSlot> trace;
  int threshold = 4;
  std::map<WeightKey, WeightEntry> weights;
  std::map<std::vector<WeightKey>, GroupEntry> groups;
  int64_t weight_bytes = 0;
  uint8_t* act = nullptr;  // activation E4M3 scratch [M_pad x K]
  size_t act_cap = 0;
  uint32_t* absmax = nullptr;  // device word
  float* act_deq = nullptr;    // device float
  bool fused_ok = true;           // RQ_ONE_PASS_QUANT=0 keeps the two-kernel path
  int64_t fused_min = 1 << 20;    // fewer elements: two kernels (RQ_ONE_PASS_MIN)
  // at most this many elements: one cluster, one launch (RQ_CLUSTER_QUANT_MAX;
  // measured on GB300, the 16-SM cluster beats the two grid-wide kernels on
  // the 57 K elements of 16 tokens x 3584 and loses from ~230 K on)
  int64_t cluster_max = 1 << 17;
  uint32_t* slots = nullptr;      // per-CTA partial maxima of the two-kernel path
  unsigned long long* fused = nullptr;        // one-pass quantization barrier word
  unsigned long long* fused_slots = nullptr;  // and its per-CTA words (SM count)
  // activation cache key
  bool act_valid = false;
  const float* act_x = nullptr;
  int act_M = 0, act_K = 0;
  uint64_t act_gen = 0, gen = 1;
  int64_t hits = 0, misses = 0;
};

namespace {

cudaError_t record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// Brackets one kernel launch with a trace slot's events while tracing is on.
class TraceScope {
 public:
  TraceScope(rq_ctx* ctx, int kind, cudaStream_t st) : st_(st) {
    if (ctx != nullptr && ctx->trace_on && ((ctx->trace_mask >> kind) & 1u) != 0 &&
        ctx->trace_used < ctx->trace_cap) {
      slot_ = &ctx->trace[ctx->trace_used++];
      slot_->kind = kind;
      slot_->kernels = 1;
      record(slot_->start, st_);
    }
  }
  // the scope launches n kernels (default 1)
  void kernels(int n) {
    if (slot_ != nullptr) slot_->kernels = n;
  }
  ~TraceScope() {
    if (slot_ != nullptr) record(slot_->stop, st_);
  }
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  TraceSlot* slot_ = nullptr;
  cudaStream_t st_;
};

}  // namespace

extern "C" {

int rq_abi_version(void) { return RQ_ABI_VERSION; }

const char* rq_status_string(rq_status s) {
  switch (s) {
    case RQ_OK: return "ok";
    case RQ_ERR_NULL: return "null pointer";
    case RQ_ERR_SHAPE: return "invalid shape or alignment";
    case RQ_ERR_QTYPE: return "unsupported quantization type";
    case RQ_ERR_NOT_CACHED: return "weight not cached";
    case RQ_ERR_ALLOC: return "allocation failed";
    case RQ_ERR_CUDA: return "CUDA error";
    case RQ_ERR_TIMEOUT: return "device pipeline wait timed out";
    case RQ_ERR_ARCH: return "device lacks sm_103 features";
  }
  return "unknown status";
}

rq_status rq_ctx_create(rq_ctx** out) {
  if (out == nullptr) return RQ_ERR_NULL;
  *out = nullptr;
  rq_ctx* c = new (std::nothrow) rq_ctx();
  if (c == nullptr) return RQ_ERR_ALLOC;
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    delete c;
    return RQ_ERR_CUDA;
  }
  const char* env = std::getenv("RQ_GEMM_THRESHOLD");
  if (env != nullptr) {
    const int v = std::atoi(env);
    if (v >= 1) c->threshold = v;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, 256) != cudaSuccess) {
    delete c;
    return RQ_ERR_ALLOC;
  }
  c->absmax = static_cast<uint32_t*>(p);
  c->act_deq = reinterpret_cast<float*>(static_cast<uint8_t*>(p) + 128);
  c->fused = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(p) + 192);
  if (cudaMemset(p, 0, 256) != cudaSuccess) {
    cudaFree(p);
    delete c;
    return RQ_ERR_CUDA;
  }
  const char* one_pass = std::getenv("RQ_ONE_PASS_QUANT");
  if (one_pass != nullptr && std::atoi(one_pass) == 0) c->fused_ok = false;
  // a small activation goes through the two plain kernels: measured on
  // GB300, the cooperative one-pass launch costs more than it saves there
  // (the 28-layer stack at 16 tokens: 2.32 ms per pass one-pass, 2.10 ms
  // with two kernels)
  if (const char* e = std::getenv("RQ_ONE_PASS_MIN")) c->fused_min = std::atoll(e);
  if (const char* e = std::getenv("RQ_CLUSTER_QUANT_MAX")) c->cluster_max = std::atoll(e);
  void* sl = nullptr;
  if (cudaMalloc(&sl, sizeof(uint32_t) * (size_t)act_quant_slots()) != cudaSuccess) {
    cudaFree(p);
    delete c;
    return RQ_ERR_ALLOC;
  }
  c->slots = static_cast<uint32_t*>(sl);
  void* fs = nullptr;
  const size_t fs_bytes = sizeof(unsigned long long) * (size_t)device_sm_count();
  if (cudaMalloc(&fs, fs_bytes) != cudaSuccess) {
    cudaFree(sl);
    cudaFree(p);
    delete c;
    return RQ_ERR_ALLOC;
  }
  if (cudaMemset(fs, 0, fs_bytes) != cudaSuccess) {
    cudaFree(fs);
    cudaFree(sl);
    cudaFree(p);
    delete c;
    return RQ_ERR_CUDA;
  }
  c->fused_slots = static_cast<unsigned long long*>(fs);
  *out = c;
  return RQ_OK;
}

void rq_ctx_destroy(rq_ctx* ctx) {
  if (ctx == nullptr) return;
  for (auto& t : ctx->trace) {
    if (t.start) cudaEventDestroy(t.start);
    if (t.stop) cudaEventDestroy(t.stop);
  }
  for (auto& kv : ctx->weights) cudaFree(kv.second.fp8);
  for (auto& kv : ctx->groups) cudaFree(kv.second.fp8);
  if (ctx->act) cudaFree(ctx->act);
  if (ctx->absmax) cudaFree(ctx->absmax);
  if (ctx->slots) cudaFree(ctx->slots);
  if (ctx->fused_slots) cudaFree(ctx->fused_slots);
  delete ctx;
}

rq_status rq_ctx_set_gemm_threshold(rq_ctx* ctx, int m_threshold) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  if (m_threshold < 1) return RQ_ERR_SHAPE;
  ctx->threshold = m_threshold;
  return RQ_OK;
}

int rq_ctx_get_gemm_threshold(const rq_ctx* ctx) {
  return ctx == nullptr ? -1 : ctx->threshold;
}

rq_status rq_ctx_get_stats(const rq_ctx* ctx, int64_t* act_hits_host,
                           int64_t* act_misses_host, int64_t* weights_host,
                           int64_t* weight_bytes_host) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  if (act_hits_host) *act_hits_host = ctx->hits;
  if (act_misses_host) *act_misses_host = ctx->misses;
  if (weights_host) *weights_host = (int64_t)(ctx->weights.size() + ctx->groups.size());
  if (weight_bytes_host) *weight_bytes_host = ctx->weight_bytes;
  return RQ_OK;
}

rq_status rq_absmax(const float* x, int64_t n, uint32_t* absmax_bits, rq_stream_t stream) {
  if (absmax_bits == nullptr || (x == nullptr && n > 0)) return RQ_ERR_NULL;
  if (n < 0 || !aligned(absmax_bits, 4)) return RQ_ERR_SHAPE;
  return launch_absmax(x, n, absmax_bits, reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_quant_e4m3(const float* x, int64_t n, const uint32_t* absmax_bits,
                        uint8_t* out, float* dequant_out, rq_stream_t stream) {
  if (absmax_bits == nullptr || dequant_out == nullptr) return RQ_ERR_NULL;
  if (n > 0 && (x == nullptr || out == nullptr)) return RQ_ERR_NULL;
  if (n < 0 || !aligned(absmax_bits, 4) || !aligned(dequant_out, 4)) return RQ_ERR_SHAPE;
  return launch_quant(x, n, n, absmax_bits, out, dequant_out,
                      reinterpret_cast<cudaStream_t>(stream));
}

static rq_status check_gemv(const void* w, const float* x, const float* y, int M, int N,
                            int K, uintptr_t w_align) {
  if (w == nullptr || x == nullptr || y == nullptr) return RQ_ERR_NULL;
  if (M < 1 || M > 8 || N < 1 || K < 256 || K % 256 != 0) return RQ_ERR_SHAPE;
  if (!aligned(w, w_align) || !aligned(x, 16) || !aligned(y, 4)) return RQ_ERR_SHAPE;
  // the per-CTA sums of x must fit in shared memory
  if ((int64_t)M * K > 57344 * 8) return RQ_ERR_SHAPE;
  return RQ_OK;
}

rq_status rq_q4k_gemv(const void* w, const float* x, float* y, int M, int N, int K,
                      rq_stream_t stream) {
  rq_status s = check_gemv(w, x, y, M, N, K, 16);
  if (s != RQ_OK) return s;
  return launch_q4k_gemv(static_cast<const uint8_t*>(w), x, y, M, N, K,
                         reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_q6k_gemv(const void* w, const float* x, float* y, int M, int N, int K,
                      rq_stream_t stream) {
  rq_status s = check_gemv(w, x, y, M, N, K, 4);
  if (s != RQ_OK) return s;
  return launch_q6k_gemv(static_cast<const uint8_t*>(w), x, y, M, N, K,
                         reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_fp8_weight_cache(rq_ctx* ctx, rq_qtype qtype, const void* w, int N, int K,
                              const uint8_t** w_fp8, const float** w_dequant,
                              rq_stream_t stream) {
  if (ctx == nullptr || w == nullptr || w_fp8 == nullptr || w_dequant == nullptr)
    return RQ_ERR_NULL;
  rq_status s = check_quant_shape(qtype, N, K);
  if (s != RQ_OK) return s;
  if (!aligned(w, qtype == RQ_Q4K ? 16 : 4)) return RQ_ERR_SHAPE;
  const WeightKey key{w, (int)qtype, N, K};
  auto it = ctx->weights.find(key);
  if (it == ctx->weights.end()) {
    const size_t body = (size_t)N * (size_t)K;
    const size_t bytes = (body + 255) / 256 * 256 + 256;
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return RQ_ERR_ALLOC;
    }
    WeightEntry e;
    e.fp8 = static_cast<uint8_t*>(p);
    e.deq = reinterpret_cast<float*>(e.fp8 + (body + 255) / 256 * 256);
    e.bytes = bytes;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t* wb = static_cast<const uint8_t*>(w);
    s = cuda_status(cudaMemsetAsync(ctx->absmax, 0, sizeof(uint32_t), st));
    if (s == RQ_OK) s = launch_dequant_absmax(qtype, wb, N, K, ctx->absmax, st);
    if (s == RQ_OK)
      s = launch_dequant_encode(qtype, wb, N, K, ctx->absmax, e.fp8, e.deq, st);
    if (s != RQ_OK) {
      cudaFree(p);
      return s;
    }
    it = ctx->weights.emplace(key, e).first;
    ctx->weight_bytes += (int64_t)bytes;
  }
  *w_fp8 = it->second.fp8;
  *w_dequant = it->second.deq;
  return RQ_OK;
}

rq_status rq_fp8_gemm(const uint8_t* x_fp8, const float* x_dequant, const uint8_t* w_fp8,
                      const float* w_dequant, float* y, int M, int N, int K,
                      rq_stream_t stream) {
  if (x_fp8 == nullptr || x_dequant == nullptr || w_fp8 == nullptr ||
      w_dequant == nullptr || y == nullptr)
    return RQ_ERR_NULL;
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0) return RQ_ERR_SHAPE;
  if (!aligned(x_fp8, 16) || !aligned(w_fp8, 16) || !aligned(y, 4) ||
      !aligned(x_dequant, 4) || !aligned(w_dequant, 4))
    return RQ_ERR_SHAPE;
  return launch_fp8_gemm(x_fp8, x_dequant, w_fp8, w_dequant, y, M, N, K,
                         reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_fp8_act_cache(rq_ctx* ctx, const float* x, int M, int K,
                           const uint8_t** x_fp8, const float** x_dequant,
                           rq_stream_t stream) {
  if (ctx == nullptr || x == nullptr || x_fp8 == nullptr || x_dequant == nullptr)
    return RQ_ERR_NULL;
  if (M < 1 || K < 1 || !aligned(x, 16)) return RQ_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rq_status s = RQ_OK;
  const bool hit = ctx->act_valid && ctx->act_x == x && ctx->act_M == M &&
                   ctx->act_K == K && ctx->act_gen == ctx->gen;
  if (hit) {
    ++ctx->hits;
  } else {
    const int m_pad = (M + 15) / 16 * 16;
    const size_t need = (size_t)m_pad * (size_t)K;
    if (need > ctx->act_cap) {
      if (ctx->act) cudaFree(ctx->act);
      ctx->act = nullptr;
      ctx->act_cap = 0;
      ctx->act_valid = false;
      void* p = nullptr;
      if (cudaMalloc(&p, need) != cudaSuccess) {
        cudaGetLastError();
        return RQ_ERR_ALLOC;
      }
      ctx->act = static_cast<uint8_t*>(p);
      ctx->act_cap = need;
    }
    const int64_t n = (int64_t)M * K;
    s = RQ_ERR_SHAPE;
    if (n <= ctx->cluster_max) {
      // a few tokens: one cluster reads x twice (the second time from L2)
      TraceScope ts(ctx, RQ_TRACE_QUANT, st);
      s = launch_act_quant_cluster(x, n, (int64_t)need, ctx->act, ctx->absmax, ctx->act_deq, st);
      if (s == RQ_ERR_SHAPE) ts.kernels(0);
    } else if (ctx->fused_ok && n >= ctx->fused_min && act_quant_fused_fits(x, n, ctx->act)) {
      TraceScope ts(ctx, RQ_TRACE_QUANT, st);
      s = launch_act_quant_fused(x, n, (int64_t)need, ctx->act, ctx->absmax, ctx->act_deq,
                                 ctx->fused, ctx->fused_slots, device_sm_count(), st);
      if (s == RQ_ERR_SHAPE) ts.kernels(0);
    }
    // RQ_ERR_SHAPE from the one-cluster or one-pass launcher: nothing was
    // launched
    if (s == RQ_ERR_SHAPE) {
      // two kernels: per-CTA maxima into slots, then the encoding
      TraceScope ts(ctx, RQ_TRACE_QUANT, st);
      ts.kernels(2);
      s = launch_act_quant_two_pass(x, n, (int64_t)need, ctx->act, ctx->slots, ctx->absmax,
                                    ctx->act_deq, st);
    }
    if (s != RQ_OK) {
      ctx->act_valid = false;
      return s;
    }
    ctx->act_valid = true;
    ctx->act_x = x;
    ctx->act_M = M;
    ctx->act_K = K;
    ctx->act_gen = ctx->gen;
    ++ctx->misses;
  }
  *x_fp8 = ctx->act;
  *x_dequant = ctx->act_deq;
  return RQ_OK;
}

rq_status rq_linear(rq_ctx* ctx, rq_qtype qtype, const void* w, const float* x, float* y,
                    int M, int N, int K, rq_stream_t stream) {
  if (ctx == nullptr || w == nullptr || x == nullptr || y == nullptr) return RQ_ERR_NULL;
  rq_status s = check_quant_shape(qtype, N, K);
  if (s != RQ_OK) return s;
  if (M < 1) return RQ_ERR_SHAPE;
  if (!aligned(w, qtype == RQ_Q4K ? 16 : 4) || !aligned(x, 16) || !aligned(y, 4))
    return RQ_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  if (M < ctx->threshold) {
    // GEMV straight from the packed weight: Q4_K one launch per token, Q6_K
    // up to 8 tokens per launch
    const int per = qtype == RQ_Q4K ? 1 : 8;
    for (int m0 = 0; m0 < M; m0 += per) {
      const int mc = M - m0 < per ? M - m0 : per;
      TraceScope ts(ctx, RQ_TRACE_GEMV, st);
      s = qtype == RQ_Q4K
              ? rq_q4k_gemv(w, x + (size_t)m0 * K, y + (size_t)m0 * N, mc, N, K, stream)
              : rq_q6k_gemv(w, x + (size_t)m0 * K, y + (size_t)m0 * N, mc, N, K, stream);
      if (s != RQ_OK) return s;
    }
    return RQ_OK;
  }

  const uint8_t* wq = nullptr;
  const float* wdeq = nullptr;
  const bool miss = ctx->weights.find(WeightKey{w, (int)qtype, N, K}) == ctx->weights.end();
  {
    TraceScope ts(miss ? ctx : nullptr, RQ_TRACE_WCACHE, st);
    ts.kernels(2);  // decode + absmax, decode + encode
    s = rq_fp8_weight_cache(ctx, qtype, w, N, K, &wq, &wdeq, stream);
  }
  if (s != RQ_OK) return s;

  const uint8_t* xq = nullptr;
  const float* xdeq = nullptr;
  s = rq_fp8_act_cache(ctx, x, M, K, &xq, &xdeq, stream);
  if (s != RQ_OK) return s;
  TraceScope ts(ctx, RQ_TRACE_GEMM, st);
  // a cached weight built by an earlier call was complete before the launch
  // preceding this GEMM began, so its first tiles may load early
  return launch_fp8_gemm(xq, xdeq, wq, wdeq, y, M, N, K, st, !miss);
}

rq_status rq_linear_group(rq_ctx* ctx, int count, const rq_qtype* qtypes, const void* const* w,
                          const float* x, float* const* y, const int* N, int M, int K,
                          rq_stream_t stream) {
  if (ctx == nullptr || qtypes == nullptr || w == nullptr || x == nullptr || y == nullptr ||
      N == nullptr)
    return RQ_ERR_NULL;
  if (count < 1 || count > RQ_MAX_GROUP || M < 1) return RQ_ERR_SHAPE;
  for (int i = 0; i < count; ++i) {
    if (w[i] == nullptr || y[i] == nullptr) return RQ_ERR_NULL;
    rq_status s = check_quant_shape(qtypes[i], N[i], K);
    if (s != RQ_OK) return s;
    if (!aligned(w[i], qtypes[i] == RQ_Q4K ? 16 : 4) || !aligned(y[i], 4)) return RQ_ERR_SHAPE;
  }
  if (!aligned(x, 16)) return RQ_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (count == 1) return rq_linear(ctx, qtypes[0], w[0], x, y[0], M, N[0], K, stream);

  if (M < ctx->threshold) {
    // GEMV route, one token at a time: the Q4_K members in one launch,
    // joined by the Q6_K member when there is exactly one
    int starts[RQ_MAX_GROUP + 1];
    const uint8_t* ws[RQ_MAX_GROUP];
    int idx4[RQ_MAX_GROUP];
    int n4 = 0, i6 = -1, n6 = 0;
    starts[0] = 0;
    for (int i = 0; i < count; ++i) {
      if (qtypes[i] == RQ_Q4K) {
        ws[n4] = static_cast<const uint8_t*>(w[i]);
        idx4[n4] = i;
        starts[n4 + 1] = starts[n4] + N[i];
        ++n4;
      } else {
        i6 = i;
        ++n6;
      }
    }
    for (int m = 0; m < M; ++m) {
      const float* xm = x + (size_t)m * K;
      float* ys[RQ_MAX_GROUP];
      for (int j = 0; j < n4; ++j) ys[j] = y[idx4[j]] + (size_t)m * N[idx4[j]];
      bool grouped = false, dual = false;
      if (n4 >= 1 && n6 == 1 && std::getenv("RQ_GEMV_NO_DUAL") == nullptr) {
        TraceScope ts(ctx, RQ_TRACE_GEMV, st);
        const rq_status s = launch_gemv_m1_dual(n4, starts, ws, ys,
                                                static_cast<const uint8_t*>(w[i6]),
                                                y[i6] + (size_t)m * N[i6], N[i6], xm, K, st);
        if (s != RQ_OK && s != RQ_ERR_SHAPE) return s;
        grouped = dual = s == RQ_OK;
      }
      if (!grouped && n4 >= 2) {
        TraceScope ts(ctx, RQ_TRACE_GEMV, st);
        const rq_status s = launch_q4k_gemv_group(n4, starts, ws, ys, xm, K, st);
        if (s != RQ_OK && s != RQ_ERR_SHAPE) return s;
        grouped = s == RQ_OK;
      }
      for (int i = 0; i < count; ++i) {
        if (grouped && qtypes[i] == RQ_Q4K) continue;
        if (dual && i == i6) continue;
        const rq_status s =
            rq_linear(ctx, qtypes[i], w[i], xm, y[i] + (size_t)m * N[i], 1, N[i], K, stream);
        if (s != RQ_OK) return s;
      }
    }
    return RQ_OK;
  }

  // FP8 route: the group's weights, concatenated by rows, cached once
  std::vector<WeightKey> key;
  for (int i = 0; i < count; ++i) key.push_back(WeightKey{w[i], (int)qtypes[i], N[i], K});
  auto it = ctx->groups.find(key);
  const bool hit = it != ctx->groups.end();
  if (!hit) {
    GroupEntry e;
    e.starts[0] = 0;
    for (int i = 0; i < count; ++i) e.starts[i + 1] = e.starts[i] + N[i];
    for (int i = count; i < RQ_MAX_GROUP; ++i) e.starts[i + 1] = e.starts[count];
    const size_t body = (size_t)e.starts[count] * (size_t)K;
    const size_t bytes = (body + 255) / 256 * 256 + 256;
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return RQ_ERR_ALLOC;
    }
    e.fp8 = static_cast<uint8_t*>(p);
    e.deq = reinterpret_cast<float*>(e.fp8 + (body + 255) / 256 * 256);
    e.bytes = bytes;
    rq_status s = RQ_OK;
    {
      TraceScope ts(ctx, RQ_TRACE_WCACHE, st);
      ts.kernels(2 * count);
      for (int i = 0; i < count && s == RQ_OK; ++i) {
        const uint8_t* wb = static_cast<const uint8_t*>(w[i]);
        s = cuda_status(cudaMemsetAsync(ctx->absmax, 0, sizeof(uint32_t), st));
        if (s == RQ_OK) s = launch_dequant_absmax(qtypes[i], wb, N[i], K, ctx->absmax, st);
        if (s == RQ_OK)
          s = launch_dequant_encode(qtypes[i], wb, N[i], K, ctx->absmax,
                                    e.fp8 + (size_t)e.starts[i] * K, e.deq + i, st);
      }
    }
    if (s != RQ_OK) {
      cudaFree(p);
      return s;
    }
    it = ctx->groups.emplace(key, e).first;
    ctx->weight_bytes += (int64_t)bytes;
  }
  const uint8_t* xq = nullptr;
  const float* xdeq = nullptr;
  rq_status s = rq_fp8_act_cache(ctx, x, M, K, &xq, &xdeq, stream);
  if (s != RQ_OK) return s;
  const float* deqs[RQ_MAX_GROUP];
  for (int i = 0; i < count; ++i) deqs[i] = it->second.deq + i;
  TraceScope ts(ctx, RQ_TRACE_GEMM, st);
  // a group cache built by an earlier call may be loaded early (as in rq_linear)
  return launch_fp8_gemm_group(xq, xdeq, it->second.fp8, count, it->second.starts, y, deqs, M,
                               K, st, hit);
}

rq_status rq_ctx_trace_begin(rq_ctx* ctx, int capacity) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  if (capacity < 1) return RQ_ERR_SHAPE;
  while ((int)ctx->trace.size() < capacity) {
    TraceSlot t;
    if (cudaEventCreate(&t.start) != cudaSuccess) return RQ_ERR_ALLOC;
    if (cudaEventCreate(&t.stop) != cudaSuccess) {
      cudaEventDestroy(t.start);
      return RQ_ERR_ALLOC;
    }
    ctx->trace.push_back(t);
  }
  ctx->trace_cap = capacity;
  ctx->trace_used = 0;
  ctx->trace_on = true;
  return RQ_OK;
}

rq_status rq_ctx_trace_kinds(rq_ctx* ctx, unsigned int mask) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  if (mask == 0u || (mask >> RQ_TRACE_KINDS) != 0u) return RQ_ERR_SHAPE;
  ctx->trace_mask = mask;
  return RQ_OK;
}

rq_status rq_ctx_trace_end(rq_ctx* ctx, int64_t* counts_host, double* ms_host) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  int64_t counts[RQ_TRACE_KINDS] = {0};
  double ms[RQ_TRACE_KINDS] = {0.0};
  rq_status s = RQ_OK;
  for (int i = 0; i < ctx->trace_used; ++i) {
    const TraceSlot& t = ctx->trace[i];
    float e = 0.f;
    if (cudaEventSynchronize(t.stop) != cudaSuccess ||
        cudaEventElapsedTime(&e, t.start, t.stop) != cudaSuccess) {
      s = RQ_ERR_CUDA;
      continue;
    }
    counts[t.kind] += t.kernels;
    ms[t.kind] += e;
  }
  ctx->trace_on = false;
  ctx->trace_used = 0;
  for (int k = 0; k < RQ_TRACE_KINDS; ++k) {
    if (counts_host) counts_host[k] = counts[k];
    if (ms_host) ms_host[k] = ms[k];
  }
  return s;
}

rq_status rq_act_cache_invalidate(rq_ctx* ctx) {
  if (ctx == nullptr) return RQ_ERR_NULL;
  ++ctx->gen;
  ctx->act_valid = false;
  return RQ_OK;
}

rq_status rq_get_device_status(rq_stream_t stream) {
  return read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_debug_wait_timeout(int64_t limit_ns, rq_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 10000000000LL) return RQ_ERR_SHAPE;
  return launch_debug_wait_timeout(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

rq_status rq_gemv_exact_outputs(rq_stream_t stream, int64_t* count_host) {
  if (count_host == nullptr) return RQ_ERR_NULL;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return RQ_ERR_CUDA;
  return read_and_clear_gemv_exact_outputs(count_host);
}

}  // extern "C"
