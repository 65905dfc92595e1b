/*
 * rq.h -- C ABI of librq.so, the quantized linear layer for GB300 (sm_103a).
 *
 * The operations follow the three source pages of realizar 0.8.4 (docs.rs):
 *   [gemm.rs]  src/cuda/executor/layers/cublas_prefill/gemm.rs
 *   [mod.rs]   src/cuda/executor/layers/cublas_prefill/mod.rs
 *   [q6k.rs]   src/cuda/executor/q6k_gemv_indexed.rs
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors) unless
 *    the name ends in _host.  The caller owns every pointer it passes in.
 *  - `stream` is a cudaStream_t (0 = legacy default stream).  Every call is
 *    asynchronous and stream-ordered: nothing synchronises the host, except
 *    rq_get_device_status and allocations on a cache miss (documented below).
 *  - Arguments are validated on the host before anything is launched; on a
 *    validation error nothing is launched or written and the status says why.
 *    A failed launch returns RQ_ERR_CUDA.  No entry point traps or aborts.
 *  - Matrices are row-major and densely packed (row stride = row length).
 *  - Shapes: M = tokens (rows of x and y), N = output features (weight rows),
 *    K = input features.  Quantized weights need K % 256 == 0.
 *  - Not thread-safe per rq_ctx: one thread and one stream at a time per ctx.
 *  - One CUDA device per process (one process per GPU): a kernel's
 *    shared-memory and cluster-size opt-ins are made once, on the device
 *    current at its first launch, and reused.
 */
#ifndef RQ_H
#define RQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RQ_ABI_VERSION 1

typedef enum {
    RQ_OK = 0,
    RQ_ERR_NULL = 1,       /* a required pointer is NULL                      */
    RQ_ERR_SHAPE = 2,      /* a size is out of range or misaligned            */
    RQ_ERR_QTYPE = 3,      /* unsupported weight quantization type            */
    RQ_ERR_NOT_CACHED = 4, /* reserved: a weight has no FP8 cache entry       */
    RQ_ERR_ALLOC = 5,      /* device or host allocation failed                */
    RQ_ERR_CUDA = 6,       /* a CUDA call or kernel launch failed             */
    RQ_ERR_TIMEOUT = 7,    /* a kernel gave up on a pipeline wait (see below) */
    RQ_ERR_ARCH = 8        /* device lacks sm_103 features (tcgen05, TMA)     */
} rq_status;

/* GGUF tensor type ids. */
typedef enum { RQ_Q4K = 12, RQ_Q6K = 14 } rq_qtype;

/* ABI-identical to cudaStream_t. */
typedef struct CUstream_st *rq_stream_t;

/* Opaque context: owns the FP8 weight cache, the activation FP8 scratch and
 * the device scalars of the prefill path. */
typedef struct rq_ctx rq_ctx;

int rq_abi_version(void);
const char *rq_status_string(rq_status s);

/* ------------------------------------------------------------ context -- */

/* Create a context on the current CUDA device.  Default GEMM threshold 4,
 * or the value of the environment variable RQ_GEMM_THRESHOLD (read once,
 * here), mirroring [mod.rs] cublas_gemm_threshold.
 * Errors: RQ_ERR_NULL (out == NULL), RQ_ERR_ALLOC. */
rq_status rq_ctx_create(rq_ctx **out);

/* Free every buffer the context owns (FP8 weights, scratch, scalars).  The
 * caller must make sure no work using them is still in flight.  NULL is a
 * no-op. */
void rq_ctx_destroy(rq_ctx *ctx);

/* M at or above the threshold goes to the FP8 GEMM, below it to the GEMV
 * ([mod.rs], cublas_gemm_threshold: "Minimum M ... to use GEMM instead of
 * batched GEMV", default 4).  Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (< 1). */
rq_status rq_ctx_set_gemm_threshold(rq_ctx *ctx, int m_threshold);
int rq_ctx_get_gemm_threshold(const rq_ctx *ctx);

/* Host-side counters: activation-cache hits and misses of rq_linear, number
 * of cached FP8 weights and the device bytes they hold.  Any out pointer may
 * be NULL.  Errors: RQ_ERR_NULL (ctx). */
rq_status rq_ctx_get_stats(const rq_ctx *ctx, int64_t *act_hits_host,
                           int64_t *act_misses_host, int64_t *weights_host,
                           int64_t *weight_bytes_host);

/* ---------------------------------------------------- absmax + E4M3 ---- */

/* Per-tensor absmax ([mod.rs], ABSMAX_REDUCE_PTX and gpu_absmax_device):
 * *absmax_bits = IEEE bits of max_i |x[i]| over the n floats of x, starting
 * from +0; NaNs are skipped, +-Inf count as +Inf.  The word is zeroed on
 * `stream` first (no host copy from a stack temporary), then reduced with an
 * unsigned atomic max, which orders non-negative floats correctly.
 *   x: n floats (any alignment).  absmax_bits: one device word (4-aligned).
 * Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (n < 0).  n == 0 yields 0. */
rq_status rq_absmax(const float *x, int64_t n, uint32_t *absmax_bits,
                    rq_stream_t stream);

/* Scaled FP32 -> E4M3 ([mod.rs], F32_TO_E4M3_DEVICE_SCALED_PTX): reads the
 * absmax word A from the device, uses A' = (A == 0 ? 1 : A), s = 448 / A'
 * (correctly rounded fp32 division), writes out[i] = E4M3(fl32(x[i] * s)) and
 * *dequant_out = A' / 448.  Encoder rules: exponent rebias 127 -> 7, mantissa
 * round-to-nearest-even 23 -> 3 bits, values below 2^-6 flush to 0x00,
 * overflow saturates to sign|0x7E (+-448), 0x7F/0xFF are never produced,
 * NaN/Inf inputs give sign(x)|0x7E and +-0 gives 0x00 (decided before the
 * multiply).  Bit-exact with the CPU reference.
 *   x: n floats.  out: n bytes.  dequant_out: one device float.
 * Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (n < 0). */
rq_status rq_quant_e4m3(const float *x, int64_t n, const uint32_t *absmax_bits,
                        uint8_t *out, float *dequant_out, rq_stream_t stream);

/* ------------------------------------------------------------- GEMV ---- */

/* Decode GEMV on GGUF Q4_K weights, dequantized inside the dot product
 * ([q6k.rs], q4k_gemv_into; [mod.rs] cublas_gemm_threshold doc: batched GEMV
 * for small M reads Q4_K directly at 0.5625 B/weight):
 *   y[m, n] = sum_k x[m, k] * w(n, k),  0 <= m < M, 0 <= n < N.
 *   w: N rows of K/256 Q4_K super-blocks, 144 B each (fp16 d, fp16 dmin,
 *      12 packed 6-bit scale/min bytes, 128 bytes of 4-bit quants), rows
 *      contiguous; 16-byte aligned.
 *   x: f32 [M x K], 16-byte aligned.  y: f32 [M x N] (written, not added to).
 * Accuracy: for finite x, every output whose sum_k |x[m,k] * w(n,k)| is at
 * least 2^-100 is within 1e-4 * sum_k |x[m,k] * w(n,k)| of the exact result
 * (outputs beyond fp32's range are +-Inf; non-finite x give Inf / NaN as in
 * IEEE arithmetic).  The fast paths prove this per output with an error
 * certificate computed alongside the sum; an output whose certificate fails
 * (extreme ranges of x within 32 values, weights whose two terms cancel on
 * the largest x) is recomputed exactly in fp64 inside the same launch, which
 * is slow but never wrong (see rq_gemv_exact_outputs).  Several tokens run
 * one launch per token (the weight is read once per token).
 * Ordering: the kernel may start streaming w before the kernel launched just
 * before it on the stream has finished (programmatic dependent launch); it
 * reads x and writes y only after that kernel has completed.  So w must not
 * be written by the immediately preceding kernel on the stream (a copy or
 * any earlier kernel is fine).  The same holds for rq_q6k_gemv and for the
 * GEMV route of rq_linear.
 * Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (M not in 1..8, N < 1, K < 256,
 * K % 256 != 0, misaligned w or x). */
rq_status rq_q4k_gemv(const void *w, const float *x, float *y, int M, int N,
                      int K, rq_stream_t stream);

/* The same on GGUF Q6_K weights ([q6k.rs], q6k_gemv_indexed_async, which
 * returns InvalidLaunchConfig for a null weight pointer; here the output is
 * caller-owned, nothing is allocated):
 *   w: N rows of K/256 Q6_K super-blocks, 210 B each (ql[128], qh[64],
 *      16 int8 scales, fp16 d), rows contiguous; 4-byte aligned.
 *   weight = d * scale * (q - 32), q the 6-bit quant.
 * Accuracy as rq_q4k_gemv (certificate per output, exact fp64 path when it
 * fails); 2..8 tokens are one launch.
 * Errors: as rq_q4k_gemv (w need only be 4-byte aligned). */
rq_status rq_q6k_gemv(const void *w, const float *x, float *y, int M, int N,
                      int K, rq_stream_t stream);

/* ------------------------------------------------------- FP8 prefill --- */

/* FP8 weight cache ([gemm.rs], get_or_cache_fp8_weight): on the first call
 * for (w, qtype, N, K) the packed weight is dequantized to fp32 in the fixed
 * order w = (d*sc)*q - dmin*m (Q4_K) or (d*scale)*(q-32) (Q6_K), its absmax
 * A_w is taken, and every weight is encoded as in rq_quant_e4m3 with
 * 448 / A_w'.  Unlike the pages, the dequant scale A_w'/448 stays in device
 * memory (no host read-back, no host sync); no fp32 scratch is used (the
 * weight is decoded twice instead).  Later calls return the cached pointers.
 *   *w_fp8: device E4M3 bytes [N x K] owned by ctx, valid until
 *           rq_ctx_destroy.  *w_dequant: one device float owned by ctx.
 * A miss allocates with cudaMalloc (which may synchronise the device).
 * Errors: RQ_ERR_NULL, RQ_ERR_QTYPE, RQ_ERR_SHAPE, RQ_ERR_ALLOC. */
rq_status rq_fp8_weight_cache(rq_ctx *ctx, rq_qtype qtype, const void *w,
                              int N, int K, const uint8_t **w_fp8,
                              const float **w_dequant, rq_stream_t stream);

/* FP8 E4M3 GEMM with a fused fp32 epilogue ([gemm.rs],
 * cublas_prefill_fp8_gemm: raw FP8 products, then the activation scale
 * act_absmax/448 and the weight scale w_absmax/448, both read from device
 * memory, with no host sync):
 *   y[m, n] = (sum_k e4m3(x_fp8[m, k]) * e4m3(w_fp8[n, k]))
 *             * (*x_dequant) * (*w_dequant)            for m < M, n < N.
 * Tensor cores (tcgen05 kind::f8f6f4), fp32 accumulation; agrees with the
 * exact reference within 2e-3*|ref| + 1e-3*rms(row of ref).
 *   x_fp8: E4M3 [M_pad x K], M_pad = (M + 15) / 16 * 16; rows M..M_pad-1
 *          are read but do not affect y.  16-byte aligned.
 *   w_fp8: E4M3 [N x K], 16-byte aligned.   y: f32 [M x N]; rows >= M and
 *          columns >= N are never written.
 * Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (M, N < 1, K < 128, K % 128 != 0,
 * misaligned operands), RQ_ERR_CUDA. */
rq_status rq_fp8_gemm(const uint8_t *x_fp8, const float *x_dequant,
                      const uint8_t *w_fp8, const float *w_dequant, float *y,
                      int M, int N, int K, rq_stream_t stream);

/* FP8 activation cache ([gemm.rs], cublas_prefill_fp8_gemm: the
 * activation's per-tensor absmax and E4M3 conversion, and the PMAT-084
 * reuse of that FP8 copy by the next linears that read the same input):
 * returns device pointers to the E4M3 form of x and its dequant scale
 * absmax'/448 (absmax' = absmax, or 1 for an all-zero x), quantizing x into
 * the ctx's scratch on a miss.  The bytes are those of rq_absmax followed by
 * rq_quant_e4m3, with rows M..M_pad-1 zero (M_pad = M rounded up to 16), so
 * the result feeds rq_fp8_gemm directly.  The key is (x, M, K, generation),
 * as for rq_linear, which calls this on its FP8 route.
 *   x: f32 [M x K], 16-byte aligned.   *x_fp8: E4M3 [M_pad x K] (owned by
 *   ctx).   *x_dequant: one device float (owned by ctx).
 * The pointers stay valid until a later miss on this ctx needs a larger
 * scratch, or the ctx is destroyed; a later miss of the same or smaller size
 * overwrites the bytes in stream order.  Allocates on a miss that needs a
 * larger scratch.  Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (M, K < 1, x
 * misaligned), RQ_ERR_ALLOC, RQ_ERR_CUDA. */
rq_status rq_fp8_act_cache(rq_ctx *ctx, const float *x, int M, int K,
                           const uint8_t **x_fp8, const float **x_dequant,
                           rq_stream_t stream);

/* Quantized linear layer with M-threshold routing ([mod.rs],
 * cublas_gemm_threshold; [gemm.rs], cublas_prefill_gemm FP8 branch):
 *   M <  threshold: Q4_K / Q6_K GEMV straight from the packed weights
 *                   (M > 8 is processed 8 rows at a time);
 *   M >= threshold: FP8 weight cache (a hit after the first call), then, on
 *                   an activation-cache miss, absmax + E4M3 quantization of
 *                   x into the ctx's [M_pad x K] scratch (pad rows zeroed),
 *                   then the FP8 GEMM.  Up to 2^17 elements, absmax and
 *                   quantization are one launch of one thread-block
 *                   cluster (x read twice, the second time from L2); from
 *                   2^20 elements on, one cooperative kernel while x fits
 *                   on chip in one wave of CTAs (per SM 512 x 24 float4
 *                   in registers plus about 220 KB of shared memory: x
 *                   read once) or, with x held in shared memory, while
 *                   what does not fit is at most 16 MB (128 MB from 2^24
 *                   elements on; only that rest read twice); otherwise
 *                   two kernels, the second reading x backwards (the same
 *                   bytes every way; at ctx creation the environment
 *                   variables RQ_CLUSTER_QUANT_MAX (elements, 0 = never)
 *                   and RQ_ONE_PASS_QUANT=0 turn the first two off).
 * The activation cache ([gemm.rs], PMAT-084 reuse across Q/K/V and gate/up)
 * is keyed by (x, M, K, generation); rq_act_cache_invalidate bumps the
 * generation and must be called when x's contents change in place.
 * Errors: those of the routes taken. */
rq_status rq_linear(rq_ctx *ctx, rq_qtype qtype, const void *w, const float *x,
                    float *y, int M, int N, int K, rq_stream_t stream);

/* Linear layers that share one input ([gemm.rs], PMAT-084: Q, K and V read
 * the same activation, and so do gate and up):
 *   y_i = x . W_i^T   for i < count,  W_i: N_i rows of qtypes[i] super-blocks.
 * Routes like rq_linear.  On the FP8 route the activation is quantized once
 * (activation cache) and the group is one GEMM launch over the members'
 * FP8 weights, cached once per group contiguously by rows (member i keeps
 * its own per-tensor scale; its bytes equal rq_fp8_weight_cache's).  On
 * the GEMV route the Q4_K members are one launch (one pass of x) for up to
 * 8 tokens; for a single token the group's Q6_K member joins that launch
 * when it has exactly one (the CTAs split between the two formats); other
 * members are launched one by one.  Results are those of count rq_linear calls within the same
 * tolerances.
 *   count: 1 .. RQ_MAX_GROUP.  qtypes, w, y, N: host arrays of count
 *   entries (w[i], y[i] device pointers as for rq_linear).  All members
 *   share x (f32 [M x K], 16-byte aligned), M and K.
 * The group's FP8 weights are owned by ctx (keyed by the members' pointers,
 * types and shapes) and freed by rq_ctx_destroy.
 * Errors: RQ_ERR_NULL, RQ_ERR_QTYPE, RQ_ERR_SHAPE (count out of range, or
 * as rq_linear), RQ_ERR_ALLOC, RQ_ERR_CUDA. */
#define RQ_MAX_GROUP 4
rq_status rq_linear_group(rq_ctx *ctx, int count, const rq_qtype *qtypes,
                          const void *const *w, const float *x, float *const *y,
                          const int *N, int M, int K, rq_stream_t stream);

/* FP8 linear layer that allocates nothing.  The source pages have no
 * counterpart to this entry point.
 *
 * For callers that cannot call cudaMalloc while serving: code that runs
 * inside a host framework which owns and pre-reserves all device memory (an
 * inference engine's plugin or operator callback, say), or a process under a
 * fixed device-memory budget where a new allocation would fail or stall.
 * Given an E4M3 weight and its dequant scale (for example the pointers
 * rq_fp8_weight_cache returns), it computes the same result as the FP8 route
 * of rq_linear: absmax of x, E4M3 quantization of x, FP8 GEMM with both
 * scales applied to the fp32 accumulator:
 *   y[m, n] = (sum_k e4m3(xq[m, k]) * e4m3(w_fp8[n, k])) * x_deq * (*w_dequant)
 *   x: f32 [M x K], 16-byte aligned.  w_fp8: E4M3 [N x K], 16-byte aligned.
 *   w_dequant: one device float.  y: f32 [M x N].
 * The quantized activation (M_pad x K bytes, M_pad = M rounded up to 16) and
 * two device scalars live in one fixed array inside the library, of
 * RQ_NOALLOC_MAX_ACT_BYTES + 256 bytes, which the GPU holds until the process
 * exits.  No call allocates: no cudaMalloc, cudaFree or allocating library
 * routine.
 *   - The first call looks up the array's device address (with the device
 *     current).  Under CUDA's lazy module loading that lookup may also be
 *     what loads the library's module and reserves the array, so the first
 *     call may take device memory once: make it a warm-up call before
 *     serving or any stream capture, and before fixing a memory budget.
 *   - The library serves one device per process (see the conventions at
 *     the top).  All calls share the array, and it keeps the last call's
 *     contents; each call re-zeroes what must start at zero.  Calls whose
 *     work overlaps on the GPU (on two streams, say) race on the array:
 *     serialise them.
 * Errors: RQ_ERR_NULL; RQ_ERR_SHAPE for M, N < 1, K < 128, K % 128 != 0,
 * misaligned pointers, or M_pad * K > RQ_NOALLOC_MAX_ACT_BYTES (the array
 * is too small for this activation); RQ_ERR_CUDA. */
#define RQ_NOALLOC_MAX_ACT_BYTES (8u * 1024u * 1024u)
rq_status rq_fp8_linear_noalloc(const float *x, const uint8_t *w_fp8,
                                const float *w_dequant, float *y, int M, int N,
                                int K, rq_stream_t stream);

/* Forget the cached FP8 activation (bump the generation). */
rq_status rq_act_cache_invalidate(rq_ctx *ctx);

/* ----------------------------------------------------------- tracing --- */

/* Kernel-level tracing of rq_linear, the device-side counterpart of the
 * pages' PREFILL_DETAIL_TRACE phases ([gemm.rs], cublas_prefill_fp8_gemm:
 * absmax+convert / gemm / convert) without their host synchronisations:
 * while tracing is on, every kernel rq_linear launches is bracketed by two
 * CUDA events recorded on the call's stream (as external event nodes when the
 * stream is being captured).  Kinds: */
typedef enum {
    RQ_TRACE_GEMV = 0,    /* Q4_K / Q6_K GEMV                         */
    RQ_TRACE_ABSMAX = 1,  /* (not emitted by rq_linear, which traces the
                             activation's absmax and encoding together
                             as RQ_TRACE_QUANT)                       */
    RQ_TRACE_QUANT = 2,   /* activation absmax + E4M3 quantization    */
    RQ_TRACE_GEMM = 3,    /* FP8 GEMM                                 */
    RQ_TRACE_WCACHE = 4,  /* FP8 weight-cache build (a miss)          */
    RQ_TRACE_KINDS = 5
} rq_trace_kind;

/* Start tracing with room for `capacity` kernels (events are created here,
 * reused across begin/end pairs).  Kernels beyond the capacity are not
 * traced.  Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (capacity < 1),
 * RQ_ERR_ALLOC. */
rq_status rq_ctx_trace_begin(rq_ctx *ctx, int capacity);

/* Restrict tracing to the kinds whose bit (1 << kind) is set in `mask`
 * (all kinds by default): the events of a traced kernel keep it from
 * overlapping its neighbours (programmatic dependent launch), so a caller
 * timing a whole pass traces only the kernels it needs.  Takes effect for
 * kernels launched after the call.  Errors: RQ_ERR_NULL, RQ_ERR_SHAPE (mask
 * 0 or with bits at or above RQ_TRACE_KINDS). */
rq_status rq_ctx_trace_kinds(rq_ctx *ctx, unsigned int mask);

/* Stop tracing, wait for the traced events, and return per kind the number
 * of kernels and their summed device time in milliseconds (arrays of
 * RQ_TRACE_KINDS host entries; either may be NULL).  Errors: RQ_ERR_NULL,
 * RQ_ERR_CUDA. */
rq_status rq_ctx_trace_end(rq_ctx *ctx, int64_t *counts_host, double *ms_host);

/* Synchronise `stream`, then report and clear the library's device error
 * word: RQ_ERR_TIMEOUT if a GEMM or GEMV pipeline wait, or the one-pass
 * quantization's grid barrier, exceeded its time limit (the kernel then
 * stopped early and its output is incomplete), RQ_ERR_CUDA if
 * the synchronisation itself failed, RQ_OK otherwise. */
rq_status rq_get_device_status(rq_stream_t stream);

/* Test hook for the timeout path: launches one block that waits on an
 * mbarrier nothing will ever complete, with a wait limit of `limit_ns`
 * nanoseconds, and records a timeout exactly like the GEMM would.  The
 * caller then reads it with rq_get_device_status.  Errors: RQ_ERR_SHAPE
 * (limit_ns outside 1 .. 10^10), RQ_ERR_CUDA. */
rq_status rq_debug_wait_timeout(int64_t limit_ns, rq_stream_t stream);

/* Diagnostics of the GEMVs' accuracy guarantee (rq_q4k_gemv): synchronise
 * `stream`, then return in *count_host the number of GEMV outputs (one per
 * token and row) that were recomputed on the exact fp64 path since the last
 * call, and reset the count.  The count is per process and device; kernels
 * still running on other streams may or may not be included.
 * Errors: RQ_ERR_NULL, RQ_ERR_CUDA. */
rq_status rq_gemv_exact_outputs(rq_stream_t stream, int64_t *count_host);

#ifdef __cplusplus
}
#endif

#endif /* RQ_H */
