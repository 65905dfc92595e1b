/*
 * oracle.c -- plain, slow CPU oracle for the quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library and its Python binding) never links, imports or calls it, and
 * shares no code, header, table or constant generator with it.
 *
 * Source pages (realizar 0.8.4, docs.rs source view):
 *   [gemm.rs]  src/cuda/executor/layers/cublas_prefill/gemm.rs
 *   [mod.rs]   src/cuda/executor/layers/cublas_prefill/mod.rs
 *   [q6k.rs]   src/cuda/executor/q6k_gemv_indexed.rs
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math), so
 * every float operation below is a single IEEE-754 round-to-nearest-even
 * operation with subnormals preserved.
 *
 * Parity pins: every exported function is pinned by CPU tests against facts
 * the pages or the mathematics fix (closed forms, exhaustive code tables,
 * hand-built blocks, brute force on tiny inputs, library routines).  None is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_Q4K 12 /* GGUF type id of Q4_K */
#define ORC_Q6K 14 /* GGUF type id of Q6_K */
#define ORC_QK 256 /* weights per super-block */
#define ORC_Q4K_BYTES 144
#define ORC_Q6K_BYTES 210

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ------------------------------------------------------------------------ */
/* E4M3                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Value of one E4M3 byte: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits ([mod.rs], doc comment of F32_TO_E4M3_PTX: "sign(1) + exponent(4) +
 * mantissa(3), bias=7, range +-448").  Exponent field 0 is the subnormal range
 * 2^-6 * m/8.  Codes 0x7F / 0xFF are NaN in the OCP E4M3FN format; this
 * decoder returns NaN for them (the encoder never produces them).
 */
double orc_e4m3_decode(uint8_t b)
{
    int s = b >> 7;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/*
 * Unscaled FP32 -> E4M3 encoder ([mod.rs], F32_TO_E4M3_PTX and its doc
 * comment), steps in the pages' order:
 *   fp32 exponent field 0 (zero or fp32 subnormal)   -> 0x00 (sign dropped)
 *   fp32 exponent field 255 (NaN or +-Inf)           -> sign | 0x7E
 *   rebias the exponent 127 -> 7 (subtract 120)
 *   rebiased exponent < 1, i.e. |v| < 2^-6           -> 0x00 (no E4M3 subnormals)
 *   rebiased exponent > 15                           -> sign | 0x7E
 *   keep the top 3 mantissa bits, round to nearest even on bit 19 with the
 *   19 bits below it as sticky; a carry out of the mantissa bumps the exponent
 *   and can overflow to sign | 0x7E
 *   pack sign | exponent | mantissa
 * One deliberate deviation from the pages: the code for exponent 15 and
 * mantissa 7 (0x7F / 0xFF, NaN in E4M3FN) is never emitted; the saturated
 * value sign | 0x7E (+-448) is emitted instead.
 */
uint8_t orc_e4m3_encode(float v)
{
    const uint32_t bits = f2u(v);
    const uint32_t sign = bits >> 31;
    const uint32_t e32 = (bits >> 23) & 0xFFu;
    const uint32_t man = bits & 0x7FFFFFu;
    const uint8_t saturated = (uint8_t)((sign << 7) | 0x7Eu);
    int e;
    uint32_t top, round_bit, sticky;

    if (e32 == 0) return 0x00;
    if (e32 == 255) return saturated;
    e = (int)e32 - 120;
    if (e < 1) return 0x00;
    if (e > 15) return saturated;

    top = man >> 20;
    round_bit = (man >> 19) & 1u;
    sticky = man & 0x7FFFFu;
    if (round_bit && (sticky != 0 || (top & 1u) != 0)) top += 1;
    if (top == 8) {
        top = 0;
        e += 1;
        if (e > 15) return saturated;
    }
    if (e == 15 && top == 7) return saturated; /* never 0x7F / 0xFF */
    return (uint8_t)((sign << 7) | ((uint32_t)e << 3) | top);
}

/*
 * Per-tensor absmax ([mod.rs], ABSMAX_REDUCE_PTX): the maximum of |x_i|
 * starting from +0.  NaN inputs are skipped (a max with a NaN operand keeps the
 * other operand), +-Inf count as +Inf, -0 counts as +0.  The result is returned
 * as the IEEE-754 bits of a non-negative float, the form the device keeps it in.
 */
uint32_t orc_absmax_bits(const float *x, int64_t n)
{
    float best = 0.0f;
    int64_t i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (isnan(a)) continue;
        if (a > best) best = a;
    }
    return f2u(best);
}

/*
 * Quantization scale and dequantization scale for a tensor with the given
 * absmax ([mod.rs], F32_TO_E4M3_DEVICE_SCALED_PTX; [gemm.rs],
 * get_or_cache_fp8_weight): an absmax of zero is replaced by 1, then
 * quant = 448 / absmax and dequant = absmax / 448, each one correctly rounded
 * fp32 division.
 */
void orc_scales(uint32_t absmax_bits, float *quant_scale, float *dequant_scale)
{
    float a = u2f(absmax_bits);
    if (a == 0.0f) a = 1.0f;
    if (quant_scale) *quant_scale = 448.0f / a;
    if (dequant_scale) *dequant_scale = a / 448.0f;
}

/*
 * Scaled encoder for one element with quantization scale s
 * ([mod.rs], F32_TO_E4M3_SCALED_PTX / _DEVICE_SCALED_PTX: one fp32 multiply,
 * then the unscaled encoder).  Two readings where the pages are silent:
 *   - a non-finite input (NaN or +-Inf) keeps its own sign: sign(x) | 0x7E,
 *     decided before scaling, as the unscaled encoder does for such values
 *     (so the result never depends on how a multiply makes or signs a NaN,
 *     e.g. Inf * 0 when the absmax itself was Inf);
 *   - an input of +-0 gives 0x00 before scaling (0 * Inf would be NaN when the
 *     scale overflowed).
 */
uint8_t orc_encode_scaled(float x, float s)
{
    const uint32_t bits = f2u(x);
    if (isnan(x) || isinf(x)) return (uint8_t)(((bits >> 31) << 7) | 0x7Eu);
    if (x == 0.0f) return 0x00;
    return orc_e4m3_encode(x * s);
}

/*
 * Activation quantization ([gemm.rs], cublas_prefill_fp8_gemm steps 1+2):
 * out[i] = scaled-encode(x[i]) with s = 448 / absmax'.  Writes n bytes and the
 * dequant scale absmax'/448.
 */
void orc_quant_e4m3(const float *x, int64_t n, uint32_t absmax_bits,
                    uint8_t *out, float *dequant_scale)
{
    float s, deq;
    int64_t i;
    orc_scales(absmax_bits, &s, &deq);
    for (i = 0; i < n; ++i) out[i] = orc_encode_scaled(x[i], s);
    if (dequant_scale) *dequant_scale = deq;
}

/* ------------------------------------------------------------------------ */
/* GGUF super-blocks                                                         */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 -> binary32, written out from the format definition. */
float orc_half_to_float(uint16_t h)
{
    uint32_t s = (uint32_t)(h >> 15);
    int e = (h >> 10) & 31;
    uint32_t m = h & 1023u;
    float mag;
    if (e == 31) {
        mag = m ? NAN : INFINITY;
    } else if (e == 0) {
        mag = ldexpf((float)m, -24); /* subnormal: m * 2^-24, exact */
    } else {
        mag = ldexpf(1.0f + (float)m / 1024.0f, e - 15); /* exact */
    }
    return s ? -mag : mag;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/*
 * 6-bit scale and min of sub-block j (0..7) of a Q4_K super-block, from its
 * 12 packed bytes (GGML get_scale_min_k4 packing): the first four sub-blocks
 * use the low 6 bits of bytes j and j+4; the last four take their low 4 bits
 * from the nibbles of byte j+4 and their top 2 bits from the top bits of bytes
 * j-4 (scale) and j (min).
 */
void orc_q4k_scale_min(const uint8_t *scales, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *mn = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *mn = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* Quant (0..15) and sub-block index of weight i (0..255) of a Q4_K block. */
static void q4k_quant(const uint8_t *qs, int i, int *q, int *j)
{
    int chunk = i / 64, pos = i % 64;
    if (pos < 32) {
        *q = qs[32 * chunk + pos] & 15;
        *j = 2 * chunk;
    } else {
        *q = qs[32 * chunk + pos - 32] >> 4;
        *j = 2 * chunk + 1;
    }
}

/*
 * Q4_K super-block (144 bytes per 256 weights, [gemm.rs] doc comments of the
 * Q4_K GEMM launches): fp16 d, fp16 dmin, 12 packed scale/min bytes, 128 bytes
 * of 4-bit quants.  Weight = d * sc_j * q - dmin * m_j.
 *
 * fp32 evaluation order (the pages are silent; this order is the one the FP8
 * weight cache must reproduce bit for bit): w = (d*sc)*q - dmin*m, each
 * product and the difference a single correctly rounded fp32 operation.
 */
void orc_q4k_decode_block(const uint8_t *blk, float *w)
{
    const float d = orc_half_to_float(rd16(blk));
    const float dmin = orc_half_to_float(rd16(blk + 2));
    const uint8_t *scales = blk + 4, *qs = blk + 16;
    int i;
    for (i = 0; i < ORC_QK; ++i) {
        int q, j, sc, mn;
        float dsc, term, off;
        q4k_quant(qs, i, &q, &j);
        orc_q4k_scale_min(scales, j, &sc, &mn);
        dsc = d * (float)sc;
        term = dsc * (float)q;
        off = dmin * (float)mn;
        w[i] = term - off;
    }
}

/* The same weights evaluated exactly in fp64 (the mathematical definition). */
void orc_q4k_decode_block_f64(const uint8_t *blk, double *w)
{
    const double d = orc_half_to_float(rd16(blk));
    const double dmin = orc_half_to_float(rd16(blk + 2));
    const uint8_t *scales = blk + 4, *qs = blk + 16;
    int i;
    for (i = 0; i < ORC_QK; ++i) {
        int q, j, sc, mn;
        q4k_quant(qs, i, &q, &j);
        orc_q4k_scale_min(scales, j, &sc, &mn);
        w[i] = d * sc * q - dmin * mn;
    }
}

/* 6-bit quant (0..63) and scale slot (0..15) of weight i of a Q6_K block. */
static void q6k_quant(const uint8_t *blk, int i, int *q, int *slot)
{
    const uint8_t *ql = blk, *qh = blk + 128;
    int half = i / 128, r = i % 128;
    int quarter = r / 32, l = r % 32;
    const uint8_t *qlh = ql + 64 * half, *qhh = qh + 32 * half;
    int lo, hi;
    switch (quarter) {
    case 0: lo = qlh[l] & 15; hi = qhh[l] & 3; break;
    case 1: lo = qlh[l + 32] & 15; hi = (qhh[l] >> 2) & 3; break;
    case 2: lo = qlh[l] >> 4; hi = (qhh[l] >> 4) & 3; break;
    default: lo = qlh[l + 32] >> 4; hi = (qhh[l] >> 6) & 3; break;
    }
    *q = lo | (hi << 4);
    *slot = 8 * half + l / 16 + 2 * quarter;
}

/*
 * Q6_K super-block (210 bytes per 256 weights): ql[128] low nibbles, qh[64]
 * top 2-bit pairs, 16 signed 8-bit scales, fp16 d.  Weight = d*scale*(q-32).
 * fp32 order (the pages are silent): w = (d*scale)*(q-32).
 */
void orc_q6k_decode_block(const uint8_t *blk, float *w)
{
    const int8_t *sc = (const int8_t *)(blk + 192);
    const float d = orc_half_to_float(rd16(blk + 208));
    int i;
    for (i = 0; i < ORC_QK; ++i) {
        int q, slot;
        float ds;
        q6k_quant(blk, i, &q, &slot);
        ds = d * (float)sc[slot];
        w[i] = ds * (float)(q - 32);
    }
}

void orc_q6k_decode_block_f64(const uint8_t *blk, double *w)
{
    const int8_t *sc = (const int8_t *)(blk + 192);
    const double d = orc_half_to_float(rd16(blk + 208));
    int i;
    for (i = 0; i < ORC_QK; ++i) {
        int q, slot;
        q6k_quant(blk, i, &q, &slot);
        w[i] = d * sc[slot] * (q - 32);
    }
}

static int block_bytes(int qtype)
{
    if (qtype == ORC_Q4K) return ORC_Q4K_BYTES;
    if (qtype == ORC_Q6K) return ORC_Q6K_BYTES;
    return 0;
}

/* Row-major dequantization of an N x K packed matrix to fp32 (fp32 order). */
int orc_dequant(int qtype, const uint8_t *W, int64_t N, int64_t K, float *out)
{
    const int bb = block_bytes(qtype);
    const int64_t nsb = K / ORC_QK;
    int64_t n, s;
    if (bb == 0 || K % ORC_QK != 0) return -1;
    for (n = 0; n < N; ++n)
        for (s = 0; s < nsb; ++s) {
            const uint8_t *blk = W + (n * nsb + s) * bb;
            float *dst = out + n * K + s * ORC_QK;
            if (qtype == ORC_Q4K) orc_q4k_decode_block(blk, dst);
            else orc_q6k_decode_block(blk, dst);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* GEMV (decode)                                                             */
/* ------------------------------------------------------------------------ */

/*
 * y[m, n] = sum_k x[m, k] * w(n, k) for the listed rows n, with w the exact
 * (fp64) weight and every product and sum in fp64 ([q6k.rs], q4k_gemv_into /
 * q6k_gemv_indexed_async: one output per weight row, x of length K).  Also
 * returns absdot[m, n] = sum_k |x[m, k] * w(n, k)|, the scale of the GEMV
 * tolerance.  Outputs are indexed [m * nrows + r].
 */
int orc_gemv_rows(int qtype, const uint8_t *W, const float *x, int64_t M,
                  int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                  double *y, double *absdot)
{
    const int bb = block_bytes(qtype);
    const int64_t nsb = K / ORC_QK;
    double w[ORC_QK];
    int64_t r, m, s, i;
    if (bb == 0 || K % ORC_QK != 0) return -1;
    for (r = 0; r < nrows; ++r) {
        const int64_t n = rows[r];
        if (n < 0 || n >= N) return -2;
        for (m = 0; m < M; ++m) {
            y[m * nrows + r] = 0.0;
            if (absdot) absdot[m * nrows + r] = 0.0;
        }
        for (s = 0; s < nsb; ++s) {
            const uint8_t *blk = W + (n * nsb + s) * bb;
            if (qtype == ORC_Q4K) orc_q4k_decode_block_f64(blk, w);
            else orc_q6k_decode_block_f64(blk, w);
            for (m = 0; m < M; ++m) {
                const float *xr = x + m * K + s * ORC_QK;
                double acc = 0.0, aacc = 0.0;
                for (i = 0; i < ORC_QK; ++i) {
                    double p = (double)xr[i] * w[i];
                    acc += p;
                    aacc += fabs(p);
                }
                y[m * nrows + r] += acc;
                if (absdot) absdot[m * nrows + r] += aacc;
            }
        }
    }
    return 0;
}

/* Full GEMV: every row, output y[m * N + n]. */
int orc_gemv(int qtype, const uint8_t *W, const float *x, int64_t M, int64_t N,
             int64_t K, double *y, double *absdot)
{
    int64_t n, m;
    int rc;
    double yy[8], aa[8];
    if (M < 1 || M > 8) return -3;
    for (n = 0; n < N; ++n) {
        rc = orc_gemv_rows(qtype, W, x, M, N, K, &n, 1, yy, aa);
        if (rc) return rc;
        for (m = 0; m < M; ++m) {
            y[m * N + n] = yy[m];
            if (absdot) absdot[m * N + n] = aa[m];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 GEMM (prefill)                                                        */
/* ------------------------------------------------------------------------ */

/*
 * Y[m, n] = (sum_k dec(Xb[m, k]) * dec(Wb[n, k])) * x_deq * w_deq
 * ([gemm.rs], cublas_prefill_fp8_gemm: raw FP8 dot products, then the
 * activation scale absmax_x/448 and the weight scale absmax_w/448).  Every
 * E4M3 product is exact in fp64 and the sum stays inside fp64's 53 bits for
 * K up to 2^20, so the sum is exact whatever its order.  Both scales are
 * applied to the fp32-free fp64 sum (no fp16 intermediate).
 * Xb is [M x K] row-major, Wb is [N x K] row-major; pairs (ms[i], ns[i]) are
 * evaluated, y[i] receives the result.
 */
int orc_fp8_gemm_pairs(const uint8_t *Xb, float x_deq, const uint8_t *Wb,
                       float w_deq, int64_t M, int64_t N, int64_t K,
                       const int64_t *ms, const int64_t *ns, int64_t count,
                       double *y)
{
    double lut[256];
    int64_t i, k;
    int b;
    for (b = 0; b < 256; ++b) lut[b] = orc_e4m3_decode((uint8_t)b);
    for (i = 0; i < count; ++i) {
        const int64_t m = ms[i], n = ns[i];
        const uint8_t *xr, *wr;
        double acc = 0.0;
        if (m < 0 || m >= M || n < 0 || n >= N) return -2;
        xr = Xb + m * K;
        wr = Wb + n * K;
        for (k = 0; k < K; ++k) acc += lut[xr[k]] * lut[wr[k]];
        y[i] = acc * (double)x_deq * (double)w_deq;
    }
    return 0;
}

/* Full FP8 GEMM, Y[m * N + n]. */
int orc_fp8_gemm(const uint8_t *Xb, float x_deq, const uint8_t *Wb, float w_deq,
                 int64_t M, int64_t N, int64_t K, double *Y)
{
    int64_t m, n;
    int rc;
    for (m = 0; m < M; ++m)
        for (n = 0; n < N; ++n) {
            rc = orc_fp8_gemm_pairs(Xb, x_deq, Wb, w_deq, M, N, K, &m, &n, 1,
                                    &Y[m * N + n]);
            if (rc) return rc;
        }
    return 0;
}

/*
 * FP8 weight cache ([gemm.rs], get_or_cache_fp8_weight): dequantize the packed
 * weight to fp32, take its absmax, encode every weight with 448/absmax' and
 * keep absmax'/448 as the weight's dequant scale.  `scratch` must hold N*K
 * floats.
 */
int orc_fp8_weight_cache(int qtype, const uint8_t *W, int64_t N, int64_t K,
                         float *scratch, uint8_t *out, float *w_deq)
{
    uint32_t a;
    int rc = orc_dequant(qtype, W, N, K, scratch);
    if (rc) return rc;
    a = orc_absmax_bits(scratch, N * K);
    orc_quant_e4m3(scratch, N * K, a, out, w_deq);
    return 0;
}

/*
 * M-threshold routing ([mod.rs], cublas_gemm_threshold: M at or above the
 * threshold goes to the GEMM, below it to the batched GEMV).  Returns 1 for
 * the GEMM route, 0 for the GEMV route.
 */
int orc_route_is_gemm(int64_t M, int64_t threshold) { return M >= threshold; }

/* M padded up to a multiple of 16 ([gemm.rs], cublas_prefill_fp8_gemm). */
int64_t orc_pad_m(int64_t M) { return (M + 15) / 16 * 16; }

/* Array forms of the encoders and decoder (loops over the scalar functions). */
void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_encode_scaled_array(const float *x, int64_t n, float s, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_encode_scaled(x[i], s);
}

void orc_e4m3_decode_array(const uint8_t *b, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_e4m3_decode(b[i]);
}

void orc_half_to_float_array(const uint16_t *h, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = orc_half_to_float(h[i]);
}
