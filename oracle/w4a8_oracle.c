/*
 * w4a8_oracle.c -- plain, slow, scalar CPU reference for the W4A8 quantized linear.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file: only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark load it.  It shares
 * no code, table or header with the CUDA library.
 *
 * Sources (web pages; each function names the passage it follows):
 *   [nvfp4]  "radiance_nvfp4.py" -- unpack_e2m1, dequant_nvfp4, e2m1_index, _block_exponent,
 *            _encode_blocks, quant_mxfp4, dequant_mxfp4, requant_rows and the
 *            process_weights_after_loading of RadianceNvfp4ToMxfp4, RadianceFp8ChannelToMxfp4
 *            and RadianceBf16ToMxfp4.
 *   [readme] "vllm-radiance (MXFP4)" -- section "How the MXFP4 path works", subsection
 *            "The W4A8 fp8-WMMA kernel" (fp8 activations x e2m1 weights with folded e8m0).
 *   [ar]     "radiance_autoround.py" -- module docstring (format), autoround_linear (per-token
 *            fp8 activation quant), _exact_ref (dequantize-and-matmul definition).
 *
 * Precision: the pages fix fp32 for the requant arithmetic (torch fp32 tensors) and for the
 * activation scale; those steps are written in float with every operation rounded on its own
 * (build with -ffp-contract=off).  The GEMMs are exact definitions and accumulate in double.
 *
 * Readings where the pages are silent are listed in the design notes and repeated at each
 * function below.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ----------------------------------------------------------------------------------------- */
/* Number formats                                                                            */
/* ----------------------------------------------------------------------------------------- */

/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, 0x7F and 0xFF are NaN, largest finite magnitude 448, subnormals m * 2^-9. */
double orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int ex = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (ex == 0xF && m == 7) return NAN;
    if (ex == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, ex - 7);
    return s ? -v : v;
}

/* E4M3 encode: round to nearest representable value, ties to the even mantissa code,
 * saturating at 448 (the "satfinite" behaviour of a per-token fp8 cast whose scale maps the
 * row amax to 448).  Written from the format definition: find the binade of |y|, divide by
 * that binade's step (exact), round half to even, re-assemble.  A negative input keeps its
 * sign bit even when it rounds to zero (IEEE signed zero).  NaN input is outside the
 * contract and returns 0x7F. */
uint8_t orc_e4m3_encode(float y)
{
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal binade (and the rounding boundary into the first normal): step 2^-9 */
        double q = nearbyint(a / ldexp(1.0, -9)); /* a * 2^9 exact, rounded half-even */
        int m = (int)q;                             /* 0..8; 8 is the smallest normal */
        if (m == 8) return sign | 0x08;
        return sign | (uint8_t)m;
    }
    int E;
    frexp(a, &E);       /* a = f * 2^E, f in [0.5, 1): the binade is [2^(E-1), 2^E) */
    int eb = E - 1;     /* unbiased exponent, -6..8 */
    double step = ldexp(1.0, eb - 3);
    int m = (int)nearbyint(a / step); /* 8..16 */
    if (m == 16) { m = 8; eb += 1; }
    if (eb > 8 || (eb == 8 && m > 14)) return sign | 0x7E; /* unreachable below 448 */
    return sign | (uint8_t)(((eb + 7) << 3) | (m - 8));
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
float orc_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double orc_fp16_decode(uint16_t h)
{
    int s = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (ex == 0x1F) v = m ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + m / 1024.0, ex - 15);
    return s ? -v : v;
}

/* e2m1 magnitudes indexed by the low three code bits; bit 3 is the sign
 * ([nvfp4] _E2M1 grid and unpack_e2m1). */
static const float E2M1_GRID[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

double orc_e2m1_decode(uint8_t code)
{
    double v = E2M1_GRID[code & 7];
    return (code & 8) ? -v : v;
}

/* e8m0 block scale: code c is 2^(c-127); c = 255 (NaN) is outside the contract. */
double orc_e8m0_decode(uint8_t c) { return ldexp(1.0, (int)c - 127); }

/* ----------------------------------------------------------------------------------------- */
/* Activation quant ([ar] autoround_linear: dynamic per-token fp8; [readme] "fp8 activations") */
/* ----------------------------------------------------------------------------------------- */

/* Per row m: amax = max_k |x|, scale = amax / 448 (fp32, correctly rounded), codes =
 * e4m3(x / scale) with a correctly rounded fp32 division.  Reading for an all-zero row
 * (the pages are silent; amax/448 would give 0 and 0/0): scale = 1 and every code is the
 * signed zero of its input. */
void orc_act_quant(const uint16_t *x_bf16, int64_t M, int64_t K, uint8_t *xq, float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x_bf16 + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(orc_bf16_decode(row[k]));
            if (a > amax) amax = a;
        }
        float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        scale[m] = s;
        for (int64_t k = 0; k < K; ++k) {
            float v = orc_bf16_decode(row[k]) / s;
            xq[m * K + k] = orc_e4m3_encode(v);
        }
    }
}

/* ----------------------------------------------------------------------------------------- */
/* NVFP4 -> MXFP4 requant ([nvfp4])                                                           */
/* ----------------------------------------------------------------------------------------- */

/* [nvfp4] e2m1_index: |v| already divided by the block scale, clamped to 6, mapped to the
 * nearest grid index with ties to the even index, in three uniform pieces:
 *   a < 2: step 0.5 -> round(2a); 2 <= a < 4: step 1 -> round(a) + 2; a >= 4: round(a/2) + 4,
 * where round is half-to-even. */
int orc_e2m1_index(float a)
{
    if (a > 6.0f) a = 6.0f;
    float r;
    if (a < 2.0f)
        r = nearbyintf(a * 2.0f);
    else if (a < 4.0f)
        r = nearbyintf(a) + 2.0f;
    else
        r = nearbyintf(a * 0.5f) + 4.0f;
    return (int)r;
}

/* [nvfp4] _block_exponent, written exactly from the exponent bits rather than through a
 * rounded log2 (reading: the exact rule).  mode 0 = ocp: e = floor(log2 amax) - 2;
 * mode 1 = noclip: e = ceil(log2(amax / 6)), the smallest e with amax <= 6 * 2^e.
 * amax == 0 gives 0; the result is clamped to [-127, 127]. */
int orc_block_exponent(float amax, int mode)
{
    if (!(amax > 0.0f)) return 0;
    int E;
    double f = frexp((double)amax, &E); /* amax = f * 2^E, f in [0.5, 1) */
    int e;
    if (mode == 0)
        e = (E - 1) - 2;                 /* floor(log2 amax) = E - 1 */
    else
        e = (f <= 0.75) ? E - 3 : E - 2; /* 6 * 2^(E-3) = 0.75 * 2^E */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* [nvfp4] _encode_blocks for one 32-block at exponent e: v = w * 2^-e (exact), index from
 * e2m1_index(|v|), code sign bit set only when the index is nonzero (quant_mxfp4: "-0 stays
 * code 0").  Returns the block's squared error in units of the block scale,
 *   S = sum_k (|v_k| - G[idx_k])^2,
 * each square rounded to fp32 and added in ascending k with no fused multiply-add (reading:
 * the page sums in fp32 without fixing an order; this fixes one).  Because the grid step
 * is a power of two times the scale, the page's error (q - w)^2 summed is exactly S * 4^e. */
float orc_encode_block(const float *w, int e, uint8_t *codes)
{
    float S = 0.0f;
    for (int k = 0; k < 32; ++k) {
        float v = ldexpf(w[k], -e);
        float av = fabsf(v);
        int idx = orc_e2m1_index(av);
        float d = av - E2M1_GRID[idx];
        float d2 = d * d;
        S = S + d2;
        uint8_t c = (uint8_t)idx;
        if (signbit(w[k]) && idx != 0) c |= 8;
        codes[k] = c;
    }
    return S;
}

/* [nvfp4] quant_mxfp4 on one 32-block.  mode 2 = mse: e0 = noclip, e1 = e0 - 1 (one binade
 * finer, the top of the block may clip); take e1 iff its error is strictly lower.  In scale
 * units that is S1 * 4^(e0-1) < S0 * 4^e0, i.e. S1 < 4 * S0.  Reading: when e0 = -127 the
 * finer exponent is not encodable in e8m0 and e0 is kept.  Returns the chosen exponent,
 * writes the 32 codes, and stores the block's squared error in unscaled units. */
int orc_quant_block(const float *w, int mode, uint8_t *codes, double *err)
{
    float amax = 0.0f;
    for (int k = 0; k < 32; ++k) {
        float a = fabsf(w[k]);
        if (a > amax) amax = a;
    }
    int e;
    float S;
    if (mode == 2) {
        int e0 = orc_block_exponent(amax, 1);
        uint8_t c0[32], c1[32];
        float S0 = orc_encode_block(w, e0, c0);
        int take1 = 0;
        float S1 = 0.0f;
        if (e0 > -127) {
            S1 = orc_encode_block(w, e0 - 1, c1);
            take1 = (S1 < 4.0f * S0);
        }
        if (take1) { e = e0 - 1; S = S1; memcpy(codes, c1, 32); }
        else       { e = e0;     S = S0; memcpy(codes, c0, 32); }
    } else {
        e = orc_block_exponent(amax, mode);
        S = orc_encode_block(w, e, codes);
    }
    *err = ldexp((double)S, 2 * e);
    return e;
}

/* [nvfp4] dequant_nvfp4 for one row: W[k] = e2m1 * (fp32(scale_e4m3[k/16]) / divisor), the
 * per-16 scale divided by the partition's global divisor first (one fp32 division, correctly
 * rounded -- reading: the page's scalar division), then one rounded fp32 product. */
void orc_dequant_nvfp4_row(const uint8_t *packed, const uint8_t *scale_e4m3, float divisor,
                           int64_t K, float *w)
{
    for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = packed[k / 2];
        uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0x0F); /* low nibble = even k */
        float g = E2M1_GRID[code & 7];
        if (code & 8) g = -g;
        float s = (float)orc_e4m3_decode(scale_e4m3[k / 16]) / divisor;
        w[k] = g * s;
    }
}

/* [nvfp4] RadianceNvfp4ToMxfp4.process_weights_after_loading + requant_rows + quant_mxfp4:
 * each partition p (rows partition_rows[p], in order) is dequantized with its own divisor and
 * requantized per 32-block; codes pack two per byte with the even k in the low nibble and
 * the block exponent is stored as e + 127.  err_ssq, when non-NULL, receives per partition
 * {sum of squared requant error, sum of squared dequantized weights} in double. */
int orc_requant(const uint8_t *nv_packed, const uint8_t *nv_scale, const float *divisor,
                const int64_t *partition_rows, int P, int64_t N, int64_t K, int mode,
                uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq)
{
    if (K % 32 != 0 || mode < 0 || mode > 2) return 1;
    int64_t total = 0;
    for (int p = 0; p < P; ++p) total += partition_rows[p];
    if (total != N) return 1;
    int64_t row0 = 0;
    for (int p = 0; p < P; ++p) {
        double err_sum = 0.0, ssq_sum = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : err_sum, ssq_sum)
        for (int64_t n = row0; n < row0 + partition_rows[p]; ++n) {
            float w[32];
            uint8_t codes[32];
            for (int64_t b = 0; b < K / 32; ++b) {
                orc_dequant_nvfp4_row(nv_packed + n * (K / 2) + b * 16,
                                      nv_scale + n * (K / 16) + b * 2, divisor[p], 32, w);
                double err;
                int e = orc_quant_block(w, mode, codes, &err);
                for (int j = 0; j < 16; ++j)
                    out_packed[n * (K / 2) + b * 16 + j] =
                        (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
                out_e8m0[n * (K / 32) + b] = (uint8_t)(e + 127);
                err_sum += err;
                for (int k = 0; k < 32; ++k) ssq_sum += (double)w[k] * (double)w[k];
            }
        }
        if (err_ssq) { err_ssq[2 * p] = err_sum; err_ssq[2 * p + 1] = ssq_sum; }
        row0 += partition_rows[p];
    }
    return 0;
}

/* One layer of already-dequantized rows -> MXFP4 (quant_mxfp4 per 32-block, packing as in
 * orc_requant).  row(n, w) fills w[0..K) with row n's fp32 weights.  err_ssq, when non-NULL,
 * receives {sum of squared requant error, sum of squared weights} for the whole layer. */
typedef void (*orc_row_fn)(const void *ctx, int64_t n, int64_t K, float *w);

static void orc_requant_rows(orc_row_fn row, const void *ctx, int64_t N, int64_t K, int mode,
                             uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq)
{
    double err_sum = 0.0, ssq_sum = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : err_sum, ssq_sum)
    for (int64_t n = 0; n < N; ++n) {
        float *w = (float *)malloc(sizeof(float) * (size_t)K);
        uint8_t codes[32];
        row(ctx, n, K, w);
        for (int64_t b = 0; b < K / 32; ++b) {
            double err;
            int e = orc_quant_block(w + 32 * b, mode, codes, &err);
            for (int j = 0; j < 16; ++j)
                out_packed[n * (K / 2) + b * 16 + j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
            out_e8m0[n * (K / 32) + b] = (uint8_t)(e + 127);
            err_sum += err;
        }
        for (int64_t k = 0; k < K; ++k) ssq_sum += (double)w[k] * (double)w[k];
        free(w);
    }
    if (err_ssq) { err_ssq[0] = err_sum; err_ssq[1] = ssq_sum; }
}

/* [nvfp4] RadianceFp8ChannelToMxfp4.process_weights_after_loading: W[n, k] = fp32(w8[n, k]) *
 * scale[n], the e4m3 code cast to fp32 (exact) times the row's fp32 channel scale, one rounded
 * fp32 product per element; then quant_mxfp4 and the layer's relRMS sums, as for NVFP4 with the
 * whole layer as one partition. */
struct orc_fp8ch { const uint8_t *w8; const float *scale; };

static void orc_fp8ch_row(const void *ctx, int64_t n, int64_t K, float *w)
{
    const struct orc_fp8ch *c = (const struct orc_fp8ch *)ctx;
    const float s = c->scale[n];
    for (int64_t k = 0; k < K; ++k) w[k] = (float)orc_e4m3_decode(c->w8[n * K + k]) * s;
}

int orc_requant_fp8_channel(const uint8_t *w8, const float *scale, int64_t N, int64_t K, int mode,
                            uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq)
{
    if (K % 32 != 0 || mode < 0 || mode > 2 || N < 0) return 1;
    struct orc_fp8ch c = {w8, scale};
    orc_requant_rows(orc_fp8ch_row, &c, N, K, mode, out_packed, out_e8m0, err_ssq);
    return 0;
}

/* [nvfp4] RadianceBf16ToMxfp4.process_weights_after_loading: requant_rows on the bf16 weight;
 * the fp32 cast of a bf16 value is exact, so W[n, k] = fp32(w[n, k]). */
static void orc_bf16_row(const void *ctx, int64_t n, int64_t K, float *w)
{
    const uint16_t *wb = (const uint16_t *)ctx;
    for (int64_t k = 0; k < K; ++k) w[k] = orc_bf16_decode(wb[n * K + k]);
}

int orc_requant_bf16(const uint16_t *w_bf16, int64_t N, int64_t K, int mode, uint8_t *out_packed,
                     uint8_t *out_e8m0, double *err_ssq)
{
    if (K % 32 != 0 || mode < 0 || mode > 2 || N < 0) return 1;
    orc_requant_rows(orc_bf16_row, w_bf16, N, K, mode, out_packed, out_e8m0, err_ssq);
    return 0;
}

/* [nvfp4] dequant_mxfp4: W[n, k] = e2m1 * 2^(e8m0 - 127). */
void orc_dequant_mxfp4(const uint8_t *packed, const uint8_t *e8m0, int64_t N, int64_t K,
                       double *w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = packed[n * (K / 2) + k / 2];
            uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0x0F);
            w[n * K + k] = orc_e2m1_decode(code) * orc_e8m0_decode(e8m0[n * (K / 32) + k / 32]);
        }
}

/* ----------------------------------------------------------------------------------------- */
/* NVFP4 producer (input synthesis for the requant workloads; not part of the method)        */
/* ----------------------------------------------------------------------------------------- */

/* The pages only state the checkpoint layout ([nvfp4] create_weights / dequant_nvfp4): e2m1
 * codes, an e4m3 scale per 16, and a per-partition global scale stored as the divisor
 * 6 * 448 / amax.  The plainest producer consistent with that layout: div_p = 6*448/amax_p;
 * per 16-block s = e4m3(amax16 * div_p / 6); codes = e2m1_index(|w| * div_p / s) with the
 * same sign rule; a block whose scale encodes to zero gets all-zero codes. */
void orc_nvfp4_quantize(const float *w, const int64_t *partition_rows, int P, int64_t K,
                        uint8_t *packed, uint8_t *scale_e4m3, float *divisor)
{
    int64_t row0 = 0;
    for (int p = 0; p < P; ++p) {
        int64_t r1 = row0 + partition_rows[p];
        float amax = 0.0f;
        for (int64_t n = row0; n < r1; ++n)
            for (int64_t k = 0; k < K; ++k) {
                float a = fabsf(w[n * K + k]);
                if (a > amax) amax = a;
            }
        float div = (amax > 0.0f) ? (6.0f * 448.0f) / amax : 1.0f;
        divisor[p] = div;
#pragma omp parallel for schedule(static)
        for (int64_t n = row0; n < r1; ++n)
            for (int64_t b = 0; b < K / 16; ++b) {
                const float *wb = w + n * K + b * 16;
                float a16 = 0.0f;
                for (int k = 0; k < 16; ++k) {
                    float a = fabsf(wb[k]);
                    if (a > a16) a16 = a;
                }
                uint8_t sc = orc_e4m3_encode((a16 * div) / 6.0f);
                scale_e4m3[n * (K / 16) + b] = sc;
                float sv = (float)orc_e4m3_decode(sc);
                for (int k = 0; k < 16; ++k) {
                    int idx = 0;
                    if (sv > 0.0f) idx = orc_e2m1_index((fabsf(wb[k]) * div) / sv);
                    uint8_t c = (uint8_t)idx;
                    if (signbit(wb[k]) && idx != 0) c |= 8;
                    int64_t kk = b * 16 + k;
                    uint8_t *dst = &packed[n * (K / 2) + kk / 2];
                    if (kk & 1) *dst = (uint8_t)((*dst & 0x0F) | (c << 4));
                    else        *dst = (uint8_t)((*dst & 0xF0) | c);
                }
            }
        row0 = r1;
    }
}

/* ----------------------------------------------------------------------------------------- */
/* GEMMs: dequantize exactly, multiply, accumulate in double with k ascending                 */
/* ----------------------------------------------------------------------------------------- */

/* [readme] "The W4A8 fp8-WMMA kernel" with [nvfp4] item 3 of the module docstring (weight
 * [N, K/2] low nibble = even k, weight_scale [N, K/32] e8m0):
 *   out[m, n] = scale[m] * sum_k e4m3(xq[m, k]) * e2m1(W[n, k]) * 2^(E[n, k/32] - 127).
 * Computes the (m, n) pairs listed in idx_m/idx_n (count pairs) into out[i]; the unrounded
 * double result is returned (the bf16 store is the kernel's last step and the tolerance
 * accounts for it). */
void orc_mxfp4_linear_pairs(const uint8_t *xq, const float *x_scale, const uint8_t *w_packed,
                            const uint8_t *w_e8m0, int64_t K, const int64_t *idx_m,
                            const int64_t *idx_n, int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = idx_m[i], n = idx_n[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = w_packed[n * (K / 2) + k / 2];
            uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0x0F);
            double wv = orc_e2m1_decode(code) * orc_e8m0_decode(w_e8m0[n * (K / 32) + k / 32]);
            acc += orc_e4m3_decode(xq[m * K + k]) * wv;
        }
        out[i] = (double)x_scale[m] * acc;
    }
}

/* Whole output [M, N] (row-major). */
void orc_mxfp4_linear(const uint8_t *xq, const float *x_scale, const uint8_t *w_packed,
                      const uint8_t *w_e8m0, int64_t M, int64_t N, int64_t K, double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = w_packed[n * (K / 2) + k / 2];
                uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0x0F);
                double wv = orc_e2m1_decode(code) * orc_e8m0_decode(w_e8m0[n * (K / 32) + k / 32]);
                acc += orc_e4m3_decode(xq[m * K + k]) * wv;
            }
            out[m * N + n] = (double)x_scale[m] * acc;
        }
}

/* [ar] module docstring and _exact_ref: qweight [K/8, N] int32 with nibble j of word (i, n)
 * holding k = 8i + j; code c means the integer c - 8 (qzeros uniformly 0x77777777, i.e. a
 * zero point of 8); scales [K/128, N] fp16, one per 128 along K:
 *   out[m, n] = scale[m] * sum_k e4m3(xq[m, k]) * (c[k, n] - 8) * fp16(s[k/128, n]). */
void orc_int4g128_linear_pairs(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                               const uint16_t *scales_fp16, int64_t N, int64_t K,
                               const int64_t *idx_m, const int64_t *idx_n, int64_t count,
                               double *out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = idx_m[i], n = idx_n[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            uint32_t word = (uint32_t)qweight[(k / 8) * N + n];
            int c = (int)((word >> (4 * (k % 8))) & 0xF);
            double wv = (double)(c - 8) * orc_fp16_decode(scales_fp16[(k / 128) * N + n]);
            acc += orc_e4m3_decode(xq[m * K + k]) * wv;
        }
        out[i] = (double)x_scale[m] * acc;
    }
}

void orc_int4g128_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                         const uint16_t *scales_fp16, int64_t M, int64_t N, int64_t K,
                         double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint32_t word = (uint32_t)qweight[(k / 8) * N + n];
                int c = (int)((word >> (4 * (k % 8))) & 0xF);
                double wv = (double)(c - 8) * orc_fp16_decode(scales_fp16[(k / 128) * N + n]);
                acc += orc_e4m3_decode(xq[m * K + k]) * wv;
            }
            out[m * N + n] = (double)x_scale[m] * acc;
        }
}

/* Asymmetric int4 group-128 ("vllm-radiance (MXFP4)", section "ParoQuant (int4 W4A8 and int5 W5A8)":
 * int4 group-128 asymmetric, the zero point folded into the GEMM as a row-sum correction).  The
 * zero point of group g and column n is z = 1 + nibble (n % 8) of qzeros[g, n / 8] -- reading:
 * the packed-qzeros convention under which the symmetric checkpoint's 0x77777777 means the
 * zero point 8 that "radiance_autoround.py" states -- and the weight is (c - z) * s:
 *   out[m, n] = scale[m] * sum_k e4m3(xq[m, k]) * (c[k, n] - z[k/128, n]) * fp16(s[k/128, n]). */
static double orc_int4_asym_dot(const uint8_t *xq, const int32_t *qweight, const uint16_t *scales_fp16,
                                const int32_t *qzeros, int64_t N, int64_t K, int64_t m, int64_t n)
{
    const int64_t NZ = (N + 7) / 8;
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        uint32_t word = (uint32_t)qweight[(k / 8) * N + n];
        int c = (int)((word >> (4 * (k % 8))) & 0xF);
        uint32_t zw = (uint32_t)qzeros[(k / 128) * NZ + n / 8];
        int z = 1 + (int)((zw >> (4 * (n % 8))) & 0xF);
        double wv = (double)(c - z) * orc_fp16_decode(scales_fp16[(k / 128) * N + n]);
        acc += orc_e4m3_decode(xq[m * K + k]) * wv;
    }
    return acc;
}

void orc_int4g128_asym_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                              const uint16_t *scales_fp16, const int32_t *qzeros, int64_t M, int64_t N,
                              int64_t K, double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = (double)x_scale[m] * orc_int4_asym_dot(xq, qweight, scales_fp16, qzeros, N, K, m, n);
}

void orc_int4g128_asym_linear_pairs(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                                    const uint16_t *scales_fp16, const int32_t *qzeros, int64_t N, int64_t K,
                                    const int64_t *idx_m, const int64_t *idx_n, int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = (double)x_scale[idx_m[i]] *
                 orc_int4_asym_dot(xq, qweight, scales_fp16, qzeros, N, K, idx_m[i], idx_n[i]);
}

/* int5 group-128 ("vllm-radiance (MXFP4)", section "int5 (W5A8)": the int4 path with 5-bit
 * codes, c - 16 spanning -16..15; the low nibbles keep the int4 word layout and the fifth bit
 * sits in a plane of one byte per word).  Reading of the plane: qhigh [K/8, N] uint8, bit j of
 * byte (i, n) is bit 4 of the code of k = 8i + j, the byte beside word (i, n) of qweight.  So
 *   c[k, n] = nibble (k % 8) of qweight[k/8, n]  +  16 * bit (k % 8) of qhigh[k/8, n].
 * Zero point: 16 (symmetric), or z[k/128, n] from a byte per group and column when zeros is
 * given (the page folds a zero point in for int5 as for int4 but does not give its storage; a
 * byte per (group, column) holding z itself is the reading taken):
 *   out[m, n] = scale[m] * sum_k e4m3(xq[m, k]) * (c[k, n] - z[k/128, n]) * fp16(s[k/128, n]). */
static double orc_int5_dot(const uint8_t *xq, const int32_t *qweight, const uint8_t *qhigh,
                           const uint16_t *scales_fp16, const uint8_t *zeros, int64_t N, int64_t K,
                           int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        uint32_t word = (uint32_t)qweight[(k / 8) * N + n];
        int lo = (int)((word >> (4 * (k % 8))) & 0xF);
        int hi = (int)((qhigh[(k / 8) * N + n] >> (k % 8)) & 1);
        int c = lo + 16 * hi;
        int z = zeros ? (int)zeros[(k / 128) * N + n] : 16;
        double wv = (double)(c - z) * orc_fp16_decode(scales_fp16[(k / 128) * N + n]);
        acc += orc_e4m3_decode(xq[m * K + k]) * wv;
    }
    return acc;
}

void orc_int5g128_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                         const uint8_t *qhigh, const uint16_t *scales_fp16, const uint8_t *zeros,
                         int64_t M, int64_t N, int64_t K, double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * N + n] = (double)x_scale[m] * orc_int5_dot(xq, qweight, qhigh, scales_fp16, zeros, N, K, m, n);
}

void orc_int5g128_linear_pairs(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                               const uint8_t *qhigh, const uint16_t *scales_fp16, const uint8_t *zeros,
                               int64_t N, int64_t K, const int64_t *idx_m, const int64_t *idx_n,
                               int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = (double)x_scale[idx_m[i]] *
                 orc_int5_dot(xq, qweight, qhigh, scales_fp16, zeros, N, K, idx_m[i], idx_n[i]);
}

/* W4A4 ("vllm-radiance (MXFP4)", section "Native MXFP4": Quark OCP micro-scaling checkpoints with
 * MXFP4 weights AND activations, group 32, e8m0 scales; and "The W4A8 fp8-WMMA kernel", which
 * names that W4A4 path as the less accurate alternative to fp8 activations).
 *
 * Activation quant: the pages do not spell out the activation quantizer; the reading taken is
 * the OCP micro-scaling rule, which "radiance_nvfp4.py" names "ocp" (_block_exponent: e =
 * floor(log2 amax) - 2, then e2m1_index of x * 2^-e with the sign rule), applied per 32 along
 * each token row -- quant_mxfp4 in ocp mode on the bf16 row, the same routine as the bf16
 * requant source above.  No per-token scale: each block carries its own e8m0. */
void orc_act_quant_mxfp4(const uint16_t *x_bf16, int64_t M, int64_t K, uint8_t *xa_packed, uint8_t *xa_e8m0)
{
    orc_requant_rows(orc_bf16_row, x_bf16, M, K, 0 /* ocp */, xa_packed, xa_e8m0, NULL);
}

/* W4A4 GEMM: both operands dequantized exactly (e2m1 * 2^(e8m0 - 127)), fp64 sum, k ascending:
 *   out[m, n] = sum_k e2m1(xa[m, k]) 2^(xe[m, k/32] - 127) * e2m1(w[n, k]) 2^(we[n, k/32] - 127). */
static double orc_a4_dot(const uint8_t *xa, const uint8_t *xe, const uint8_t *w_packed, const uint8_t *w_e8m0,
                         int64_t K, int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        uint8_t xb = xa[m * (K / 2) + k / 2], wb = w_packed[n * (K / 2) + k / 2];
        uint8_t xc = (k & 1) ? (xb >> 4) : (xb & 0x0F), wc = (k & 1) ? (wb >> 4) : (wb & 0x0F);
        double xv = orc_e2m1_decode(xc) * orc_e8m0_decode(xe[m * (K / 32) + k / 32]);
        double wv = orc_e2m1_decode(wc) * orc_e8m0_decode(w_e8m0[n * (K / 32) + k / 32]);
        acc += xv * wv;
    }
    return acc;
}

void orc_mxfp4_a4_linear(const uint8_t *xa, const uint8_t *xe, const uint8_t *w_packed, const uint8_t *w_e8m0,
                         int64_t M, int64_t N, int64_t K, double *out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) out[m * N + n] = orc_a4_dot(xa, xe, w_packed, w_e8m0, K, m, n);
}

void orc_mxfp4_a4_linear_pairs(const uint8_t *xa, const uint8_t *xe, const uint8_t *w_packed,
                               const uint8_t *w_e8m0, int64_t K, const int64_t *idx_m, const int64_t *idx_n,
                               int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) out[i] = orc_a4_dot(xa, xe, w_packed, w_e8m0, K, idx_m[i], idx_n[i]);
}

/* Number of threads the parallel loops above use (1 without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Vectorised helpers for the pins (loops over the scalar codecs above). */
void orc_e4m3_encode_many(const float *y, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(y[i]);
}

void orc_fp16_decode_many(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_fp16_decode(h[i]);
}

void orc_e4m3_decode_many(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
