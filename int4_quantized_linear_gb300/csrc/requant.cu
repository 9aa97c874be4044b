// requant.cu -- NVFP4 / FP8-per-channel / bf16 -> MXFP4 requant of a linear at load time.
//
// "radiance_nvfp4.py": dequant_nvfp4 (W = e2m1 * fp32(e4m3 scale per 16) / global divisor,
// per partition of a merged linear), _block_exponent (ocp / noclip), quant_mxfp4 (mse: the
// no-clip exponent or one binade finer, whichever has the lower squared error), e2m1_index
// (nearest grid point, ties to the even code), _encode_blocks, and the packing of item 3 of
// the module docstring (low nibble = even k, e8m0 = e + 127).  The FP8-per-channel and bf16
// sources (RadianceFp8ChannelToMxfp4, RadianceBf16ToMxfp4) differ only in the dequantize step
// and treat the layer as one partition.
//
// One thread per 32-block: a 16-byte load of 32 NVFP4 codes plus two e4m3 scale bytes in (32
// bytes of FP8 codes, or 64 of bf16), a 16-byte store of 32 MXFP4 codes plus one e8m0 byte out,
// so a warp moves 512 contiguous bytes of codes each way; a persistent grid strides over the
// blocks of each partition.  The whole block lives in registers; the page's fp32 transient and
// its row chunking are not needed.  Every fp32 operation is written with an explicit rounding
// intrinsic so that no multiply-add is contracted and the results match the oracle bit for
// bit: the exponent comes from the float's bits (exact), the scaling by 2^-e is an exact
// power-of-two product, and the squared errors are summed in ascending k.
#include <algorithm>

#include "common.cuh"

namespace w4a8 {

constexpr int RQ_THREADS = 256;
constexpr int RQ_MAX_PARTS = 16;

struct Partitions {
    int P;
    int64_t row_end[RQ_MAX_PARTS];
};

// floor(log2 a) for finite a > 0, from the bits (subnormals normalised).
W4A8_DEVICE int floor_log2_exact(float a)
{
    uint32_t u = __float_as_uint(a);
    int ex = (u >> 23) & 0xff;
    if (ex) return ex - 127;
    return (31 - __clz(u)) - 149;
}

// Is the significand of a (in [1, 2)) at most 1.5?
W4A8_DEVICE bool significand_le_1p5(float a)
{
    uint32_t u = __float_as_uint(a);
    int ex = (u >> 23) & 0xff;
    uint32_t f = ex ? (u & 0x7fffffu) : ((u << (__clz(u) - 8)) & 0x7fffffu);
    return f <= 0x400000u;
}

// _block_exponent: mode 0 ocp -> floor(log2 amax) - 2; otherwise noclip -> the smallest e
// with amax <= 6 * 2^e, i.e. ceil(log2(amax / 6)).  amax = 0 -> 0; clamped to [-127, 127].
W4A8_DEVICE int block_exponent(float amax, int mode)
{
    if (!(amax > 0.0f)) return 0;
    int fl = floor_log2_exact(amax);
    int e = (mode == 0) ? fl - 2 : (significand_le_1p5(amax) ? fl - 2 : fl - 1);
    return min(127, max(-127, e));
}

// Two fp32 values -> their signed e2m1 codes in one byte (low nibble = a0): the hardware
// conversion rounds |a| to the nearest grid point {0, .5, 1, 1.5, 2, 3, 4, 6} with ties to the
// even code and saturates at 6 -- e2m1_index of min(|a|, 6), whose ties go to the even index --
// and keeps the sign, also on a zero magnitude (-0 and small negatives give code 8).
W4A8_DEVICE uint32_t e2m1x2_from_float(float a0, float a1)
{
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(a1), "f"(a0));
    return r;
}

// Encode 32 values at exponent e.  Returns the squared error in scale units (fp32, squares
// rounded and added in ascending k; only when ERR, else 0) and the 32 codes as four words of
// eight nibbles.
template <bool ERR>
W4A8_DEVICE float encode_block(const float (&w)[32], int e, uint32_t (&codes)[4])
{
    const float inv = exp2i(-e);
    float S = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) codes[j] = 0;
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
        // v = w 2^-e is exact (a power-of-two product); |v| may exceed 6 (up to 12 one binade
        // finer), and the error is taken against the unclamped value.  The signed value and its
        // signed grid point differ by exactly -(|v| - grid) when v < 0, so the square is the same.
        const float a0 = __fmul_rn(w[k], inv), a1 = __fmul_rn(w[k + 1], inv);
        const uint32_t b = e2m1x2_from_float(a0, a1);
        if constexpr (ERR) {
            const float2 g = e2m1x2_to_float2(b);  // the chosen grid values, signed (exact)
            const float d0 = __fsub_rn(a0, g.x), d1 = __fsub_rn(a1, g.y);
            S = __fadd_rn(S, __fmul_rn(d0, d0));
            S = __fadd_rn(S, __fmul_rn(d1, d1));
        }
        codes[k >> 3] |= b << (4 * (k & 7));
    }
    // the sign bit only on a nonzero index, so -0 and small negatives give code 0, never 8: per
    // nibble, (index + 7) carries into bit 3 exactly when the index is nonzero
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t keep = ((codes[j] & 0x77777777u) + 0x77777777u) & 0x88888888u;
        codes[j] &= 0x77777777u | keep;
    }
    return S;
}

// R2-R4 on one 32-block of fp32 weights: choose the exponent (R2), encode (R3) and pack (R4).
// Returns the block exponent e; with ERR, S receives the squared error in scale units and ssq
// the block's sum of squared weights (the mse rule computes the errors either way).
template <bool ERR>
W4A8_DEVICE int quantize_block(const float (&w)[32], int mode, uint4 &out, float &S, float &ssq)
{
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(w[k]));
    uint32_t codes[4];
    int e;
    if (mode == 2) {
        const int e0 = block_exponent(amax, 1);
        uint32_t c0[4];
        const float S0 = encode_block<true>(w, e0, c0);
        bool take1 = false;
        uint32_t c1[4] = {0, 0, 0, 0};
        float S1 = 0.0f;
        if (e0 > -127) {
            S1 = encode_block<true>(w, e0 - 1, c1);
            take1 = S1 < __fmul_rn(4.0f, S0);
        }
        e = take1 ? e0 - 1 : e0;
        S = take1 ? S1 : S0;
#pragma unroll
        for (int j = 0; j < 4; ++j) codes[j] = take1 ? c1[j] : c0[j];
    } else {
        e = block_exponent(amax, mode);
        S = encode_block<ERR>(w, e, codes);
    }
    // R4: nibble k of word j is element 8j + k (the even k lands in the low nibble)
    out = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    // sum of squares for the relRMS report (a float-precision statistic): the block's 32
    // squares rounded and added in fp32, ascending k; blocks are then summed in fp64.  fp64
    // arithmetic per element would cost more than the rest of the kernel on GB300.
    float q = 0.0f;
    if constexpr (ERR) {
#pragma unroll
        for (int k = 0; k < 32; ++k) q = __fadd_rn(q, __fmul_rn(w[k], w[k]));
    }
    ssq = q;
    return e;
}

// R1 sources.  Each yields block g's 32 fp32 weights (row n = g / (K / 32)).
// NVFP4 ("radiance_nvfp4.py", dequant_nvfp4): w = fl(e2m1 * fl(fp32(e4m3 scale per 16) / divisor))
// for partition p's divisor: 16 packed bytes and two scale bytes per block.
// The scale byte has 256 values, so the CTA divides each by the partition's divisor once, into a
// shared table, before the partition's blocks.
struct SrcNvfp4 {
    const uint8_t *packed, *scale;
    const float *divisor;
    W4A8_DEVICE void prepare(int p, float *tab) const
    {
        const float dv = divisor[p];
        for (int c = threadIdx.x; c < 256; c += blockDim.x)
            tab[c] = __fdiv_rn(e4m3x2_to_float2((uint16_t)c).x, dv);
    }
    W4A8_DEVICE void load(int64_t g, int64_t, int, const float *tab, float (&w)[32]) const
    {
        const uint4 pk = *reinterpret_cast<const uint4 *>(packed + g * 16);
        const uint16_t sc = *reinterpret_cast<const uint16_t *>(scale + g * 2);
        const float sd0 = tab[sc & 0xffu], sd1 = tab[sc >> 8];
        const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float2 gv = e2m1x2_to_float2((words[j >> 2] >> (8 * (j & 3))) & 0xffu);
            float sd = j < 8 ? sd0 : sd1;
            w[2 * j] = __fmul_rn(gv.x, sd);
            w[2 * j + 1] = __fmul_rn(gv.y, sd);
        }
    }
};
// FP8 per channel ("radiance_nvfp4.py", RadianceFp8ChannelToMxfp4): w = fl(fp32(e4m3 code) *
// scale[n]), 32 code bytes per block.
struct SrcFp8Channel {
    const uint8_t *w8;
    const float *scale;
    W4A8_DEVICE void prepare(int, float *) const {}
    W4A8_DEVICE void load(int64_t g, int64_t n, int, const float *, float (&w)[32]) const
    {
        const uint4 a = *reinterpret_cast<const uint4 *>(w8 + g * 32);
        const uint4 b = *reinterpret_cast<const uint4 *>(w8 + g * 32 + 16);
        const uint32_t words[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float s = scale[n];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 v = e4m3x2_to_float2((uint16_t)(words[j >> 1] >> (16 * (j & 1))));
            w[2 * j] = __fmul_rn(v.x, s);
            w[2 * j + 1] = __fmul_rn(v.y, s);
        }
    }
};
// bf16 ("radiance_nvfp4.py", RadianceBf16ToMxfp4): the fp32 value of each bf16 weight (exact),
// 64 bytes per block.
struct SrcBf16 {
    const uint16_t *wb;
    W4A8_DEVICE void prepare(int, float *) const {}
    W4A8_DEVICE void load(int64_t g, int64_t, int, const float *, float (&w)[32]) const
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(wb + g * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = src[q];
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[8 * q + 2 * j] = __uint_as_float(words[j] << 16);
                w[8 * q + 2 * j + 1] = __uint_as_float(words[j] & 0xffff0000u);
            }
        }
    }
};

// Persistent grid: the partitions one after another; inside a partition every thread walks the
// 32-blocks with a grid stride, so a warp handles 32 consecutive blocks of a row (512 bytes of
// codes each way).  The error sums are kept per thread, reduced per CTA and added to the output
// with one atomic per CTA and partition.
template <class Src, bool ERR>
__global__ void __launch_bounds__(RQ_THREADS)
requant_kernel(const Src src, Partitions parts, int64_t N, int64_t K, int mode,
               uint8_t *__restrict__ out_packed, uint8_t *__restrict__ out_e8m0,
               double *__restrict__ err_ssq)
{
    __shared__ double red[2][RQ_THREADS / 32];
    __shared__ float tab[256];
    const int64_t KB = K / 32;
    const int64_t stride = (int64_t)gridDim.x * RQ_THREADS;
    int64_t row_beg = 0;
    for (int p = 0; p < parts.P; ++p) {
        const int64_t row_end = parts.row_end[p];
        __syncthreads();  // the previous partition's table is no longer read
        src.prepare(p, tab);
        __syncthreads();
        double err = 0.0, ssq = 0.0;
        for (int64_t g = row_beg * KB + (int64_t)blockIdx.x * RQ_THREADS + threadIdx.x; g < row_end * KB; g += stride) {
            float w[32];
            src.load(g, g / KB, p, tab, w);
            uint4 codes;
            float S, q;
            const int e = quantize_block<ERR>(w, mode, codes, S, q);
            *reinterpret_cast<uint4 *>(out_packed + g * 16) = codes;
            out_e8m0[g] = (uint8_t)(e + 127);
            if (ERR) {
                err += ldexp((double)S, 2 * e);
                ssq += (double)q;
            }
        }
        if (ERR) {
            err = warp_sum_d(err);
            ssq = warp_sum_d(ssq);
            if ((threadIdx.x & 31) == 0) {
                red[0][threadIdx.x >> 5] = err;
                red[1][threadIdx.x >> 5] = ssq;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                double a = 0.0, b2 = 0.0;
                for (int i = 0; i < RQ_THREADS / 32; ++i) {
                    a += red[0][i];
                    b2 += red[1][i];
                }
                if (a != 0.0 || b2 != 0.0) {
                    atomicAdd(&err_ssq[2 * p], a);
                    atomicAdd(&err_ssq[2 * p + 1], b2);
                }
            }
            __syncthreads();
        }
        row_beg = row_end;
    }
}

}  // namespace w4a8

namespace w4a8 {

// Persistent grid over all of the layer's 32-blocks: as many CTAs as fit on the GPU at once (or
// fewer for small layers); err_ssq is zeroed first and receives one atomic pair per CTA and
// partition.
template <class Src>
static w4a8_status launch_requant(const Src &src, const Partitions &parts, int64_t N, int64_t K, int mode,
                                  uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq, cudaStream_t stream)
{
    if (err_ssq && cudaMemsetAsync(err_ssq, 0, sizeof(double) * 2 * parts.P, stream) != cudaSuccess)
        return W4A8_ERR_CUDA;
    const int64_t blocks = N * (K / 32);
    // SM count and residency per device, queried once (a per-call query costs microseconds of
    // host time, as much as the kernel itself for a few activation rows)
    constexpr int MAX_DEV = 64;
    static int sms_of[MAX_DEV] = {0}, per_sm_of[MAX_DEV] = {0};  // (both instantiations: same residency)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4A8_ERR_CUDA;
    int sms = dev < MAX_DEV ? sms_of[dev] : 0, per_sm = dev < MAX_DEV ? per_sm_of[dev] : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_kernel<Src, true>, RQ_THREADS, 0) != cudaSuccess)
            return W4A8_ERR_CUDA;
        if (dev < MAX_DEV) {
            per_sm_of[dev] = per_sm;
            sms_of[dev] = sms;
        }
    }
    const int64_t need = (blocks + RQ_THREADS - 1) / RQ_THREADS;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sms * std::max(per_sm, 1)));
    if (err_ssq)
        requant_kernel<Src, true><<<(unsigned)grid, RQ_THREADS, 0, stream>>>(src, parts, N, K, mode, out_packed,
                                                                            out_e8m0, err_ssq);
    else
        requant_kernel<Src, false><<<(unsigned)grid, RQ_THREADS, 0, stream>>>(src, parts, N, K, mode, out_packed,
                                                                             out_e8m0, nullptr);
    return w4a8_launch_status();
}

static Partitions one_partition(int64_t N)
{
    Partitions parts;
    parts.P = 1;
    for (int p = 0; p < RQ_MAX_PARTS; ++p) parts.row_end[p] = N;
    return parts;
}

}  // namespace w4a8

extern "C" w4a8_status nvfp4_to_mxfp4_requant(const uint8_t *nv_packed, const uint8_t *nv_scale_e4m3,
                                              const float *global_divisor,
                                              const int64_t *partition_rows, int P, int64_t N,
                                              int64_t K, int mode, uint8_t *out_packed,
                                              uint8_t *out_e8m0, double *err_ssq,
                                              cudaStream_t stream)
{
    if (N < 0 || K < 0 || mode < 0 || mode > 2) return W4A8_ERR_INVALID_ARG;
    if (P < 1 || P > w4a8::RQ_MAX_PARTS || !partition_rows) return W4A8_ERR_INVALID_ARG;
    w4a8::Partitions parts;
    parts.P = P;
    int64_t total = 0;
    for (int p = 0; p < P; ++p) {
        if (partition_rows[p] < 0) return W4A8_ERR_INVALID_ARG;
        total += partition_rows[p];
        parts.row_end[p] = total;
    }
    for (int p = P; p < w4a8::RQ_MAX_PARTS; ++p) parts.row_end[p] = total;
    if (total != N) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || K == 0) return W4A8_OK;
    if (!nv_packed || !nv_scale_e4m3 || !global_divisor || !out_packed || !out_e8m0)
        return W4A8_ERR_INVALID_ARG;
    if (!w4a8_aligned(nv_packed, 16) || !w4a8_aligned(out_packed, 16) ||
        !w4a8_aligned(nv_scale_e4m3, 2) || !w4a8_aligned(global_divisor, 4) ||
        (err_ssq && !w4a8_aligned(err_ssq, 8)))
        return W4A8_ERR_MISALIGNED;
    // a row's 32-blocks are contiguous in both arrays: block g of the whole tensor sits at
    // packed byte 16 g and scale byte 2 g, so the kernel indexes blocks linearly
    return w4a8::launch_requant(w4a8::SrcNvfp4{nv_packed, nv_scale_e4m3, global_divisor}, parts, N, K, mode,
                                out_packed, out_e8m0, err_ssq, stream);
}

extern "C" w4a8_status fp8_channel_to_mxfp4_requant(const uint8_t *w_e4m3, const float *row_scale, int64_t N,
                                                    int64_t K, int mode, uint8_t *out_packed,
                                                    uint8_t *out_e8m0, double *err_ssq, cudaStream_t stream)
{
    if (N < 0 || K < 0 || mode < 0 || mode > 2) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || K == 0) return W4A8_OK;
    if (!w_e4m3 || !row_scale || !out_packed || !out_e8m0) return W4A8_ERR_INVALID_ARG;
    if (!w4a8_aligned(w_e4m3, 16) || !w4a8_aligned(out_packed, 16) || !w4a8_aligned(row_scale, 4) ||
        (err_ssq && !w4a8_aligned(err_ssq, 8)))
        return W4A8_ERR_MISALIGNED;
    return w4a8::launch_requant(w4a8::SrcFp8Channel{w_e4m3, row_scale}, w4a8::one_partition(N), N, K, mode,
                                out_packed, out_e8m0, err_ssq, stream);
}

extern "C" w4a8_status bf16_to_mxfp4_requant(const uint16_t *w_bf16, int64_t N, int64_t K, int mode,
                                             uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq,
                                             cudaStream_t stream)
{
    if (N < 0 || K < 0 || mode < 0 || mode > 2) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (N == 0 || K == 0) return W4A8_OK;
    if (!w_bf16 || !out_packed || !out_e8m0) return W4A8_ERR_INVALID_ARG;
    if (!w4a8_aligned(w_bf16, 16) || !w4a8_aligned(out_packed, 16) || (err_ssq && !w4a8_aligned(err_ssq, 8)))
        return W4A8_ERR_MISALIGNED;
    return w4a8::launch_requant(w4a8::SrcBf16{w_bf16}, w4a8::one_partition(N), N, K, mode, out_packed, out_e8m0,
                                err_ssq, stream);
}

// W4A4 activation quant ("vllm-radiance (MXFP4)", section "Native MXFP4": MXFP4 activations,
// group 32, e8m0): each token row of x by the OCP rule ("radiance_nvfp4.py", _block_exponent
// "ocp", _encode_blocks), i.e. the bf16 source of the requant kernel in ocp mode without the
// error sums.
extern "C" w4a8_status w4a4_act_quant(const uint16_t *x_bf16, uint8_t *xa_packed, uint8_t *xa_e8m0, int64_t M,
                                      int64_t K, cudaStream_t stream)
{
    return bf16_to_mxfp4_requant(x_bf16, M, K, 0, xa_packed, xa_e8m0, nullptr, stream);
}
