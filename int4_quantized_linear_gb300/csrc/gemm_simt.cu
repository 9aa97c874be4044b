// gemm_simt.cu -- CUDA-core W4A8 GEMMs (MXFP4 and int4 group-128).
//
// The general-shape kernels: any M, K a multiple of 32 (MXFP4) or 128 (int4), no alignment
// beyond 16 bytes.  The tensor-core kernels in gemm_tc.cu take the shapes their TMA tiles
// allow; these take the rest, and serve as the second implementation the tests compare.
//
// MXFP4 ("vllm-radiance (MXFP4)", "The W4A8 fp8-WMMA kernel"): one warp per weight row n and
// up to MT tokens; lane l walks the 32-blocks l, l+32, ... of the row, so each weight byte is
// read once per MT tokens with 16-byte loads.  Per 32-block the e2m1 x e4m3 products are
// summed in fp32 and the block's power-of-two scale is applied once (the e8m0 "fold").
//
// int4 ("radiance_autoround.py", module docstring / _exact_ref): one thread per output column
// n and up to MT tokens; a warp reads 32 consecutive qweight words of one K/8 row (128
// coalesced bytes of the checkpoint's [K/8, N] layout).  Per 128-group the (c - z) x e4m3
// products are summed in fp32 and multiplied by the group's fp16 scale; z = 8, or for the
// asymmetric format ("vllm-radiance (MXFP4)", ParoQuant) 1 + the column's qzeros nibble.
#include "common.cuh"

namespace w4a8 {

constexpr int SIMT_MT = 8;

template <int MT>
__global__ void __launch_bounds__(256)
mxfp4_simt_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ x_scale,
                  const uint8_t *__restrict__ wp, const uint8_t *__restrict__ we,
                  uint16_t *__restrict__ out, int64_t M, int64_t N, int64_t K)
{
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    if (n >= N) return;
    const int64_t KB = K / 32;
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
    for (int64_t b = lane; b < KB; b += 32) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(wp + n * (K / 2) + b * 16));
        const float sw = exp2i((int)we[n * KB + b] - 127);
        float w[32];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float2 f = e2m1x2_to_float2((ww[j >> 2] >> (8 * (j & 3))) & 0xffu);
            w[2 * j] = f.x;
            w[2 * j + 1] = f.y;
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (m0 + t < M) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(xq + (m0 + t) * K + b * 32);
                const uint4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
                const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                float part = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float2 a = e4m3x2_to_float2((uint16_t)(xw[j] & 0xffffu));
                    float2 c = e4m3x2_to_float2((uint16_t)(xw[j] >> 16));
                    part = fmaf(a.x, w[4 * j], part);
                    part = fmaf(a.y, w[4 * j + 1], part);
                    part = fmaf(c.x, w[4 * j + 2], part);
                    part = fmaf(c.y, w[4 * j + 3], part);
                }
                acc[t] = fmaf(part, sw, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        float v = warp_sum(acc[t]);
        if (lane == 0 && m0 + t < M) out[(m0 + t) * N + n] = float_to_bf16_bits(v * x_scale[m0 + t]);
    }
}

// W4A4 ("vllm-radiance (MXFP4)", section "Native MXFP4"): the same walk with MXFP4 activations
// (e2m1 codes [M, K/2] and e8m0 [M, K/32]); per 32-block the e2m1 x e2m1 products are summed in
// fp32 and both blocks' power-of-two scales applied once.
template <int MT>
__global__ void __launch_bounds__(256)
mxfp4_a4_simt_kernel(const uint8_t *__restrict__ xa, const uint8_t *__restrict__ xe,
                     const uint8_t *__restrict__ wp, const uint8_t *__restrict__ we,
                     uint16_t *__restrict__ out, int64_t M, int64_t N, int64_t K)
{
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    if (n >= N) return;
    const int64_t KB = K / 32;
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
    for (int64_t b = lane; b < KB; b += 32) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(wp + n * (K / 2) + b * 16));
        const float sw = exp2i((int)we[n * KB + b] - 127);
        float w[32];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float2 f = e2m1x2_to_float2((ww[j >> 2] >> (8 * (j & 3))) & 0xffu);
            w[2 * j] = f.x;
            w[2 * j + 1] = f.y;
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            if (m0 + t < M) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(xa + (m0 + t) * (K / 2) + b * 16));
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float part = 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 a = e2m1x2_to_float2((xw[j >> 2] >> (8 * (j & 3))) & 0xffu);
                    part = fmaf(a.x, w[2 * j], part);
                    part = fmaf(a.y, w[2 * j + 1], part);
                }
                acc[t] = fmaf(part, sw * exp2i((int)xe[(m0 + t) * KB + b] - 127), acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        float v = warp_sum(acc[t]);
        if (lane == 0 && m0 + t < M) out[(m0 + t) * N + n] = float_to_bf16_bits(v);
    }
}

template <int MT>
__global__ void __launch_bounds__(128)
int4_simt_kernel(const uint8_t *__restrict__ xq, const float *__restrict__ x_scale,
                 const uint32_t *__restrict__ qw, const uint16_t *__restrict__ s16,
                 const uint32_t *__restrict__ qz, const uint8_t *__restrict__ qh,
                 const uint8_t *__restrict__ z5, uint16_t *__restrict__ out, int64_t M, int64_t N, int64_t K)
{
    const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.y * MT;
    if (n >= N) return;
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
    for (int64_t g = 0; g < K / 128; ++g) {
        float part[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) part[t] = 0.0f;
        // int4: zero point 8, or (asymmetric) 1 + the column's nibble of the group's qzeros word;
        // int5 (fifth-bit plane qh): zero point 16, or the column's byte of the group's zeros
        const int z = qh ? (z5 ? (int)__ldg(z5 + g * N + n) : 16)
                         : qz ? 1 + (int)((__ldg(qz + g * ((N + 7) / 8) + n / 8) >> (4 * (n & 7))) & 0xfu) : 8;
        for (int i = 0; i < 16; ++i) {
            const uint32_t word = __ldg(qw + (g * 16 + i) * N + n);
            const uint32_t hb = qh ? (uint32_t)__ldg(qh + (g * 16 + i) * N + n) : 0u;
            float w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                w[j] = (float)((int)((word >> (4 * j)) & 0xfu) + 16 * (int)((hb >> j) & 1u) - z);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (m0 + t < M) {
                    const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xq + (m0 + t) * K + g * 128 + 8 * i));
                    float2 a = e4m3x2_to_float2((uint16_t)(xv.x & 0xffffu));
                    float2 b = e4m3x2_to_float2((uint16_t)(xv.x >> 16));
                    float2 c = e4m3x2_to_float2((uint16_t)(xv.y & 0xffffu));
                    float2 d = e4m3x2_to_float2((uint16_t)(xv.y >> 16));
                    float p = part[t];
                    p = fmaf(a.x, w[0], p); p = fmaf(a.y, w[1], p);
                    p = fmaf(b.x, w[2], p); p = fmaf(b.y, w[3], p);
                    p = fmaf(c.x, w[4], p); p = fmaf(c.y, w[5], p);
                    p = fmaf(d.x, w[6], p); p = fmaf(d.y, w[7], p);
                    part[t] = p;
                }
            }
        }
        const float s = __half2float(__ushort_as_half(s16[g * N + n]));
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = fmaf(s, part[t], acc[t]);
    }
#pragma unroll
    for (int t = 0; t < MT; ++t)
        if (m0 + t < M) out[(m0 + t) * N + n] = float_to_bf16_bits(acc[t] * x_scale[m0 + t]);
}

}  // namespace w4a8

w4a8_status w4a8_launch_mxfp4_simt(const uint8_t *xq, const float *x_scale, const uint8_t *wp,
                                   const uint8_t *we, uint16_t *out, int64_t M, int64_t N,
                                   int64_t K, cudaStream_t stream)
{
    dim3 grid((unsigned)((N + 7) / 8), (unsigned)((M + w4a8::SIMT_MT - 1) / w4a8::SIMT_MT));
    if (grid.y > 65535u) return W4A8_ERR_UNSUPPORTED_SHAPE;
    w4a8::mxfp4_simt_kernel<w4a8::SIMT_MT><<<grid, 256, 0, stream>>>(xq, x_scale, wp, we, out, M, N, K);
    return w4a8_launch_status();
}

w4a8_status w4a8_launch_int4_simt(const uint8_t *xq, const float *x_scale, const int32_t *qw,
                                  const uint16_t *s16, uint16_t *out, int64_t M, int64_t N,
                                  int64_t K, cudaStream_t stream, const int32_t *qzeros,
                                  const uint8_t *qhigh, const uint8_t *zeros5)
{
    dim3 grid((unsigned)((N + 127) / 128), (unsigned)((M + w4a8::SIMT_MT - 1) / w4a8::SIMT_MT));
    if (grid.y > 65535u) return W4A8_ERR_UNSUPPORTED_SHAPE;
    w4a8::int4_simt_kernel<w4a8::SIMT_MT><<<grid, 128, 0, stream>>>(
        xq, x_scale, reinterpret_cast<const uint32_t *>(qw), s16, reinterpret_cast<const uint32_t *>(qzeros), qhigh, zeros5,
        out, M, N, K);
    return w4a8_launch_status();
}

w4a8_status w4a8_launch_mxfp4_a4_simt(const uint8_t *xa, const uint8_t *xe, const uint8_t *wp, const uint8_t *we,
                                      uint16_t *out, int64_t M, int64_t N, int64_t K, cudaStream_t stream)
{
    dim3 grid((unsigned)((N + 7) / 8), (unsigned)((M + w4a8::SIMT_MT - 1) / w4a8::SIMT_MT));
    if (grid.y > 65535u) return W4A8_ERR_UNSUPPORTED_SHAPE;
    w4a8::mxfp4_a4_simt_kernel<w4a8::SIMT_MT><<<grid, 256, 0, stream>>>(xa, xe, wp, we, out, M, N, K);
    return w4a8_launch_status();
}
