// act_quant.cu -- per-token dynamic fp8 (e4m3) activation quant.
//
// "radiance_autoround.py", autoround_linear: each token's activations are cast to fp8 with a
// dynamic per-token scale before the GEMM; the scale is amax / 448 so the row maximum maps to
// the largest e4m3 magnitude, and codes are rounded to nearest even.
//
// One CTA per row.  Pass 1 streams the row with 16-byte loads and takes the amax on the bf16
// bit patterns (|x| ordering equals the ordering of the 15 low bits for finite values), warp
// shuffles then shared memory reduce it; pass 2 re-reads the row (now in L1/L2, so HBM sees it
// once), divides each element by the scale with a correctly rounded fp32 division and packs
// eight e4m3 codes per 8-byte store.  HBM-bound: 2 bytes read + 1 byte written per element.
#include "common.cuh"

namespace w4a8 {

constexpr int AQ_THREADS = 256;

__global__ void __launch_bounds__(AQ_THREADS)
act_quant_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ xq,
                 float *__restrict__ x_scale, int64_t K)
{
    // a GEMM launched after this kernel with programmatic dependent launch may start its own
    // set-up now; it waits for this grid to finish before it reads xq or x_scale
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
    const int nchunk = (int)(K / 8);

    uint32_t amax2 = 0;  // two 15-bit magnitudes packed, per-halfword max
    for (int c = threadIdx.x; c < nchunk; c += AQ_THREADS) {
        uint4 v = __ldg(row + c);
        amax2 = __vmaxu2(amax2, v.x & 0x7fff7fffu);
        amax2 = __vmaxu2(amax2, v.y & 0x7fff7fffu);
        amax2 = __vmaxu2(amax2, v.z & 0x7fff7fffu);
        amax2 = __vmaxu2(amax2, v.w & 0x7fff7fffu);
    }
    uint32_t hb = max(amax2 & 0xffffu, amax2 >> 16);
    float amax = bf16_bits_to_float(hb);
    amax = warp_max(amax);
    __shared__ float red[AQ_THREADS / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < AQ_THREADS / 32 ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    amax = red[0];
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0) x_scale[m] = s;

    uint2 *out = reinterpret_cast<uint2 *>(xq + m * K);
    for (int c = threadIdx.x; c < nchunk; c += AQ_THREADS) {
        uint4 v = row[c];
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float lo = __fdiv_rn(bf16_bits_to_float(w[j] & 0xffffu), s);
            float hi = __fdiv_rn(bf16_bits_to_float(w[j] >> 16), s);
            q[j] = float2_to_e4m3x2(lo, hi);
        }
        out[c] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
    }
}

}  // namespace w4a8

extern "C" w4a8_status w4a8_act_quant(const uint16_t *x_bf16, uint8_t *xq, float *x_scale,
                                      int64_t M, int64_t K, cudaStream_t stream)
{
    if (M < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0) return W4A8_OK;
    if (!x_bf16 || !xq || !x_scale || K == 0) return W4A8_ERR_INVALID_ARG;
    if (K % 8 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(x_bf16, 16) || !w4a8_aligned(xq, 8) || !w4a8_aligned(x_scale, 4))
        return W4A8_ERR_MISALIGNED;
    if (M > 0x7fffffffLL) return W4A8_ERR_UNSUPPORTED_SHAPE;
    w4a8::act_quant_kernel<<<(unsigned)M, w4a8::AQ_THREADS, 0, stream>>>(x_bf16, xq, x_scale, K);
    return w4a8_launch_status();
}
