// common.cuh -- small device helpers shared by the library's kernels (number formats,
// exact power-of-two arithmetic, warp reductions).  Nothing here is shared with the oracle.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/w4a8.h"

#define W4A8_DEVICE __device__ __forceinline__

namespace w4a8 {

// Two e4m3 codes (low byte = first element) -> two fp32 values, exact.
W4A8_DEVICE float2 e4m3x2_to_float2(uint16_t codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
    __half2 h = *reinterpret_cast<__half2 *>(&h2);
    return __half22float2(h);
}

// Two fp32 values -> two e4m3 codes (low byte = lo), round to nearest even, saturating at
// the largest finite magnitude 448.
W4A8_DEVICE uint16_t float2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight bf16 activations (a 16-byte chunk, low element first) -> their eight e4m3 codes for the
// per-token scale s: each x / s with a correctly rounded fp32 division, then round to nearest
// even with saturation at 448 ("radiance_autoround.py", autoround_linear: the dynamic per-token
// fp8 cast).  Shared by the activation-quant kernel and the GEMM's fused quant, so both produce
// the same bytes.
W4A8_DEVICE uint2 quant8_e4m3(const uint4 &w, float s)
{
    const uint32_t h[4] = {w.x, w.y, w.z, w.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        q[j] = float2_to_e4m3x2(__fdiv_rn(__uint_as_float(h[j] << 16), s),
                                __fdiv_rn(__uint_as_float(h[j] & 0xffff0000u), s));
    return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// The same for four bf16 activations (8 bytes) -> four e4m3 codes, low byte first.
W4A8_DEVICE uint32_t quant4_e4m3(const uint2 &w, float s)
{
    const uint32_t lo = float2_to_e4m3x2(__fdiv_rn(__uint_as_float(w.x << 16), s),
                                         __fdiv_rn(__uint_as_float(w.x & 0xffff0000u), s));
    const uint32_t hi = float2_to_e4m3x2(__fdiv_rn(__uint_as_float(w.y << 16), s),
                                         __fdiv_rn(__uint_as_float(w.y & 0xffff0000u), s));
    return lo | (hi << 16);
}

// Two e2m1 codes in one byte (low nibble = first element) -> two fp32 values, exact.
W4A8_DEVICE float2 e2m1x2_to_float2(uint32_t byte)
{
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
    __half2 h = *reinterpret_cast<__half2 *>(&h2);
    return __half22float2(h);
}

// 2^e as an fp32 value, exact for e in [-149, 127].
W4A8_DEVICE float exp2i(int e)
{
    if (e >= -126) return __int_as_float((e + 127) << 23);
    return __int_as_float(1u << (e + 149));
}

W4A8_DEVICE float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

W4A8_DEVICE uint16_t float_to_bf16_bits(float f)
{
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}

W4A8_DEVICE float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

W4A8_DEVICE float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

W4A8_DEVICE double warp_sum_d(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace w4a8

static inline bool w4a8_aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Launch status helper: converts the last launch error into a status.
static inline w4a8_status w4a8_launch_status()
{
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return W4A8_OK;
}
