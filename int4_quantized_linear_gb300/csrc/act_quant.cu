// act_quant.cu -- per-token dynamic fp8 (e4m3) activation quant.
//
// "radiance_autoround.py", autoround_linear: each token's activations are cast to fp8 with a
// dynamic per-token scale before the GEMM; the scale is amax / 448 so the row maximum maps to
// the largest e4m3 magnitude, and codes are rounded to nearest even.
//
// Grid (M, S): S CTAs per row.  Every CTA of a row reads the whole row once (each thread keeps
// its 16-byte chunks in registers for rows up to AQ_THREADS * CACHE * 8 elements, CACHE 4, 12 or
// 16 by row length -- the smallest that holds the row keeps the registers down and the CTAs an SM
// can hold up; longer rows are re-read from L1/L2 for the second pass) and takes the amax on the bf16 bit patterns (|x|
// ordering equals the ordering of the 15 low bits for finite values), reduced by warp shuffles
// and shared memory; it then quantizes only its 1/S slice of the row: each element divided by the
// scale with a correctly rounded fp32 division, eight e4m3 codes per 8-byte store.  Splitting a
// row over S CTAs costs S reads of the row from L2 but spreads the divisions over S SMs, which
// for decode batches (a few rows) is what bounds the kernel's latency.
//
// Launched with programmatic dependent launch: the kernel first waits for the previous kernel
// in the stream (which may produce x, or still read xq / x_scale), and only then lets the next
// kernel start early.  So when that next kernel is the library's GEMM, everything before this
// kernel has completed by the time the GEMM starts, and it may fetch its weights before waiting
// for this kernel.
#include <algorithm>

#include "common.cuh"
#include "dispatch.h"

namespace w4a8 {

constexpr int AQ_THREADS = 256;

// Optional timeline (a development aid, compiled in only when W4A8_TRACE is defined): global timer
// stamps (ns) of every CTA c < 256 at trace[AQ_TRACE_OFF + 4 c + k], k = 0 entry, 1 past the wait
// on the previous kernel, 3 thread 0's share of the row loaded, 2 done.
constexpr int AQ_TRACE_OFF = 16384;
__device__ __forceinline__ void aq_stamp(unsigned long long *trace, int k)
{
#ifdef W4A8_TRACE
    const unsigned c = blockIdx.x * gridDim.y + blockIdx.y;
    if (trace != nullptr && c < 256 && threadIdx.x == 0) {
        unsigned long long ns;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
        trace[AQ_TRACE_OFF + 4 * c + k] = ns;
    }
#endif
}

// CACHE: chunks of 8 elements kept per thread (rows up to AQ_THREADS * CACHE * 8 read once)
template <int CACHE>
__global__ void __launch_bounds__(AQ_THREADS)
act_quant_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ xq,
                 float *__restrict__ x_scale, int64_t K, unsigned long long *trace)
{
    aq_stamp(trace, 0);
    const int64_t m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
    const int nchunk = (int)(K / 8);
    const bool cached = nchunk <= AQ_THREADS * CACHE;
    // While the previous kernel finishes, pull the row into L2: one prefetch per 128-byte line
    // (every 8th chunk, and the last chunk for a row that ends inside a line).  A prefetch returns
    // nothing to the kernel, so it is harmless even if that kernel is still writing x: every load
    // below comes after the wait and reads L2, where the final values land.
    for (int c = 8 * (int)threadIdx.x; c < nchunk + 7; c += 8 * AQ_THREADS)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + min(c, nchunk - 1)));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    aq_stamp(trace, 1);
    // this CTA's slice of the row's chunks
    const int c_lo = (int)((long long)nchunk * blockIdx.y / gridDim.y);
    const int c_hi = (int)((long long)nchunk * (blockIdx.y + 1) / gridDim.y);

    uint4 v[CACHE];
    uint32_t amax2 = 0;  // two 15-bit magnitudes packed, per-halfword max
    if (cached) {
        // every load of the row goes out before the first use: one round trip, not CACHE
#pragma unroll
        for (int i = 0; i < CACHE; ++i) {
            const int c = threadIdx.x + i * AQ_THREADS;
            v[i] = c < nchunk ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < CACHE; ++i) {
            amax2 = __vmaxu2(amax2, v[i].x & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, v[i].y & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, v[i].z & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, v[i].w & 0x7fff7fffu);
        }
    } else {
        for (int c = threadIdx.x; c < nchunk; c += AQ_THREADS) {
            const uint4 w = __ldg(row + c);
            amax2 = __vmaxu2(amax2, w.x & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, w.y & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, w.z & 0x7fff7fffu);
            amax2 = __vmaxu2(amax2, w.w & 0x7fff7fffu);
        }
    }
    aq_stamp(trace, 3);
    uint32_t hb = max(amax2 & 0xffffu, amax2 >> 16);
    float amax = bf16_bits_to_float(hb);
    amax = warp_max(amax);
    __shared__ float red[AQ_THREADS / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = threadIdx.x < AQ_THREADS / 32 ? red[threadIdx.x] : 0.0f;
        t = warp_max(t);
        if (threadIdx.x == 0) red[0] = t;
    }
    __syncthreads();
    amax = red[0];
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    if (threadIdx.x == 0 && blockIdx.y == 0) x_scale[m] = s;

    uint2 *out = reinterpret_cast<uint2 *>(xq + m * K);
    auto quant8 = [&](const uint4 &w) { return quant8_e4m3(w, s); };
    if (cached) {
#pragma unroll
        for (int i = 0; i < CACHE; ++i) {
            const int c = threadIdx.x + i * AQ_THREADS;
            if (c >= c_lo && c < c_hi) out[c] = quant8(v[i]);
        }
    } else {
        for (int c = c_lo + (int)threadIdx.x; c < c_hi; c += AQ_THREADS) out[c] = quant8(row[c]);
    }
    aq_stamp(trace, 2);
}

}  // namespace w4a8

w4a8_status w4a8_launch_act_quant(const uint16_t *x_bf16, uint8_t *xq, float *x_scale, int64_t M,
                                  int64_t K, cudaStream_t stream)
{
    // about 256 CTAs in all, at most 16 per row
    const int per_row = M >= 256 ? 1 : (int)std::min<int64_t>(16, (256 + M - 1) / M);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M, (unsigned)per_row);
    cfg.blockDim = dim3(w4a8::AQ_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the smallest register cache that holds the row (fewer registers, more CTAs per SM)
    unsigned long long *trace = static_cast<unsigned long long *>(w4a8_debug_trace_ptr());
    const cudaError_t e =
        K <= 8192 ? cudaLaunchKernelEx(&cfg, w4a8::act_quant_kernel<4>, x_bf16, xq, x_scale, K, trace)
        : K <= 24576 ? cudaLaunchKernelEx(&cfg, w4a8::act_quant_kernel<12>, x_bf16, xq, x_scale, K, trace)
                     : cudaLaunchKernelEx(&cfg, w4a8::act_quant_kernel<16>, x_bf16, xq, x_scale, K, trace);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return W4A8_ERR_CUDA;
    }
    return w4a8_launch_status();
}

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
    return w4a8_launch_act_quant(x_bf16, xq, x_scale, M, K, stream);
}
