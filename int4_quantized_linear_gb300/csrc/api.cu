// api.cu -- argument validation and kernel dispatch for the GEMM entry points, the status
// strings, the kernel-selection policy and the device status word of the bounded waits.
//
// Dispatch ("vllm-radiance (MXFP4)", "The W4A8 fp8-WMMA kernel": a prefill tiling and a decode
// tiling, chosen inside the native call so no shape branch is visible to the caller;
// "radiance_autoround.py", autoround_linear: the prefill/decode choice is made natively).
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "dispatch.h"

static std::atomic<int> g_policy{0};

// Device status word written by bounded waits that give up (0 = clean).
__device__ unsigned int g_w4a8_device_status[4] = {0, 0, 0, 0};

struct W4a8SymbolCache {
    std::mutex mu;
    void *ctx[64] = {nullptr};
    void *addr[64] = {nullptr};
};

W4a8SymbolCache *w4a8_symbol_cache_new() { return new W4a8SymbolCache(); }

// cuCtxGetCurrent through the runtime's driver entry point (the library links no libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
static CtxGetCurrentFn ctx_get_current()
{
    static std::atomic<CtxGetCurrentFn> fn{nullptr};
    CtxGetCurrentFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<CtxGetCurrentFn>(p);
            fn.store(f, std::memory_order_release);
        }
    }
    return f;
}

void *w4a8_symbol_address(const void *symbol, W4a8SymbolCache *cache)
{
    int dev = 0;
    if (!cache || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
    if (!ctx) {
        // no context on this thread yet: the runtime call makes the device's primary context
        // current (the address it returns is then the one launches from this thread use)
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    }
    std::lock_guard<std::mutex> lock(cache->mu);
    if (cache->ctx[dev] != (void *)ctx || !cache->addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
        cache->addr[dev] = p;
        cache->ctx[dev] = (void *)ctx;
    }
    return cache->addr[dev];
}

unsigned int *w4a8_device_status_ptr()
{
    static W4a8SymbolCache *cache = w4a8_symbol_cache_new();
    return static_cast<unsigned int *>(w4a8_symbol_address((const void *)&g_w4a8_device_status, cache));
}

int w4a8_gemm_policy() { return g_policy.load(std::memory_order_relaxed); }

#ifdef W4A8_TRACE
// Development aid: a device buffer for the tensor-core kernels' pipeline timestamps (see the
// trace helpers in gemm_tc.cu); only builds with W4A8_TRACE defined have the setter.
static std::atomic<void *> g_trace{nullptr};
void *w4a8_debug_trace_ptr() { return g_trace.load(std::memory_order_relaxed); }
extern "C" W4A8_API void w4a8_debug_set_trace(void *device_buffer) { g_trace.store(device_buffer, std::memory_order_relaxed); }
#else
void *w4a8_debug_trace_ptr() { return nullptr; }
#endif

extern "C" void w4a8_set_gemm_policy(int policy) { g_policy.store(policy, std::memory_order_relaxed); }

extern "C" int w4a8_decode_max_m(void) { return W4A8_DECODE_MAX_M; }

extern "C" const char *w4a8_status_string(w4a8_status s)
{
    switch (s) {
    case W4A8_OK: return "W4A8_OK";
    case W4A8_ERR_INVALID_ARG: return "W4A8_ERR_INVALID_ARG";
    case W4A8_ERR_UNSUPPORTED_SHAPE: return "W4A8_ERR_UNSUPPORTED_SHAPE";
    case W4A8_ERR_MISALIGNED: return "W4A8_ERR_MISALIGNED";
    case W4A8_ERR_WORKSPACE: return "W4A8_ERR_WORKSPACE";
    case W4A8_ERR_CUDA: return "W4A8_ERR_CUDA";
    case W4A8_ERR_TIMEOUT: return "W4A8_ERR_TIMEOUT";
    }
    return "W4A8_ERR_UNKNOWN";
}

extern "C" w4a8_status w4a8_check_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return W4A8_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4a8_device_status, sizeof(v)) != cudaSuccess) return W4A8_ERR_CUDA;
    if (v) {
        unsigned int z[4] = {0, 0, 0, 0};
        if (cudaMemcpyToSymbol(g_w4a8_device_status, z, sizeof(z)) != cudaSuccess) return W4A8_ERR_CUDA;
        return W4A8_ERR_TIMEOUT;
    }
    return W4A8_OK;
}

extern "C" int w4a8_debug_status_words(unsigned int *out4)
{
    unsigned int z[4] = {0, 0, 0, 0};
    if (!out4) return W4A8_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return W4A8_ERR_CUDA;
    if (cudaMemcpyFromSymbol(out4, g_w4a8_device_status, sizeof(z)) != cudaSuccess) return W4A8_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_w4a8_device_status, z, sizeof(z)) != cudaSuccess) return W4A8_ERR_CUDA;
    return W4A8_OK;
}

// Workspace sizes are the largest any kernel choice needs for the shape (the CUDA-core kernels
// need none), so a size queried under one kernel-selection policy stays valid under another.
extern "C" size_t w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return w4a8_tc_workspace_bytes(M, N, K);
}

extern "C" size_t w4a8_int4g128_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return w4a8_tc_int4_workspace_bytes(M, N, K);
}

extern "C" w4a8_status w4a8_mxfp4_linear(const uint8_t *xq, const float *x_scale,
                                         const uint8_t *w_packed, const uint8_t *w_e8m0,
                                         uint16_t *out_bf16, int64_t M, int64_t N, int64_t K,
                                         void *workspace, size_t workspace_bytes,
                                         cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !xq || !x_scale || !w_packed || !w_e8m0 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(xq, 16) || !w4a8_aligned(w_packed, 16) || !w4a8_aligned(x_scale, 4) ||
        !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    const int policy = w4a8_gemm_policy();
    if (policy != 1 && w4a8_tc_mxfp4_supported(xq, w_packed, w_e8m0, out_bf16, M, N, K)) {
        const size_t need = w4a8_tc_workspace_bytes(M, N, K);
        if (need && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
        if (need && !w4a8_aligned(workspace, 16)) return W4A8_ERR_MISALIGNED;
        return w4a8_launch_mxfp4_tc(xq, x_scale, w_packed, w_e8m0, out_bf16, M, N, K, workspace,
                                    policy, false, stream);
    }
    return w4a8_launch_mxfp4_simt(xq, x_scale, w_packed, w_e8m0, out_bf16, M, N, K, stream);
}

// Workspace of the fused entry: the GEMM's scratch first (its arrival counters at offset 0 for
// every shape; the counter region is kept even when the GEMM needs no scratch, so the
// activations never land on it), then the quantized activations and their scales, each part
// starting on a 256-byte boundary.
static size_t round256(size_t b) { return (b + 255) & ~size_t(255); }
static size_t gemm_part(int64_t M, int64_t N, int64_t K)
{
    return round256(std::max(w4a8_workspace_bytes(M, N, K), W4A8_COUNTER_BYTES));
}

extern "C" size_t w4a8_mxfp4_linear_bf16_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return gemm_part(M, N, K) + round256((size_t)M * (size_t)K) + round256((size_t)M * 4);
}

extern "C" w4a8_status w4a8_mxfp4_linear_bf16(const uint16_t *x_bf16, const uint8_t *w_packed,
                                              const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M,
                                              int64_t N, int64_t K, void *workspace,
                                              size_t workspace_bytes, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !x_bf16 || !w_packed || !w_e8m0 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0 || M > 0x7fffffffLL) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(x_bf16, 16) || !w4a8_aligned(w_packed, 16) || !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    const size_t need = w4a8_mxfp4_linear_bf16_workspace_bytes(M, N, K);
    if (!workspace || workspace_bytes < need) return W4A8_ERR_WORKSPACE;
    if (!w4a8_aligned(workspace, 256)) return W4A8_ERR_MISALIGNED;
    uint8_t *gws = static_cast<uint8_t *>(workspace);
    const size_t gws_bytes = gemm_part(M, N, K);
    uint8_t *xq = gws + gws_bytes;
    float *xs = reinterpret_cast<float *>(xq + round256((size_t)M * (size_t)K));

    const int policy = w4a8_gemm_policy();
    w4a8_status st = w4a8_launch_act_quant(x_bf16, xq, xs, M, K, stream);
    if (st != W4A8_OK) return st;
    if (policy != 1 && w4a8_tc_mxfp4_supported(xq, w_packed, w_e8m0, out_bf16, M, N, K)) {
        const size_t g_need = w4a8_tc_workspace_bytes(M, N, K);
        if (g_need > gws_bytes) return W4A8_ERR_WORKSPACE;
        // the GEMM directly follows the activation quant: it may fetch weights before waiting
        return w4a8_launch_mxfp4_tc(xq, xs, w_packed, w_e8m0, out_bf16, M, N, K, gws, policy, true, stream);
    }
    return w4a8_launch_mxfp4_simt(xq, xs, w_packed, w_e8m0, out_bf16, M, N, K, stream);
}

// The same linear as one kernel: the GEMM quantizes the activations itself.  Same arguments and
// workspace layout as w4a8_mxfp4_linear_bf16; only the GEMM-scratch part of the workspace is used.
extern "C" w4a8_status w4a8_mxfp4_linear_bf16_single(const uint16_t *x_bf16, const uint8_t *w_packed,
                                                     const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M,
                                                     int64_t N, int64_t K, void *workspace,
                                                     size_t workspace_bytes, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !x_bf16 || !w_packed || !w_e8m0 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0 || !w4a8_tc_mxfp4_aq_takes(M, K)) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(x_bf16, 16) || !w4a8_aligned(w_packed, 16) || !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    if (!w4a8_tc_mxfp4_supported(x_bf16, w_packed, w_e8m0, out_bf16, M, N, K)) return W4A8_ERR_UNSUPPORTED_SHAPE;
    const size_t need = w4a8_mxfp4_linear_bf16_workspace_bytes(M, N, K);
    if (!workspace || workspace_bytes < need) return W4A8_ERR_WORKSPACE;
    if (!w4a8_aligned(workspace, 256)) return W4A8_ERR_MISALIGNED;
    return w4a8_launch_mxfp4_tc_aq(x_bf16, w_packed, w_e8m0, out_bf16, M, N, K, workspace, stream);
}

static w4a8_status int4g128_linear_impl(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                                       const uint16_t *scales_fp16, const int32_t *qzeros, uint16_t *out_bf16,
                                       int64_t M, int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                                       cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !xq || !x_scale || !qweight || !scales_fp16 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 128 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(xq, 16) || !w4a8_aligned(qweight, 4) || !w4a8_aligned(scales_fp16, 2) ||
        !w4a8_aligned(x_scale, 4) || !w4a8_aligned(out_bf16, 2) || (qzeros && !w4a8_aligned(qzeros, 4)))
        return W4A8_ERR_MISALIGNED;
    const int policy = w4a8_gemm_policy();
    if (policy != 1 && w4a8_tc_int4_supported(xq, qweight, scales_fp16, out_bf16, M, N, K)) {
        const size_t need = w4a8_tc_int4_workspace_bytes(M, N, K);
        if (need && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
        if (need && !w4a8_aligned(workspace, 16)) return W4A8_ERR_MISALIGNED;
        return w4a8_launch_int4_tc(xq, x_scale, qweight, scales_fp16, out_bf16, M, N, K, workspace, policy,
                                   stream, qzeros);
    }
    return w4a8_launch_int4_simt(xq, x_scale, qweight, scales_fp16, out_bf16, M, N, K, stream, qzeros);
}

extern "C" w4a8_status w4a8_int4g128_linear(const uint8_t *xq, const float *x_scale,
                                            const int32_t *qweight, const uint16_t *scales_fp16,
                                            uint16_t *out_bf16, int64_t M, int64_t N, int64_t K,
                                            void *workspace, size_t workspace_bytes,
                                            cudaStream_t stream)
{
    return int4g128_linear_impl(xq, x_scale, qweight, scales_fp16, nullptr, out_bf16, M, N, K, workspace,
                                workspace_bytes, stream);
}

extern "C" w4a8_status w4a8_int4g128_asym_linear(const uint8_t *xq, const float *x_scale,
                                                 const int32_t *qweight, const uint16_t *scales_fp16,
                                                 const int32_t *qzeros, uint16_t *out_bf16, int64_t M,
                                                 int64_t N, int64_t K, void *workspace,
                                                 size_t workspace_bytes, cudaStream_t stream)
{
    if (!qzeros) return W4A8_ERR_INVALID_ARG;
    return int4g128_linear_impl(xq, x_scale, qweight, scales_fp16, qzeros, out_bf16, M, N, K, workspace,
                                workspace_bytes, stream);
}

extern "C" size_t w4a8_int5g128_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    // the int5 kernel shares the int4 kernel's work split and partial-tile scratch
    return w4a8_int4g128_workspace_bytes(M, N, K);
}

extern "C" w4a8_status w4a8_int5g128_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                                            const uint8_t *qhigh, const uint16_t *scales_fp16,
                                            const uint8_t *zeros, uint16_t *out_bf16, int64_t M, int64_t N,
                                            int64_t K, void *workspace, size_t workspace_bytes,
                                            cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !xq || !x_scale || !qweight || !qhigh || !scales_fp16 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 128 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(xq, 16) || !w4a8_aligned(qweight, 4) || !w4a8_aligned(scales_fp16, 2) ||
        !w4a8_aligned(x_scale, 4) || !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    const int policy = w4a8_gemm_policy();
    if (policy != 1 && w4a8_tc_int5_supported(xq, qweight, qhigh, scales_fp16, out_bf16, M, N, K)) {
        const size_t need = w4a8_tc_int4_workspace_bytes(M, N, K);
        if (need && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
        if (need && !w4a8_aligned(workspace, 16)) return W4A8_ERR_MISALIGNED;
        return w4a8_launch_int5_tc(xq, x_scale, qweight, qhigh, scales_fp16, zeros, out_bf16, M, N, K, workspace,
                                   policy, stream);
    }
    return w4a8_launch_int4_simt(xq, x_scale, qweight, scales_fp16, out_bf16, M, N, K, stream, nullptr, qhigh,
                                 zeros);
}

extern "C" w4a8_status w4a4_mxfp4_linear(const uint8_t *xa_packed, const uint8_t *xa_e8m0, const uint8_t *w_packed,
                                         const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M, int64_t N, int64_t K,
                                         void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !xa_packed || !xa_e8m0 || !w_packed || !w_e8m0 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(xa_packed, 16) || !w4a8_aligned(w_packed, 16) || !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    const int policy = w4a8_gemm_policy();
    if (policy != 1 && w4a8_tc_mxfp4_a4_supported(xa_packed, xa_e8m0, w_packed, w_e8m0, out_bf16, M, N, K)) {
        const size_t need = w4a8_tc_workspace_bytes(M, N, K);
        if (need && (!workspace || workspace_bytes < need)) return W4A8_ERR_WORKSPACE;
        if (need && !w4a8_aligned(workspace, 16)) return W4A8_ERR_MISALIGNED;
        return w4a8_launch_mxfp4_a4_tc(xa_packed, xa_e8m0, w_packed, w_e8m0, out_bf16, M, N, K, workspace, policy,
                                       stream);
    }
    return w4a8_launch_mxfp4_a4_simt(xa_packed, xa_e8m0, w_packed, w_e8m0, out_bf16, M, N, K, stream);
}

// ------------------------------------------------------------------ kernel-path queries
// Each mirrors its entry point's validation and dispatch without launching anything.

static int path_of(bool valid, bool tensor_core)
{
    if (!valid) return 0;
    return (w4a8_gemm_policy() != 1 && tensor_core) ? W4A8_PATH_TENSOR_CORE : W4A8_PATH_CUDA_CORE;
}

extern "C" int w4a8_mxfp4_path(const void *xq, const void *w_packed, const void *w_e8m0, const void *out_bf16,
                               int64_t M, int64_t N, int64_t K)
{
    const bool valid = M > 0 && N > 0 && K > 0 && K % 32 == 0 && xq && w_packed && w_e8m0 && out_bf16 &&
                       w4a8_aligned(xq, 16) && w4a8_aligned(w_packed, 16) && w4a8_aligned(out_bf16, 2);
    return path_of(valid, valid && w4a8_tc_mxfp4_supported(xq, w_packed, w_e8m0, out_bf16, M, N, K));
}

extern "C" int w4a8_int4g128_path(const void *xq, const void *qweight, const void *scales_fp16,
                                  const void *out_bf16, int64_t M, int64_t N, int64_t K)
{
    const bool valid = M > 0 && N > 0 && K > 0 && K % 128 == 0 && xq && qweight && scales_fp16 && out_bf16 &&
                       w4a8_aligned(xq, 16) && w4a8_aligned(qweight, 4) && w4a8_aligned(scales_fp16, 2) &&
                       w4a8_aligned(out_bf16, 2);
    return path_of(valid, valid && w4a8_tc_int4_supported(xq, qweight, scales_fp16, out_bf16, M, N, K));
}

extern "C" int w4a8_int5g128_path(const void *xq, const void *qweight, const void *qhigh, const void *scales_fp16,
                                  const void *out_bf16, int64_t M, int64_t N, int64_t K)
{
    const bool valid = M > 0 && N > 0 && K > 0 && K % 128 == 0 && xq && qweight && qhigh && scales_fp16 &&
                       out_bf16 && w4a8_aligned(xq, 16) && w4a8_aligned(qweight, 4) &&
                       w4a8_aligned(scales_fp16, 2) && w4a8_aligned(out_bf16, 2);
    return path_of(valid, valid && w4a8_tc_int5_supported(xq, qweight, qhigh, scales_fp16, out_bf16, M, N, K));
}

extern "C" int w4a4_mxfp4_path(const void *xa_packed, const void *xa_e8m0, const void *w_packed,
                               const void *w_e8m0, const void *out_bf16, int64_t M, int64_t N, int64_t K)
{
    const bool valid = M > 0 && N > 0 && K > 0 && K % 32 == 0 && xa_packed && xa_e8m0 && w_packed && w_e8m0 &&
                       out_bf16 && w4a8_aligned(xa_packed, 16) && w4a8_aligned(w_packed, 16) &&
                       w4a8_aligned(out_bf16, 2);
    return path_of(valid,
                   valid && w4a8_tc_mxfp4_a4_supported(xa_packed, xa_e8m0, w_packed, w_e8m0, out_bf16, M, N, K));
}
