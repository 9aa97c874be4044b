// noalloc.cu -- an MXFP4 linear entry point for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code that is being captured into
// a CUDA graph (cudaMalloc is not a stream operation and must not run during capture), serving
// engines that reserve all device memory in their own pool up front and forbid allocations
// outside it, and plugin interfaces that pass only input and output pointers.  This entry point
// runs the tensor-core MXFP4 GEMM with its stream-K scratch (fp32 partial tiles and arrival
// counters) in a fixed-size array that lives in the library's device image instead of a
// caller-provided workspace.  Every GPU that loads the library holds the array until exit.
#include "common.cuh"
#include "dispatch.h"

// Upper bound of the scratch: enough for the decode band (up to 64 tokens) on GPUs with up to
// 160 SMs and output widths up to a few hundred thousand columns.
#define W4A8_NOALLOC_SCRATCH_BYTES (12u << 20)

static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A8_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array for the current device.  The array's name is only a
// host-side handle; the address must come from cudaGetSymbolAddress, once per device, with that
// device current.
static void *noalloc_scratch_ptr()
{
    static void *ptr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ptr[dev] = p;
    }
    return ptr[dev];
}

extern "C" size_t w4a8_noalloc_scratch_bytes(void) { return W4A8_NOALLOC_SCRATCH_BYTES; }

extern "C" w4a8_status w4a8_mxfp4_linear_noalloc(const uint8_t *xq, const float *x_scale,
                                                 const uint8_t *w_packed, const uint8_t *w_e8m0,
                                                 uint16_t *out_bf16, int64_t M, int64_t N,
                                                 int64_t K, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return W4A8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A8_OK;
    if (K == 0 || !xq || !x_scale || !w_packed || !w_e8m0 || !out_bf16) return W4A8_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4A8_ERR_UNSUPPORTED_SHAPE;
    if (!w4a8_aligned(xq, 16) || !w4a8_aligned(w_packed, 16) || !w4a8_aligned(x_scale, 4) ||
        !w4a8_aligned(out_bf16, 2))
        return W4A8_ERR_MISALIGNED;
    const int policy = w4a8_gemm_policy();
    if (policy == 1 || !w4a8_tc_mxfp4_supported(xq, w_packed, w_e8m0, out_bf16, M, N, K))
        return w4a8_launch_mxfp4_simt(xq, x_scale, w_packed, w_e8m0, out_bf16, M, N, K, stream);
    const size_t need = w4a8_tc_workspace_bytes(M, N, K, policy);
    if (need > W4A8_NOALLOC_SCRATCH_BYTES) return W4A8_ERR_WORKSPACE;
    void *scratch = noalloc_scratch_ptr();
    if (!scratch) return W4A8_ERR_CUDA;
    // The arrival counters sit after the partial tiles and must start at zero; a call that gave
    // up part-way could have left some set, so clear them (a small memset, not an allocation).
    const size_t counters_off = w4a8_tc_workspace_counters_offset(M, N, K);
    if (need > counters_off &&
        cudaMemsetAsync(static_cast<unsigned char *>(scratch) + counters_off, 0, need - counters_off, stream) !=
            cudaSuccess)
        return W4A8_ERR_CUDA;
    return w4a8_launch_mxfp4_tc(xq, x_scale, w_packed, w_e8m0, out_bf16, M, N, K, scratch, policy, false,
                                stream);
}
