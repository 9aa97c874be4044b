// noalloc.cu -- an MXFP4 linear entry point for callers that cannot allocate device memory.
//
// The regular entry point takes a caller-provided workspace for its split-K scratch.  Some
// callers have no way to provide one: serving engines that reserve all device memory for their
// own pool up front and treat any allocation outside it as an error (it could fail, or push the
// process past its memory budget), and plugin or custom-operator interfaces that hand a kernel
// only its input and output pointers.  This entry point runs the same tensor-core MXFP4 GEMM
// with its stream-K scratch (fp32 partial tiles and arrival counters) in a fixed-size array in
// the library's device image.  Every GPU that loads the library holds that array until the
// process exits.
#include <algorithm>
#include "common.cuh"
#include "dispatch.h"

// Upper bound of the scratch: enough for the decode band (up to 64 tokens) on GPUs with up to
// 160 SMs and output widths up to a few hundred thousand columns.
#define W4A8_NOALLOC_SCRATCH_BYTES (12u << 20)

static __device__ __align__(256) unsigned char g_noalloc_scratch[W4A8_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code the array's name is
// only a host-side stand-in, never a device address: a kernel given it would fault or, where the
// GPU can reach host memory, silently use the wrong memory.  The address comes from
// cudaGetSymbolAddress with the device current, looked up on the first call on each device
// (and again if the device's context changed since, e.g. after a device reset).
static void *noalloc_scratch_ptr()
{
    static W4a8SymbolCache *cache = w4a8_symbol_cache_new();
    return w4a8_symbol_address((const void *)&g_noalloc_scratch, cache);
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
    const size_t need = w4a8_tc_workspace_bytes(M, N, K);
    if (need > W4A8_NOALLOC_SCRATCH_BYTES) return W4A8_ERR_WORKSPACE;
    void *scratch = noalloc_scratch_ptr();
    if (!scratch) return W4A8_ERR_CUDA;
    // The arrival counters open the scratch and must start at zero; a call that gave up part-way
    // could have left some set, so clear them (a small memset, not an allocation).
    if (cudaMemsetAsync(scratch, 0, std::min(need, W4A8_COUNTER_BYTES), stream) != cudaSuccess)
        return W4A8_ERR_CUDA;
    return w4a8_launch_mxfp4_tc(xq, x_scale, w_packed, w_e8m0, out_bf16, M, N, K, scratch, policy, false,
                                stream);
}
