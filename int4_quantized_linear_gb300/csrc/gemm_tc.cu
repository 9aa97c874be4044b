// gemm_tc.cu -- tensor-core (tcgen05) W4A8 GEMMs.  Placeholder: no shape is taken yet, so
// every call goes to the CUDA-core kernels.
#include "common.cuh"
#include "dispatch.h"

bool w4a8_tc_mxfp4_supported(const void *, const void *, const void *, const void *, int64_t,
                             int64_t, int64_t) { return false; }
size_t w4a8_tc_workspace_bytes(int64_t, int64_t, int64_t, int) { return 0; }
w4a8_status w4a8_launch_mxfp4_tc(const uint8_t *, const float *, const uint8_t *, const uint8_t *,
                                 uint16_t *, int64_t, int64_t, int64_t, void *, int, cudaStream_t)
{ return W4A8_ERR_UNSUPPORTED_SHAPE; }
bool w4a8_tc_int4_supported(const void *, const void *, const void *, const void *, int64_t,
                            int64_t, int64_t) { return false; }
size_t w4a8_tc_int4_workspace_bytes(int64_t, int64_t, int64_t, int) { return 0; }
w4a8_status w4a8_launch_int4_tc(const uint8_t *, const float *, const int32_t *, const uint16_t *,
                                uint16_t *, int64_t, int64_t, int64_t, void *, int, cudaStream_t)
{ return W4A8_ERR_UNSUPPORTED_SHAPE; }
