// dispatch.h -- internal (non-exported) launchers shared between the library's translation
// units.  Not part of the C ABI.
#pragma once
#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#include "../../include/w4a8.h"

#define W4A8_DECODE_MAX_M 64

int w4a8_gemm_policy();
void *w4a8_debug_trace_ptr();
unsigned int *w4a8_device_status_ptr();

w4a8_status w4a8_launch_mxfp4_simt(const uint8_t *xq, const float *x_scale, const uint8_t *wp,
                                   const uint8_t *we, uint16_t *out, int64_t M, int64_t N,
                                   int64_t K, cudaStream_t stream);
w4a8_status w4a8_launch_int4_simt(const uint8_t *xq, const float *x_scale, const int32_t *qw,
                                  const uint16_t *s16, uint16_t *out, int64_t M, int64_t N,
                                  int64_t K, cudaStream_t stream);

// Tensor-core (tcgen05) paths.
bool w4a8_tc_mxfp4_supported(const void *xq, const void *wp, const void *we, const void *out,
                             int64_t M, int64_t N, int64_t K);
size_t w4a8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, int policy);
size_t w4a8_tc_workspace_counters_offset(int64_t M, int64_t N, int64_t K);
w4a8_status w4a8_launch_mxfp4_tc(const uint8_t *xq, const float *x_scale, const uint8_t *wp,
                                 const uint8_t *we, uint16_t *out, int64_t M, int64_t N,
                                 int64_t K, void *workspace, int policy, cudaStream_t stream);

bool w4a8_tc_int4_supported(const void *xq, const void *qw, const void *s16, const void *out,
                            int64_t M, int64_t N, int64_t K);
size_t w4a8_tc_int4_workspace_bytes(int64_t M, int64_t N, int64_t K, int policy);
w4a8_status w4a8_launch_int4_tc(const uint8_t *xq, const float *x_scale, const int32_t *qw,
                                const uint16_t *s16, uint16_t *out, int64_t M, int64_t N,
                                int64_t K, void *workspace, int policy, cudaStream_t stream);
