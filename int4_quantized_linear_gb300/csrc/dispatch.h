// dispatch.h -- internal (non-exported) launchers shared between the library's translation
// units.  Not part of the C ABI.
#pragma once
#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#include "../../include/w4a8.h"

#define W4A8_DECODE_MAX_M 64

// Every GEMM workspace starts with this many bytes of stream-K arrival counters; the fp32 partial
// tiles follow.  A kernel counts only on its split tiles, whose indices are below its grid size
// (at most the SM count), and leaves every counter it touched at zero, and no partial tile ever
// lands in this region -- so one buffer serves any sequence of shapes and entry points.
#define W4A8_COUNTER_BYTES ((size_t)16384)
#define W4A8_MAX_COUNTERS ((int)(W4A8_COUNTER_BYTES / 4))

int w4a8_gemm_policy();
void *w4a8_debug_trace_ptr();
unsigned int *w4a8_device_status_ptr();

// Device address of one of the library's __device__ variables on the current device.  The
// address is looked up with cudaGetSymbolAddress (with the device current) and cached per
// device together with the context it came from; a call from another context (after a device
// reset or a primary-context teardown, which load the module again, possibly elsewhere) looks
// it up again.  Thread-safe.  Returns null if the lookup fails.
struct W4a8SymbolCache;
W4a8SymbolCache *w4a8_symbol_cache_new();
void *w4a8_symbol_address(const void *symbol, W4a8SymbolCache *cache);

w4a8_status w4a8_launch_mxfp4_simt(const uint8_t *xq, const float *x_scale, const uint8_t *wp,
                                   const uint8_t *we, uint16_t *out, int64_t M, int64_t N,
                                   int64_t K, cudaStream_t stream);
w4a8_status w4a8_launch_int4_simt(const uint8_t *xq, const float *x_scale, const int32_t *qw,
                                  const uint16_t *s16, uint16_t *out, int64_t M, int64_t N,
                                  int64_t K, cudaStream_t stream,
                                  const int32_t *qzeros = nullptr, const uint8_t *qhigh = nullptr,
                                  const uint8_t *zeros5 = nullptr);

// Tensor-core (tcgen05) paths.
bool w4a8_tc_mxfp4_supported(const void *xq, const void *wp, const void *we, const void *out,
                             int64_t M, int64_t N, int64_t K);
size_t w4a8_tc_workspace_bytes(int64_t M, int64_t N, int64_t K);
// w_early: the kernel just before this one on the stream is the library's activation quant
// (chained by programmatic dependent launch), so weights may be read before waiting on it.
w4a8_status w4a8_launch_mxfp4_tc(const uint8_t *xq, const float *x_scale, const uint8_t *wp,
                                 const uint8_t *we, uint16_t *out, int64_t M, int64_t N,
                                 int64_t K, void *workspace, int policy, bool w_early,
                                 cudaStream_t stream);
// The MXFP4 GEMM with the per-token activation quant fused in (the 16-token decode tiling, M up
// to 2, rows of at most W4A8_FUSED_AQ_MAX_X_BYTES of bf16 in all): every CTA takes the row amax
// from L2 and quantizes its own fills' activations into shared memory; bit-identical to the
// activation-quant kernel followed by the GEMM.  Only w4a8_mxfp4_linear_bf16_single runs it.
#ifndef W4A8_FUSED_AQ_MAX_X_BYTES
#define W4A8_FUSED_AQ_MAX_X_BYTES (96u << 10)
#endif
bool w4a8_tc_mxfp4_aq_takes(int64_t M, int64_t K);
w4a8_status w4a8_launch_mxfp4_tc_aq(const uint16_t *x_bf16, const uint8_t *wp, const uint8_t *we, uint16_t *out,
                                    int64_t M, int64_t N, int64_t K, void *workspace, cudaStream_t stream);
// Per-token activation quant launched with programmatic dependent launch (waits for the
// previous kernel before reading x, then lets the next kernel start).
w4a8_status w4a8_launch_act_quant(const uint16_t *x_bf16, uint8_t *xq, float *x_scale, int64_t M,
                                  int64_t K, cudaStream_t stream);

bool w4a8_tc_int4_supported(const void *xq, const void *qw, const void *s16, const void *out,
                            int64_t M, int64_t N, int64_t K);
size_t w4a8_tc_int4_workspace_bytes(int64_t M, int64_t N, int64_t K);
w4a8_status w4a8_launch_int4_tc(const uint8_t *xq, const float *x_scale, const int32_t *qw,
                                const uint16_t *s16, uint16_t *out, int64_t M, int64_t N,
                                int64_t K, void *workspace, int policy, cudaStream_t stream,
                                const int32_t *qzeros = nullptr);

// Prefill tiling of the symmetric int4 / int5 GEMM (gemm_i4_pf.cu): 256-token tiles, signed
// operand codes, no zero-point MMAs.  Taken for M > W4A8_INT4_PF_MIN_M without per-group zero
// points; w4a8_int4_pf_takes also says no when the build cannot run it.
#define W4A8_INT4_PF_MIN_M 128
bool w4a8_int4_pf_takes(int64_t M, bool int5);
size_t w4a8_int4_pf_workspace_bytes(int64_t M, int64_t N, int64_t K);
w4a8_status w4a8_launch_int4_pf(const uint8_t *xq, const float *x_scale, const int32_t *qw, const uint8_t *qh,
                                const uint16_t *s16, uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace,
                                cudaStream_t stream);

// int5 g128: qh is the fifth-bit plane [K/8, N], zeros the per-(group, column) zero points
// [K/128, N] or null (zero point 16).
bool w4a8_tc_int5_supported(const void *xq, const void *qw, const void *qh, const void *s16, const void *out,
                            int64_t M, int64_t N, int64_t K);
w4a8_status w4a8_launch_int5_tc(const uint8_t *xq, const float *x_scale, const int32_t *qw, const uint8_t *qh,
                                const uint16_t *s16, const uint8_t *zeros, uint16_t *out, int64_t M, int64_t N,
                                int64_t K, void *workspace, int policy, cudaStream_t stream);

// W4A4: MXFP4 activations (xa [M, K/2] e2m1 codes, xe [M, K/32] e8m0), no per-token scale.
bool w4a8_tc_mxfp4_a4_supported(const void *xa, const void *xe, const void *wp, const void *we, const void *out,
                                int64_t M, int64_t N, int64_t K);
w4a8_status w4a8_launch_mxfp4_a4_tc(const uint8_t *xa, const uint8_t *xe, const uint8_t *wp, const uint8_t *we,
                                    uint16_t *out, int64_t M, int64_t N, int64_t K, void *workspace, int policy,
                                    cudaStream_t stream);
w4a8_status w4a8_launch_mxfp4_a4_simt(const uint8_t *xa, const uint8_t *xe, const uint8_t *wp, const uint8_t *we,
                                      uint16_t *out, int64_t M, int64_t N, int64_t K, cudaStream_t stream);
