/*
 * w4a8.h -- C ABI of the GB300 (sm_103a) W4A8 quantized-linear library (libw4a8.so).
 *
 * The method (web pages this library follows):
 *   "radiance_nvfp4.py"        -- NVFP4 -> MXFP4 requant at load (dequant_nvfp4,
 *                                 _block_exponent, e2m1_index, _encode_blocks, quant_mxfp4,
 *                                 process_weights_after_loading) and the MXFP4 weight layout
 *                                 (module docstring, item 3).
 *   "vllm-radiance (MXFP4)"    -- section "How the MXFP4 path works", subsection "The W4A8
 *                                 fp8-WMMA kernel": fp8 activations x e2m1 weights with the
 *                                 e8m0 scale folded in, a prefill tiling and a decode tiling
 *                                 with a fused split-K whose last arrival reduces.
 *   "radiance_autoround.py"    -- AutoRound int4 group-128 symmetric W4A8 (module docstring,
 *                                 autoround_linear, _exact_ref, _ensure_scratch).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless it says "host".  The caller owns all
 *     memory; no entry point allocates or frees device memory.
 *   - All work is enqueued on `stream` (asynchronous); a return of W4A8_OK means the work was
 *     launched, not that it finished.  Launch failures come back as W4A8_ERR_CUDA.
 *   - Arguments are validated before anything is launched; on any error nothing is launched
 *     and outputs are untouched.  M == 0 is a no-op that returns W4A8_OK.
 *   - Tensors are dense and row-major.  Outputs must not alias inputs.
 *   - bf16 and fp16 values travel as their 16-bit patterns (uint16_t).
 *   - e4m3 means OCP FP8 E4M3 (bias 7, max 448, no infinities, 0x7F/0xFF NaN).
 *     e2m1 code: bit 3 sign, bits 0-2 index the grid {0, .5, 1, 1.5, 2, 3, 4, 6}.
 *     e8m0 code c is the scale 2^(c - 127).
 */
#ifndef W4A8_H_
#define W4A8_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define W4A8_API __attribute__((visibility("default")))
#else
#define W4A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A8_OK = 0,
    W4A8_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad mode, bad partitions */
    W4A8_ERR_UNSUPPORTED_SHAPE = 2, /* K not a multiple of the format's block */
    W4A8_ERR_MISALIGNED = 3,        /* a pointer violates the stated alignment */
    W4A8_ERR_WORKSPACE = 4,         /* workspace missing or smaller than required */
    W4A8_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
    W4A8_ERR_TIMEOUT = 6            /* a bounded device-side wait gave up (see below) */
} w4a8_status;

/* Per-token dynamic fp8 activation quant ("radiance_autoround.py", autoround_linear: the
 * per-token dynamic fp8 cast before the GEMM; "vllm-radiance (MXFP4)", "fp8 activations").
 *   x_bf16  [M, K] bf16 (16-byte aligned)
 *   xq      [M, K] e4m3 codes, written (8-byte aligned)
 *   x_scale [M] fp32, written: amax_m / 448 (correctly rounded); an all-zero row gets 1.0
 *   xq[m,k] = e4m3_rn_satfinite(x[m,k] / x_scale[m]) with a correctly rounded fp32 division.
 * K must be a multiple of 8. */
W4A8_API w4a8_status w4a8_act_quant(const uint16_t *x_bf16, uint8_t *xq, float *x_scale, int64_t M,
                           int64_t K, cudaStream_t stream);

/* MXFP4 W4A8 linear ("vllm-radiance (MXFP4)", "The W4A8 fp8-WMMA kernel"; weight layout from
 * "radiance_nvfp4.py" module docstring item 3):
 *   out[m,n] = bf16( x_scale[m] * sum_k e4m3(xq[m,k]) * e2m1(W[n,k]) * 2^(E[n,k/32]-127) )
 *   xq       [M, K]   e4m3 codes (16-byte aligned)
 *   x_scale  [M]      fp32 per-token scale
 *   w_packed [N, K/2] two e2m1 codes per byte, the even k in the low nibble (32-byte aligned
 *                     for the tensor-core path; 16-byte aligned otherwise)
 *   w_e8m0   [N, K/32] block scales (4-byte aligned)
 *   out_bf16 [M, N]   written (4-byte aligned)
 *   workspace: device scratch of at least w4a8_workspace_bytes(M, N, K) bytes (may be NULL
 *   when that is 0).  Its first 16 KiB hold the split tiles' arrival counters and the fp32
 *   split-K partials follow; the counters must be zero before the first call that uses the
 *   buffer and are left at zero by every call that completes.  The counters sit at the same
 *   place for every shape and no partial is ever written there, so one buffer sized for the
 *   largest need can be reused call after call on one stream, for any sequence of shapes and
 *   of the entry points that take a workspace.  Two calls that run at the same time must not
 *   share a workspace.  After a call that reported a device error, zero the buffer again.
 * K must be a multiple of 32.  M <= 64 takes the decode tiling (split-K over K), larger M the
 * prefill tiling; both are chosen inside this call. */
W4A8_API w4a8_status w4a8_mxfp4_linear(const uint8_t *xq, const float *x_scale, const uint8_t *w_packed,
                              const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M, int64_t N,
                              int64_t K, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* Bytes of workspace w4a8_mxfp4_linear needs for this shape (0 if none). */
W4A8_API size_t w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* The whole MXFP4 W4A8 linear from bf16 activations: the per-token fp8 activation quant
 * followed by the MXFP4 GEMM, in one call ("radiance_autoround.py", autoround_linear: the
 * activation cast and the GEMM form one linear step; "vllm-radiance (MXFP4)": fp8 activations
 * into the W4A8 kernel).  The result is bit-identical to w4a8_act_quant followed by
 * w4a8_mxfp4_linear.
 *   x_bf16    [M, K] bf16 (16-byte aligned)
 *   w_packed, w_e8m0, out_bf16: as for w4a8_mxfp4_linear
 *   workspace: device scratch of at least w4a8_mxfp4_linear_bf16_workspace_bytes(M, N, K)
 *              bytes, 256-byte aligned.  It holds the GEMM's scratch first (counters at offset 0,
 *              kept even where the GEMM needs no scratch), then receives the quantized
 *              activations [M, K] and their scales [M]; the zero-counter contract and the reuse
 *              across shapes are those of w4a8_mxfp4_linear.
 * The two kernels are chained with programmatic dependent launch: the activation quant waits
 * for the work before it on the stream before touching memory, and the GEMM begins fetching
 * its weights while the quant runs.  K must be a multiple of 32. */
W4A8_API w4a8_status w4a8_mxfp4_linear_bf16(const uint16_t *x_bf16, const uint8_t *w_packed,
                                            const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M,
                                            int64_t N, int64_t K, void *workspace,
                                            size_t workspace_bytes, cudaStream_t stream);

/* Bytes of workspace w4a8_mxfp4_linear_bf16 needs for this shape. */
W4A8_API size_t w4a8_mxfp4_linear_bf16_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* The same linear as w4a8_mxfp4_linear_bf16 in ONE kernel launch, for one or two tokens: every
 * CTA of the GEMM reads the rows' bf16 activations, takes their per-token amax and writes the e4m3
 * tiles of its own K range straight into shared memory, so no quantized copy of x goes through
 * HBM.  The result is bit-identical to w4a8_mxfp4_linear_bf16.  Arguments, alignment and
 * workspace (size, layout and zero-counter contract) are those of w4a8_mxfp4_linear_bf16; the
 * activation part of the workspace is left untouched.
 * Takes 1 <= M <= 2, M*K*2 bytes of activations at most 96 KiB, and the shapes the tensor-core
 * MXFP4 kernel takes (K % 512 == 0, the alignments of w4a8_mxfp4_linear); anything else returns
 * W4A8_ERR_UNSUPPORTED_SHAPE (M == 0 or N == 0 returns W4A8_OK).  It ignores
 * w4a8_set_gemm_policy.
 * On the measured GB300 this form is SLOWER than the two-kernel chain behind
 * w4a8_mxfp4_linear_bf16 (about 30 us against 25 us for one token through a 34816 x 5120 weight), because
 * each CTA repeats the amax pass over x and quantizes on its scale-staging warps; it is offered
 * for callers that count launches (e.g. a launch-limited graph), not as the fast path. */
W4A8_API w4a8_status w4a8_mxfp4_linear_bf16_single(const uint16_t *x_bf16, const uint8_t *w_packed,
                                                   const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M,
                                                   int64_t N, int64_t K, void *workspace,
                                                   size_t workspace_bytes, cudaStream_t stream);

/* w4a8_mxfp4_linear for callers that cannot allocate device memory.  The pages have no
 * counterpart; this is an addition of this library.  The regular entry point needs a
 * caller-provided workspace.  Some callers cannot provide one: serving engines that reserve all
 * device memory for their own pool up front and treat an allocation outside it as an error, and
 * plugin or custom-operator interfaces that pass a kernel only its inputs and outputs.  This call
 * keeps the GEMM's scratch (fp32 partial tiles and arrival counters) in a fixed array of
 * w4a8_noalloc_scratch_bytes() bytes (12 MiB) in the library's device image, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   Arguments, layouts and the result are those of w4a8_mxfp4_linear, minus the workspace.
 *   Sizes whose scratch would exceed the array (prefill-sized token counts, very wide outputs)
 *   are rejected with W4A8_ERR_WORKSPACE before anything is launched; w4a8_workspace_bytes(M, N,
 *   K) gives the need.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it per device and context, so a
 *   call after a device reset looks it up again.  Make that first call on a device before any
 *   stream capture.
 *   The arrival counters, which must start at zero, are cleared on the stream at every call (the
 *   partial tiles need no clearing).  All calls share the one array, which keeps the last call's
 *   contents: calls that overlap on the GPU (other streams, other threads) race on it and must
 *   be serialized by the caller. */
W4A8_API w4a8_status w4a8_mxfp4_linear_noalloc(const uint8_t *xq, const float *x_scale,
                                               const uint8_t *w_packed, const uint8_t *w_e8m0,
                                               uint16_t *out_bf16, int64_t M, int64_t N, int64_t K,
                                               cudaStream_t stream);

/* Size in bytes of the fixed scratch array used by w4a8_mxfp4_linear_noalloc. */
W4A8_API size_t w4a8_noalloc_scratch_bytes(void);

/* NVFP4 -> MXFP4 requant of a (merged) linear ("radiance_nvfp4.py": dequant_nvfp4,
 * _block_exponent, e2m1_index, _encode_blocks, quant_mxfp4, requant_rows,
 * RadianceNvfp4ToMxfp4.process_weights_after_loading).  Per 32-block of each row n in
 * partition p:
 *   R1  w = fl( e2m1 * fl( fp32(e4m3 scale per 16) / divisor[p] ) )
 *   R2  block exponent e: mode 0 ocp floor(log2 amax) - 2; mode 1 noclip ceil(log2(amax/6));
 *       mode 2 mse: noclip or one binade finer, whichever has the strictly lower squared
 *       error (fp32 squares summed in ascending k); amax = 0 gives e = 0; e in [-127, 127]
 *   R3  code = e2m1_index(|w| / 2^e) (ties to the even index), sign bit only for index != 0
 *   R4  out_packed byte j = code[2j] | code[2j+1] << 4; out_e8m0 = e + 127
 *   nv_packed      [N, K/2] e2m1 codes, low nibble = even k (16-byte aligned)
 *   nv_scale_e4m3  [N, K/16] e4m3 scale codes (2-byte aligned)
 *   global_divisor [P] fp32, the checkpoint's weight_global_scale as stored (6*448/amax)
 *   partition_rows [P] HOST array of row counts, in order, summing to N; 1 <= P <= 16
 *   out_packed [N, K/2] (16-byte aligned), out_e8m0 [N, K/32], written
 *   err_ssq    [P][2] fp64 or NULL; written with {sum of squared requant error, sum of
 *              squared dequantized weights} per partition (relRMS = sqrt(err/ssq)); each
 *              32-block's terms are rounded and summed in fp32, the blocks summed in fp64
 *              (a float-precision statistic, about 1e-7 relative)
 * K must be a multiple of 32. */
W4A8_API w4a8_status nvfp4_to_mxfp4_requant(const uint8_t *nv_packed, const uint8_t *nv_scale_e4m3,
                                   const float *global_divisor, const int64_t *partition_rows,
                                   int P, int64_t N, int64_t K, int mode, uint8_t *out_packed,
                                   uint8_t *out_e8m0, double *err_ssq, cudaStream_t stream);

/* FP8-per-channel -> MXFP4 requant ("radiance_nvfp4.py": RadianceFp8ChannelToMxfp4.
 * process_weights_after_loading, then quant_mxfp4 as above).  Per 32-block of row n:
 *   R1  w = fl( fp32(e4m3 code) * row_scale[n] ), one rounded fp32 product per element;
 *   R2-R4 as for nvfp4_to_mxfp4_requant, the whole layer being one partition.
 *   w_e4m3     [N, K] e4m3 codes, row-major (16-byte aligned)
 *   row_scale  [N] fp32 per-output-channel scale (4-byte aligned)
 *   out_packed [N, K/2] (16-byte aligned), out_e8m0 [N, K/32], written
 *   err_ssq    [1][2] fp64 or NULL: {sum of squared requant error, sum of squared weights}
 * K must be a multiple of 32; mode as above.  Device pointers, stream-ordered. */
W4A8_API w4a8_status fp8_channel_to_mxfp4_requant(const uint8_t *w_e4m3, const float *row_scale,
                                                  int64_t N, int64_t K, int mode,
                                                  uint8_t *out_packed, uint8_t *out_e8m0,
                                                  double *err_ssq, cudaStream_t stream);

/* bf16 -> MXFP4 requant ("radiance_nvfp4.py": RadianceBf16ToMxfp4.process_weights_after_loading,
 * requant_rows, quant_mxfp4).  R1 is the exact fp32 value of each bf16 weight; R2-R4 and the
 * outputs as for fp8_channel_to_mxfp4_requant.
 *   w_bf16 [N, K] bf16 bits, row-major (16-byte aligned). */
W4A8_API w4a8_status bf16_to_mxfp4_requant(const uint16_t *w_bf16, int64_t N, int64_t K, int mode,
                                           uint8_t *out_packed, uint8_t *out_e8m0, double *err_ssq,
                                           cudaStream_t stream);

/* AutoRound int4 group-128 symmetric W4A8 linear ("radiance_autoround.py": module docstring,
 * _exact_ref; the symmetric zero point 8 is folded in, so code c means c - 8):
 *   out[m,n] = bf16( x_scale[m] * sum_k e4m3(xq[m,k]) * (c[k,n] - 8) * fp16(s[k/128, n]) )
 *   qweight     [K/8, N] int32, nibble j of word (i, n) holds k = 8i + j (checkpoint layout;
 *               16-byte aligned)
 *   scales_fp16 [K/128, N] fp16 bits
 *   workspace / workspace_bytes: as for w4a8_mxfp4_linear, sized by
 *   w4a8_int4g128_workspace_bytes.
 * The caller checks qzeros == 0x77777777 before calling (the Python binding does).
 * K must be a multiple of 128. */
W4A8_API w4a8_status w4a8_int4g128_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                                 const uint16_t *scales_fp16, uint16_t *out_bf16, int64_t M,
                                 int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

W4A8_API size_t w4a8_int4g128_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Asymmetric int4 group-128 W4A8 linear ("vllm-radiance (MXFP4)", section "ParoQuant (int4 W4A8
 * and int5 W5A8)": int4 group-128 asymmetric, the zero point folded into the GEMM as a row-sum
 * correction rather than dequantized into the operand).
 *   out[m, n] = bf16( x_scale[m] * sum_g s[g, n] * sum_{k in g} e4m3(xq[m, k]) * (c[k, n] - z[g, n]) )
 * with z[g, n] = 1 + nibble (n % 8) of qzeros[g, n / 8] (the packed convention under which the
 * symmetric format's 0x77777777 is the zero point 8), so z is in [1, 16].
 *   qzeros [K/128, ceil(N/8)] int32 (4-byte aligned, non-NULL); every other argument, the
 *   workspace (w4a8_int4g128_workspace_bytes) and the errors as for w4a8_int4g128_linear.
 * The tensor-core kernel keeps the activations' per-group sums (times -8 * 2^-9) in a second
 * tensor-memory accumulator and applies each column's z in the fp32 promotion. */
W4A8_API w4a8_status w4a8_int4g128_asym_linear(const uint8_t *xq, const float *x_scale,
                                               const int32_t *qweight, const uint16_t *scales_fp16,
                                               const int32_t *qzeros, uint16_t *out_bf16, int64_t M,
                                               int64_t N, int64_t K, void *workspace,
                                               size_t workspace_bytes, cudaStream_t stream);

/* int5 group-128 W5A8 linear ("vllm-radiance (MXFP4)", section "int5 (W5A8)": 5-bit codes c
 * whose value c - 16 spans -16..15, the low nibbles kept in the int4 word layout and the fifth
 * bit in a plane of one byte per word; the zero point folded in as for int4).
 *   c[k, n]   = nibble (k % 8) of qweight[k/8, n] + 16 * bit (k % 8) of qhigh[k/8, n]
 *   out[m, n] = bf16( x_scale[m] * sum_g s[g, n] * sum_{k in g} e4m3(xq[m, k]) * (c[k, n] - z[g, n]) )
 * with z = 16 when zeros is NULL, else z[g, n] = zeros[g, n].
 *   qweight [K/8, N] int32, nibble j of word (i, n) = the low four bits of the code of k = 8i + j
 *   qhigh   [K/8, N] uint8, bit j of byte (i, n) = the fifth bit of the code of k = 8i + j
 *           (device, non-NULL; the tensor-core kernel needs it 16-byte aligned and N % 16 == 0,
 *           other shapes run on the CUDA-core kernel)
 *   scales_fp16 [K/128, N] fp16 bits
 *   zeros   [K/128, N] uint8 holding z in 0..31, or NULL (symmetric)
 *   workspace: sized by w4a8_int5g128_workspace_bytes; errors as for w4a8_int4g128_linear.
 * K must be a multiple of 128.  The tensor-core kernel converts each code into the e4m3 byte of
 * (c - 16) * 2^-9 (exact for every 5-bit code); with zeros it also keeps the activations' group
 * sums in a second accumulator and applies (z - 16) per column in the fp32 promotion. */
W4A8_API w4a8_status w4a8_int5g128_linear(const uint8_t *xq, const float *x_scale, const int32_t *qweight,
                                          const uint8_t *qhigh, const uint16_t *scales_fp16,
                                          const uint8_t *zeros, uint16_t *out_bf16, int64_t M, int64_t N,
                                          int64_t K, void *workspace, size_t workspace_bytes,
                                          cudaStream_t stream);

W4A8_API size_t w4a8_int5g128_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* W4A4 activation quant ("vllm-radiance (MXFP4)", section "Native MXFP4": Quark OCP
 * micro-scaling checkpoints quantize activations to MXFP4 too, group 32, e8m0 scales).  Each
 * token row of x, per 32 along K, by the OCP rule ("radiance_nvfp4.py", _block_exponent "ocp":
 * e = floor(log2 amax) - 2, amax = 0 gives e = 0; _encode_blocks: e2m1 code of |x| * 2^-e with
 * ties to the even code, clamped to 6, sign bit only on a nonzero code):
 *   x_bf16    [M, K] bf16 bits (device, 16-byte aligned), K a multiple of 32
 *   xa_packed [M, K/2] uint8 (out; 16-byte aligned), code of k = 2j in the low nibble of byte j
 *   xa_e8m0   [M, K/32] uint8 (out), e + 127
 * Asynchronous on `stream`; bit-exact against the oracle.  Errors as for bf16_to_mxfp4_requant. */
W4A8_API w4a8_status w4a4_act_quant(const uint16_t *x_bf16, uint8_t *xa_packed, uint8_t *xa_e8m0, int64_t M,
                                    int64_t K, cudaStream_t stream);

/* W4A4 MXFP4 linear: both operands MXFP4, no per-token scale.
 *   out[m, n] = bf16( sum_k e2m1(xa[m, k]) 2^(xe[m, k/32] - 127) * e2m1(w[n, k]) 2^(we[n, k/32] - 127) )
 *   xa_packed [M, K/2], xa_e8m0 [M, K/32] as written by w4a4_act_quant; w_packed / w_e8m0 and the
 *   workspace (w4a8_workspace_bytes) as for w4a8_mxfp4_linear.
 * The tensor-core kernel takes K % 512 == 0 with xa_packed and w_packed 32-byte aligned and
 * xa_e8m0 / w_e8m0 16-byte aligned (other shapes run on the CUDA-core kernel); both operands
 * go to tcgen05.mma kind::mxf8f6f4 as e2m1 with their block scales in tensor memory. */
W4A8_API w4a8_status w4a4_mxfp4_linear(const uint8_t *xa_packed, const uint8_t *xa_e8m0, const uint8_t *w_packed,
                                       const uint8_t *w_e8m0, uint16_t *out_bf16, int64_t M, int64_t N, int64_t K,
                                       void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
W4A8_API const char *w4a8_status_string(w4a8_status s);

/* Kernel selection for the GEMM entry points: 0 = automatic (default), 1 = always the CUDA-core
 * kernels, 2 = the tensor-core (tcgen05) kernels wherever the shape allows.  Process-wide; meant
 * for tests and measurements. */
W4A8_API void w4a8_set_gemm_policy(int policy);

/* Every device-side wait in the tensor-core kernels is bounded.  A wait that gives up records
 * a code in a device status word and the kernel returns early (its output is then invalid).
 * This call synchronizes `stream`, reads and clears that word, and returns W4A8_ERR_TIMEOUT if
 * any wait gave up since the last check, W4A8_OK otherwise. */
W4A8_API w4a8_status w4a8_check_device_status(cudaStream_t stream);

/* Diagnostic: synchronizes the device, copies the raw device status block to out4 (host, 4
 * words: [0] one bit per kind of bounded wait that ran out -- 1 TMA producer, 2 MMA issuer,
 * 4 scale staging, 8 epilogue; [1] loop index and [2], [3] raw barrier state of the first such
 * event) and clears it.  Returns a w4a8_status value. */
W4A8_API int w4a8_debug_status_words(unsigned int *out4);

/* Which kernel a GEMM call with these arguments would run.  The entry points choose inside the
 * call (the tensor-core kernels need, among other things, K a multiple of 512 and the alignments
 * stated above); these queries report that choice without launching anything, so a caller can
 * tell when a shape falls back to the CUDA-core kernels, which are 10-100x slower and meant only
 * for shapes the tensor-core kernels do not take.  The arguments are the ones the entry point
 * would get (device pointers, only their values are inspected).  Returns W4A8_PATH_TENSOR_CORE,
 * W4A8_PATH_CUDA_CORE, or 0 when the entry point would reject the arguments.  The answer follows
 * the current w4a8_set_gemm_policy setting. */
#define W4A8_PATH_TENSOR_CORE 1
#define W4A8_PATH_CUDA_CORE 2
W4A8_API int w4a8_mxfp4_path(const void *xq, const void *w_packed, const void *w_e8m0, const void *out_bf16,
                             int64_t M, int64_t N, int64_t K);
W4A8_API int w4a8_int4g128_path(const void *xq, const void *qweight, const void *scales_fp16,
                                const void *out_bf16, int64_t M, int64_t N, int64_t K);
W4A8_API int w4a8_int5g128_path(const void *xq, const void *qweight, const void *qhigh, const void *scales_fp16,
                                const void *out_bf16, int64_t M, int64_t N, int64_t K);
W4A8_API int w4a4_mxfp4_path(const void *xa_packed, const void *xa_e8m0, const void *w_packed,
                             const void *w_e8m0, const void *out_bf16, int64_t M, int64_t N, int64_t K);

/* Decode-band threshold: M <= this takes the decode tiling (64). */
W4A8_API int w4a8_decode_max_m(void);

#ifdef __cplusplus
}
#endif
#endif /* W4A8_H_ */
