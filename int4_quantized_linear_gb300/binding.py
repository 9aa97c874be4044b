"""Thin Python binding over the C ABI of ``libw4a8.so`` (declared in ``include/w4a8.h``).

Argument marshalling only: PyTorch allocates device memory and supplies the stream; every
step of the path runs in the library's CUDA kernels.  There is no fallback: if the library is
missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

OK = 0
STATUS = {0: "W4A8_OK", 1: "W4A8_ERR_INVALID_ARG", 2: "W4A8_ERR_UNSUPPORTED_SHAPE",
          3: "W4A8_ERR_MISALIGNED", 4: "W4A8_ERR_WORKSPACE", 5: "W4A8_ERR_CUDA",
          6: "W4A8_ERR_TIMEOUT"}
MODES = {"ocp": 0, "noclip": 1, "mse": 2}
EXPORTS = ("w4a8_act_quant", "w4a8_mxfp4_linear", "w4a8_workspace_bytes",
           "nvfp4_to_mxfp4_requant", "fp8_channel_to_mxfp4_requant", "bf16_to_mxfp4_requant",
           "w4a8_int4g128_linear", "w4a8_int4g128_asym_linear", "w4a8_int4g128_workspace_bytes",
           "w4a8_int5g128_linear", "w4a8_int5g128_workspace_bytes", "w4a4_act_quant", "w4a4_mxfp4_linear",
           "w4a8_status_string", "w4a8_set_gemm_policy", "w4a8_check_device_status",
           "w4a8_decode_max_m", "w4a8_debug_status_words",
           "w4a8_mxfp4_linear_noalloc", "w4a8_noalloc_scratch_bytes",
           "w4a8_mxfp4_linear_bf16", "w4a8_mxfp4_linear_bf16_workspace_bytes",
           "w4a8_mxfp4_linear_bf16_single",
           "w4a8_mxfp4_path", "w4a8_int4g128_path", "w4a8_int5g128_path", "w4a4_mxfp4_path")


class W4A8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load libw4a8.so (building it in-tree first if it is missing or older than its sources; a
    library built with extra compiler options is loaded as it is)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date(check_flags=False):
        _build.build()
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError(f"libw4a8.so not found at {_build.LIB_PATH}; run build()")
    lib = ctypes.CDLL(_build.LIB_PATH)
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    I = ctypes.c_int
    sig = {
        "w4a8_act_quant": (I, [P, P, P, I64, I64, P]),
        "w4a8_mxfp4_linear": (I, [P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_workspace_bytes": (SZ, [I64, I64, I64]),
        "nvfp4_to_mxfp4_requant": (I, [P, P, P, P, I, I64, I64, I, P, P, P, P]),
        "fp8_channel_to_mxfp4_requant": (I, [P, P, I64, I64, I, P, P, P, P]),
        "bf16_to_mxfp4_requant": (I, [P, I64, I64, I, P, P, P, P]),
        "w4a8_int4g128_linear": (I, [P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_int4g128_asym_linear": (I, [P, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_int4g128_workspace_bytes": (SZ, [I64, I64, I64]),
        "w4a8_int5g128_linear": (I, [P, P, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_int5g128_workspace_bytes": (SZ, [I64, I64, I64]),
        "w4a4_act_quant": (I, [P, P, P, I64, I64, P]),
        "w4a4_mxfp4_linear": (I, [P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_status_string": (ctypes.c_char_p, [I]),
        "w4a8_set_gemm_policy": (None, [I]),
        "w4a8_check_device_status": (I, [P]),
        "w4a8_decode_max_m": (I, []),
        "w4a8_debug_status_words": (I, [P]),
        "w4a8_mxfp4_linear_noalloc": (I, [P, P, P, P, P, I64, I64, I64, P]),
        "w4a8_noalloc_scratch_bytes": (SZ, []),
        "w4a8_mxfp4_linear_bf16": (I, [P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_mxfp4_linear_bf16_workspace_bytes": (SZ, [I64, I64, I64]),
        "w4a8_mxfp4_linear_bf16_single": (I, [P, P, P, P, I64, I64, I64, P, SZ, P]),
        "w4a8_mxfp4_path": (I, [P, P, P, P, I64, I64, I64]),
        "w4a8_int4g128_path": (I, [P, P, P, P, I64, I64, I64]),
        "w4a8_int5g128_path": (I, [P, P, P, P, P, I64, I64, I64]),
        "w4a4_mxfp4_path": (I, [P, P, P, P, P, I64, I64, I64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    # builds with the pipeline timestamps compiled in export a setter for their device buffer; its
    # argument is a 64-bit pointer, which ctypes would otherwise pass as a truncated C int
    if hasattr(lib, "w4a8_debug_set_trace"):
        lib.w4a8_debug_set_trace.restype = None
        lib.w4a8_debug_set_trace.argtypes = [P]
    _lib = lib
    return lib


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != OK:
        raise W4A8Error(fn, status)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# --------------------------------------------------------------------------------------------

def set_gemm_policy(policy: int) -> None:
    """0 automatic, 1 CUDA-core kernels only, 2 tensor-core kernels wherever possible."""
    load().w4a8_set_gemm_policy(int(policy))


def decode_max_m() -> int:
    return load().w4a8_decode_max_m()


PATHS = {0: "invalid", 1: "tensor-core", 2: "cuda-core"}


def mxfp4_path(xq, w_packed, w_e8m0, out) -> str:
    """Which kernel w4a8_mxfp4_linear would run for these tensors ("tensor-core" or "cuda-core")."""
    M, K = xq.shape
    N = w_packed.shape[0]
    return PATHS[load().w4a8_mxfp4_path(_ptr(xq), _ptr(w_packed), _ptr(w_e8m0), _ptr(out), M, N, K)]


def int4g128_path(xq, qweight, scales_fp16, out) -> str:
    M, K = xq.shape
    N = qweight.shape[1]
    return PATHS[load().w4a8_int4g128_path(_ptr(xq), _ptr(qweight), _ptr(scales_fp16), _ptr(out), M, N, K)]


def int5g128_path(xq, qweight, qhigh, scales_fp16, out) -> str:
    M, K = xq.shape
    N = qweight.shape[1]
    return PATHS[load().w4a8_int5g128_path(_ptr(xq), _ptr(qweight), _ptr(qhigh), _ptr(scales_fp16), _ptr(out),
                                           M, N, K)]


def check_device_status(stream=None) -> None:
    _check("w4a8_check_device_status", load().w4a8_check_device_status(_stream(stream)))


def debug_status_words():
    """Raw device status block (see w4a8_debug_status_words); clears it."""
    buf = (ctypes.c_uint * 4)()
    _check("w4a8_debug_status_words", load().w4a8_debug_status_words(ctypes.cast(buf, ctypes.c_void_p)))
    return list(buf)


def act_quant(x: torch.Tensor, xq: torch.Tensor | None = None, x_scale: torch.Tensor | None = None,
              stream=None):
    """x bf16 [M, K] -> (xq uint8 e4m3 codes [M, K], x_scale float32 [M])."""
    _dev(x, "x", torch.bfloat16)
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check("w4a8_act_quant", load().w4a8_act_quant(_ptr(x), _ptr(xq), _ptr(x_scale), M, K,
                                                   _stream(stream)))
    return xq, x_scale


def workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_workspace_bytes(M, N, K))


def int4_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_int4g128_workspace_bytes(M, N, K))


def int5_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_int5g128_workspace_bytes(M, N, K))


def make_workspace(nbytes: int, device) -> torch.Tensor | None:
    """Zero-initialised workspace (the arrival counters must start at zero)."""
    if nbytes == 0:
        return None
    return torch.zeros((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)


def mxfp4_linear(xq, x_scale, w_packed, w_e8m0, out=None, workspace=None, stream=None):
    """out[m, n] = bf16(x_scale[m] * sum_k e4m3(xq) * e2m1(W) * 2^(E - 127))."""
    for t, n, d in ((xq, "xq", torch.uint8), (x_scale, "x_scale", torch.float32),
                    (w_packed, "w_packed", torch.uint8), (w_e8m0, "w_e8m0", torch.uint8)):
        _dev(t, n, d)
    M, K = xq.shape
    N = w_packed.shape[0]
    if w_packed.shape != (N, K // 2) or w_e8m0.shape != (N, K // 32):
        raise ValueError("weight shapes do not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    need = workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = make_workspace(need, xq.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a8_mxfp4_linear", load().w4a8_mxfp4_linear(
        _ptr(xq), _ptr(x_scale), _ptr(w_packed), _ptr(w_e8m0), _ptr(out), M, N, K,
        _ptr(workspace), wsb, _stream(stream)))
    return out


def mxfp4_linear_noalloc(xq, x_scale, w_packed, w_e8m0, out, stream=None):
    """w4a8_mxfp4_linear without a workspace: the library's own fixed scratch array is used, so
    nothing is allocated (for callers that cannot allocate; `out` must be supplied)."""
    for t, n, d in ((xq, "xq", torch.uint8), (x_scale, "x_scale", torch.float32),
                    (w_packed, "w_packed", torch.uint8), (w_e8m0, "w_e8m0", torch.uint8),
                    (out, "out", torch.bfloat16)):
        _dev(t, n, d)
    M, K = xq.shape
    N = w_packed.shape[0]
    _check("w4a8_mxfp4_linear_noalloc", load().w4a8_mxfp4_linear_noalloc(
        _ptr(xq), _ptr(x_scale), _ptr(w_packed), _ptr(w_e8m0), _ptr(out), M, N, K, _stream(stream)))
    return out


def check_symmetric_qzeros(qzeros: torch.Tensor) -> None:
    """radiance_autoround.py, process_weights_after_loading: the kernel folds a constant zero
    point of 8, so every qzeros word must be 0x77777777."""
    z = qzeros.view(torch.int32)
    bad = int((z != 0x77777777).sum())
    if bad:
        raise ValueError(f"AutoRound checkpoint is not symmetric: {bad} of {z.numel()} qzeros "
                         "words differ from 0x77777777")


def check_autoround_config(bits: int, group_size: int, sym: bool) -> None:
    """radiance_autoround.py, AutoRoundConfig.from_config: 4 bits, group 128, symmetric."""
    if bits != 4:
        raise ValueError(f"int4 kernel supports 4 bits only, got {bits}")
    if group_size != 128:
        raise ValueError(f"int4 kernel is built for group_size=128, got {group_size}")
    if not sym:
        raise ValueError("int4 kernel requires sym=true")


def int4g128_linear(xq, x_scale, qweight, scales_fp16, out=None, workspace=None, qzeros=None,
                    stream=None):
    """out[m, n] = bf16(x_scale[m] * sum_k e4m3(xq) * (c - 8) * fp16(s[k/128, n]))."""
    _dev(xq, "xq", torch.uint8)
    _dev(x_scale, "x_scale", torch.float32)
    _dev(qweight, "qweight", torch.int32)
    _dev(scales_fp16, "scales", torch.float16)
    if qzeros is not None:
        check_symmetric_qzeros(qzeros)
    M, K = xq.shape
    N = qweight.shape[1]
    if qweight.shape != (K // 8, N) or scales_fp16.shape != (K // 128, N):
        raise ValueError("int4 weight shapes do not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    need = int4_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = make_workspace(need, xq.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a8_int4g128_linear", load().w4a8_int4g128_linear(
        _ptr(xq), _ptr(x_scale), _ptr(qweight), _ptr(scales_fp16), _ptr(out), M, N, K,
        _ptr(workspace), wsb, _stream(stream)))
    return out


def int4g128_asym_linear(xq, x_scale, qweight, scales_fp16, qzeros, out=None, workspace=None, stream=None):
    """out[m, n] = bf16(x_scale[m] * sum_k e4m3(xq) * (c - z) * fp16(s[k/128, n])), z = 1 + the
    column's nibble of qzeros [K/128, ceil(N/8)] (w4a8_int4g128_asym_linear)."""
    _dev(xq, "xq", torch.uint8)
    _dev(x_scale, "x_scale", torch.float32)
    _dev(qweight, "qweight", torch.int32)
    _dev(scales_fp16, "scales", torch.float16)
    _dev(qzeros, "qzeros", torch.int32)
    M, K = xq.shape
    N = qweight.shape[1]
    if qweight.shape != (K // 8, N) or scales_fp16.shape != (K // 128, N) or qzeros.shape != (K // 128, (N + 7) // 8):
        raise ValueError("int4 weight shapes do not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    need = int4_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = make_workspace(need, xq.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a8_int4g128_asym_linear", load().w4a8_int4g128_asym_linear(
        _ptr(xq), _ptr(x_scale), _ptr(qweight), _ptr(scales_fp16), _ptr(qzeros), _ptr(out), M, N, K,
        _ptr(workspace), wsb, _stream(stream)))
    return out


def int5g128_linear(xq, x_scale, qweight, qhigh, scales_fp16, zeros=None, out=None, workspace=None,
                    stream=None):
    """out[m, n] = bf16(x_scale[m] * sum_k e4m3(xq) * (c - z) * fp16(s[k/128, n])) with the 5-bit
    code c = nibble of qweight [K/8, N] + 16 * bit of qhigh [K/8, N] (bit j of byte (i, n) for
    k = 8i + j), z = 16 or zeros [K/128, N] uint8 (w4a8_int5g128_linear)."""
    _dev(xq, "xq", torch.uint8)
    _dev(x_scale, "x_scale", torch.float32)
    _dev(qweight, "qweight", torch.int32)
    _dev(qhigh, "qhigh", torch.uint8)
    _dev(scales_fp16, "scales", torch.float16)
    M, K = xq.shape
    N = qweight.shape[1]
    if qweight.shape != (K // 8, N) or qhigh.shape != (K // 8, N) or scales_fp16.shape != (K // 128, N):
        raise ValueError("int5 weight shapes do not match K")
    if zeros is not None:
        _dev(zeros, "zeros", torch.uint8)
        if zeros.shape != (K // 128, N):
            raise ValueError("int5 zeros must be [K/128, N]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    need = int5_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = make_workspace(need, xq.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a8_int5g128_linear", load().w4a8_int5g128_linear(
        _ptr(xq), _ptr(x_scale), _ptr(qweight), _ptr(qhigh), _ptr(scales_fp16), _ptr(zeros), _ptr(out),
        M, N, K, _ptr(workspace), wsb, _stream(stream)))
    return out


def act_quant_mxfp4(x, xa=None, xe=None, stream=None):
    """W4A4 activations: bf16 [M, K] -> (e2m1 codes uint8 [M, K/2], e8m0 uint8 [M, K/32]) by the
    OCP rule per 32 (w4a4_act_quant)."""
    _dev(x, "x", torch.bfloat16)
    M, K = x.shape
    if xa is None:
        xa = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    if xe is None:
        xe = torch.empty((M, K // 32), dtype=torch.uint8, device=x.device)
    _check("w4a4_act_quant", load().w4a4_act_quant(_ptr(x), _ptr(xa), _ptr(xe), M, K, _stream(stream)))
    return xa, xe


def mxfp4_a4_linear(xa, xe, w_packed, w_e8m0, out=None, workspace=None, stream=None):
    """W4A4: out[m, n] = bf16(sum_k dequant(xa)[m, k] * dequant(w)[n, k]) (w4a4_mxfp4_linear)."""
    for t, name in ((xa, "xa"), (xe, "xe"), (w_packed, "w_packed"), (w_e8m0, "w_e8m0")):
        _dev(t, name, torch.uint8)
    M, K2 = xa.shape
    K = 2 * K2
    N = w_packed.shape[0]
    if xe.shape != (M, K // 32) or w_packed.shape != (N, K // 2) or w_e8m0.shape != (N, K // 32):
        raise ValueError("W4A4 operand shapes do not match")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xa.device)
    need = workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = make_workspace(need, xa.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("w4a4_mxfp4_linear", load().w4a4_mxfp4_linear(
        _ptr(xa), _ptr(xe), _ptr(w_packed), _ptr(w_e8m0), _ptr(out), M, N, K, _ptr(workspace), wsb,
        _stream(stream)))
    return out


def requant(nv_packed, nv_scale, divisors, partition_rows, mode="mse", out_packed=None,
            out_e8m0=None, err_ssq=True, stream=None):
    """NVFP4 -> MXFP4.  Returns (packed uint8 [N, K/2], e8m0 uint8 [N, K/32], err_ssq float64
    [P, 2] or None)."""
    _dev(nv_packed, "nv_packed", torch.uint8)
    if nv_scale.dtype == torch.float8_e4m3fn:
        nv_scale = nv_scale.view(torch.uint8)
    _dev(nv_scale, "nv_scale", torch.uint8)
    _dev(divisors, "divisors", torch.float32)
    N, K2 = nv_packed.shape
    K = 2 * K2
    rows = (ctypes.c_int64 * len(partition_rows))(*[int(r) for r in partition_rows])
    P = len(partition_rows)
    if out_packed is None:
        out_packed = torch.empty((N, K // 2), dtype=torch.uint8, device=nv_packed.device)
    if out_e8m0 is None:
        out_e8m0 = torch.empty((N, K // 32), dtype=torch.uint8, device=nv_packed.device)
    es = torch.empty((P, 2), dtype=torch.float64, device=nv_packed.device) if err_ssq else None
    _check("nvfp4_to_mxfp4_requant", load().nvfp4_to_mxfp4_requant(
        _ptr(nv_packed), _ptr(nv_scale), _ptr(divisors), ctypes.cast(rows, ctypes.c_void_p), P, N,
        K, MODES[mode] if isinstance(mode, str) else int(mode), _ptr(out_packed), _ptr(out_e8m0),
        _ptr(es), _stream(stream)))
    return out_packed, out_e8m0, es


def _requant_outputs(N, K, device, out_packed, out_e8m0, err_ssq):
    if out_packed is None:
        out_packed = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
    if out_e8m0 is None:
        out_e8m0 = torch.empty((N, K // 32), dtype=torch.uint8, device=device)
    es = torch.empty((1, 2), dtype=torch.float64, device=device) if err_ssq else None
    return out_packed, out_e8m0, es


def requant_fp8_channel(w_e4m3, row_scale, mode="mse", out_packed=None, out_e8m0=None, err_ssq=True,
                        stream=None):
    """FP8 per-channel weight [N, K] (e4m3 codes or float8_e4m3fn) x fp32 scale [N] -> MXFP4.
    Returns (packed [N, K/2], e8m0 [N, K/32], err_ssq float64 [1, 2] or None)."""
    if w_e4m3.dtype == torch.float8_e4m3fn:
        w_e4m3 = w_e4m3.view(torch.uint8)
    _dev(w_e4m3, "w_e4m3", torch.uint8)
    row_scale = row_scale.reshape(-1)
    _dev(row_scale, "row_scale", torch.float32)
    N, K = w_e4m3.shape
    out_packed, out_e8m0, es = _requant_outputs(N, K, w_e4m3.device, out_packed, out_e8m0, err_ssq)
    _check("fp8_channel_to_mxfp4_requant", load().fp8_channel_to_mxfp4_requant(
        _ptr(w_e4m3), _ptr(row_scale), N, K, MODES[mode] if isinstance(mode, str) else int(mode),
        _ptr(out_packed), _ptr(out_e8m0), _ptr(es), _stream(stream)))
    return out_packed, out_e8m0, es


def requant_bf16(w_bf16, mode="mse", out_packed=None, out_e8m0=None, err_ssq=True, stream=None):
    """bf16 weight [N, K] -> MXFP4.  Returns (packed [N, K/2], e8m0 [N, K/32], err_ssq float64
    [1, 2] or None)."""
    _dev(w_bf16, "w_bf16", torch.bfloat16)
    N, K = w_bf16.shape
    out_packed, out_e8m0, es = _requant_outputs(N, K, w_bf16.device, out_packed, out_e8m0, err_ssq)
    _check("bf16_to_mxfp4_requant", load().bf16_to_mxfp4_requant(
        _ptr(w_bf16), N, K, MODES[mode] if isinstance(mode, str) else int(mode), _ptr(out_packed),
        _ptr(out_e8m0), _ptr(es), _stream(stream)))
    return out_packed, out_e8m0, es


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_mxfp4_linear_bf16_workspace_bytes(M, N, K))


def make_linear_workspace(M: int, N: int, K: int, device) -> torch.Tensor:
    """Zero-initialised, 256-byte aligned workspace for linear() / w4a8_mxfp4_linear_bf16."""
    nbytes = linear_workspace_bytes(M, N, K)
    buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def linear(x: torch.Tensor, w_packed: torch.Tensor, w_e8m0: torch.Tensor, out=None,
           workspace=None, stream=None, single_kernel: bool = False) -> torch.Tensor:
    """The whole W4A8 MXFP4 linear from bf16 activations in one native call: per-token fp8
    activation quant, then the GEMM (w4a8_mxfp4_linear_bf16).  single_kernel=True runs it as one
    launch with the quant inside the GEMM (w4a8_mxfp4_linear_bf16_single: 1 or 2 tokens, same
    bytes, slower than the default two-kernel chain on GB300)."""
    _dev(x, "x", torch.bfloat16)
    _dev(w_packed, "w_packed", torch.uint8)
    _dev(w_e8m0, "w_e8m0", torch.uint8)
    M, K = x.shape
    N = w_packed.shape[0]
    if w_packed.shape != (N, K // 2) or w_e8m0.shape != (N, K // 32):
        raise ValueError("weight shapes do not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = make_linear_workspace(M, N, K, x.device)
    wsb = workspace.numel() * workspace.element_size()
    fn = "w4a8_mxfp4_linear_bf16_single" if single_kernel else "w4a8_mxfp4_linear_bf16"
    _check(fn, getattr(load(), fn)(
        _ptr(x), _ptr(w_packed), _ptr(w_e8m0), _ptr(out), M, N, K, _ptr(workspace), wsb,
        _stream(stream)))
    return out
