"""ctypes front end of the scalar C oracle in ``w4a8_oracle.c``.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg
use it; the product path never does.  Every function here is argument marshalling; the
arithmetic lives in the C file, each routine citing the page passage it follows:

* "radiance_nvfp4.py": unpack_e2m1, dequant_nvfp4, e2m1_index, _block_exponent,
  _encode_blocks, quant_mxfp4, dequant_mxfp4, requant_rows, process_weights_after_loading.
* "vllm-radiance (MXFP4)", section "How the MXFP4 path works" / "The W4A8 fp8-WMMA kernel".
* "radiance_autoround.py": module docstring, autoround_linear, _exact_ref.
* "vllm-radiance (MXFP4)", section "ParoQuant (int4 W4A8 and int5 W5A8)" and "int5 (W5A8)":
  the asymmetric int4 zero point and the 5-bit codes; section "Native MXFP4": the W4A4 path
  (MXFP4 activations, OCP rule per 32).

Parity pins: every routine is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py``
(closed forms, brute force on tiny inputs, hand-built exact blocks, invariants).  Two
agreements are "parity unpinned" by design: agreement with the unspecified rounding of the
page's fp32 torch ``log2`` / ``.sum`` (the exact rule and a fixed fp32 order are pinned
instead), and the page's real-checkpoint relRMS figures (the checkpoint is not available).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

MODES = {"ocp": 0, "noclip": 1, "mse": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler supports it)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        sig = {
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_fp16_decode": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_e2m1_index": (ctypes.c_int, [ctypes.c_float]),
            "orc_block_exponent": (ctypes.c_int, [ctypes.c_float, ctypes.c_int]),
            "orc_quant_block": (ctypes.c_int, [P, ctypes.c_int, P, P]),
            "orc_act_quant": (None, [P, I64, I64, P, P]),
            "orc_requant": (ctypes.c_int, [P, P, P, P, ctypes.c_int, I64, I64, ctypes.c_int,
                                           P, P, P]),
            "orc_dequant_mxfp4": (None, [P, P, I64, I64, P]),
            "orc_requant_fp8_channel": (ctypes.c_int, [P, P, I64, I64, ctypes.c_int, P, P, P]),
            "orc_requant_bf16": (ctypes.c_int, [P, I64, I64, ctypes.c_int, P, P, P]),
            "orc_nvfp4_quantize": (None, [P, P, ctypes.c_int, I64, P, P, P]),
            "orc_mxfp4_linear": (None, [P, P, P, P, I64, I64, I64, P]),
            "orc_mxfp4_linear_pairs": (None, [P, P, P, P, I64, P, P, I64, P]),
            "orc_int4g128_linear": (None, [P, P, P, P, I64, I64, I64, P]),
            "orc_int4g128_linear_pairs": (None, [P, P, P, P, I64, I64, P, P, I64, P]),
            "orc_int4g128_asym_linear": (None, [P, P, P, P, P, I64, I64, I64, P]),
            "orc_int4g128_asym_linear_pairs": (None, [P, P, P, P, P, I64, I64, P, P, I64, P]),
            "orc_int5g128_linear": (None, [P, P, P, P, P, P, I64, I64, I64, P]),
            "orc_int5g128_linear_pairs": (None, [P, P, P, P, P, P, I64, I64, P, P, I64, P]),
            "orc_act_quant_mxfp4": (None, [P, I64, I64, P, P]),
            "orc_mxfp4_a4_linear": (None, [P, P, P, P, I64, I64, I64, P]),
            "orc_mxfp4_a4_linear_pairs": (None, [P, P, P, P, I64, P, P, I64, P]),
            "orc_e4m3_encode_many": (None, [P, I64, P]),
            "orc_e4m3_decode_many": (None, [P, I64, P]),
            "orc_fp16_decode_many": (None, [P, I64, P]),
            "orc_num_threads": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().orc_num_threads()


# --- number formats ------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e4m3_decode_many(codes) -> np.ndarray:
    a, ap = _c(codes, np.uint8)
    out = np.empty(a.shape, np.float64)
    _load().orc_e4m3_decode_many(ap, a.size, _p(out))
    return out


def e4m3_encode(y: float) -> int:
    return _load().orc_e4m3_encode(float(y))


def e4m3_encode_many(y) -> np.ndarray:
    a, ap = _c(y, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_e4m3_encode_many(ap, a.size, _p(out))
    return out


def fp16_decode(bits: int) -> float:
    return _load().orc_fp16_decode(int(bits))


def fp16_decode_many(bits) -> np.ndarray:
    a, ap = _c(bits, np.uint16)
    out = np.empty(a.shape, np.float64)
    _load().orc_fp16_decode_many(ap, a.size, _p(out))
    return out


def e2m1_index(a: float) -> int:
    return _load().orc_e2m1_index(float(a))


def block_exponent(amax: float, mode: str) -> int:
    return _load().orc_block_exponent(float(amax), MODES[mode])


def quant_block(w32, mode: str):
    """One 32-block -> (exponent e, codes uint8[32], squared error in unscaled units)."""
    w, wp = _c(w32, np.float32)
    assert w.size == 32
    codes = np.zeros(32, np.uint8)
    err = np.zeros(1, np.float64)
    e = _load().orc_quant_block(wp, MODES[mode], _p(codes), _p(err))
    return e, codes, float(err[0])


# --- the method's steps --------------------------------------------------------------------

def act_quant(x_bf16: np.ndarray):
    """x bf16 bits [M, K] (uint16) -> (codes uint8 [M, K], scale float32 [M])."""
    x, xp = _c(x_bf16, np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), np.uint8)
    sc = np.empty(M, np.float32)
    _load().orc_act_quant(xp, M, K, _p(xq), _p(sc))
    return xq, sc


def requant(nv_packed, nv_scale, divisors, partition_rows, mode: str):
    """NVFP4 -> MXFP4.  Returns (packed [N, K/2], e8m0 [N, K/32], err_ssq [P, 2])."""
    pk, pkp = _c(nv_packed, np.uint8)
    sc, scp = _c(nv_scale, np.uint8)
    dv, dvp = _c(divisors, np.float32)
    pr, prp = _c(partition_rows, np.int64)
    N, K2 = pk.shape
    K = 2 * K2
    P = pr.size
    out_p = np.empty((N, K // 2), np.uint8)
    out_e = np.empty((N, K // 32), np.uint8)
    es = np.zeros((P, 2), np.float64)
    rc = _load().orc_requant(pkp, scp, dvp, prp, P, N, K, MODES[mode], _p(out_p), _p(out_e),
                             _p(es))
    if rc != 0:
        raise ValueError("oracle requant: invalid arguments")
    return out_p, out_e, es


def requant_fp8_channel(w8, row_scale, mode: str):
    """FP8 per-channel [N, K] e4m3 codes x fp32 scale [N] -> MXFP4.  Returns (packed [N, K/2],
    e8m0 [N, K/32], err_ssq [1, 2])."""
    w, wp = _c(w8, np.uint8)
    s, sp = _c(row_scale, np.float32)
    N, K = w.shape
    out_p = np.empty((N, K // 2), np.uint8)
    out_e = np.empty((N, K // 32), np.uint8)
    es = np.zeros((1, 2), np.float64)
    if _load().orc_requant_fp8_channel(wp, sp, N, K, MODES[mode], _p(out_p), _p(out_e), _p(es)) != 0:
        raise ValueError("oracle requant: invalid arguments")
    return out_p, out_e, es


def requant_bf16(w_bf16, mode: str):
    """bf16 [N, K] (uint16 bits) -> MXFP4.  Returns (packed, e8m0, err_ssq [1, 2])."""
    w, wp = _c(w_bf16, np.uint16)
    N, K = w.shape
    out_p = np.empty((N, K // 2), np.uint8)
    out_e = np.empty((N, K // 32), np.uint8)
    es = np.zeros((1, 2), np.float64)
    if _load().orc_requant_bf16(wp, N, K, MODES[mode], _p(out_p), _p(out_e), _p(es)) != 0:
        raise ValueError("oracle requant: invalid arguments")
    return out_p, out_e, es


def rel_rms(err_ssq: np.ndarray) -> float:
    """Combined requant relRMS over partitions (process_weights_after_loading)."""
    e = float(np.sum(err_ssq[:, 0]))
    s = float(np.sum(err_ssq[:, 1]))
    return (e / max(s, 1e-30)) ** 0.5


def dequant_mxfp4(packed, e8m0) -> np.ndarray:
    pk, pkp = _c(packed, np.uint8)
    ee, eep = _c(e8m0, np.uint8)
    N, K2 = pk.shape
    w = np.empty((N, 2 * K2), np.float64)
    _load().orc_dequant_mxfp4(pkp, eep, N, 2 * K2, _p(w))
    return w


def nvfp4_quantize(w_fp32, partition_rows):
    """Synthesise an NVFP4 checkpoint tensor from fp32 weights (input synthesis only)."""
    w, wp = _c(w_fp32, np.float32)
    pr, prp = _c(partition_rows, np.int64)
    N, K = w.shape
    packed = np.zeros((N, K // 2), np.uint8)
    scale = np.zeros((N, K // 16), np.uint8)
    div = np.zeros(pr.size, np.float32)
    _load().orc_nvfp4_quantize(wp, prp, pr.size, K, _p(packed), _p(scale), _p(div))
    return packed, scale, div


def mxfp4_linear(xq, x_scale, w_packed, w_e8m0) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    wpk, wpp = _c(w_packed, np.uint8)
    we, wep = _c(w_e8m0, np.uint8)
    M, K = x.shape
    N = wpk.shape[0]
    out = np.empty((M, N), np.float64)
    _load().orc_mxfp4_linear(xp, sp, wpp, wep, M, N, K, _p(out))
    return out


def mxfp4_linear_pairs(xq, x_scale, w_packed, w_e8m0, idx_m, idx_n) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    wpk, wpp = _c(w_packed, np.uint8)
    we, wep = _c(w_e8m0, np.uint8)
    im, imp = _c(idx_m, np.int64)
    inn, inp = _c(idx_n, np.int64)
    K = x.shape[1]
    out = np.empty(im.size, np.float64)
    _load().orc_mxfp4_linear_pairs(xp, sp, wpp, wep, K, imp, inp, im.size, _p(out))
    return out


def int4g128_linear(xq, x_scale, qweight, scales_fp16) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    sc, scp = _c(scales_fp16, np.uint16)
    M, K = x.shape
    N = q.shape[1]
    out = np.empty((M, N), np.float64)
    _load().orc_int4g128_linear(xp, sp, qp, scp, M, N, K, _p(out))
    return out


def int4g128_linear_pairs(xq, x_scale, qweight, scales_fp16, idx_m, idx_n) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    sc, scp = _c(scales_fp16, np.uint16)
    im, imp = _c(idx_m, np.int64)
    inn, inp = _c(idx_n, np.int64)
    K = x.shape[1]
    N = q.shape[1]
    out = np.empty(im.size, np.float64)
    _load().orc_int4g128_linear_pairs(xp, sp, qp, scp, N, K, imp, inp, im.size, _p(out))
    return out


def int4g128_asym_linear(xq, x_scale, qweight, scales_fp16, qzeros) -> np.ndarray:
    """Asymmetric int4 g128: zero point 1 + nibble of qzeros [K/128, ceil(N/8)] per (group, column)."""
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    sc, scp = _c(scales_fp16, np.uint16)
    z, zp = _c(qzeros, np.int32)
    M, K = x.shape
    N = q.shape[1]
    out = np.empty((M, N), np.float64)
    _load().orc_int4g128_asym_linear(xp, sp, qp, scp, zp, M, N, K, _p(out))
    return out


def int4g128_asym_linear_pairs(xq, x_scale, qweight, scales_fp16, qzeros, idx_m, idx_n) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    sc, scp = _c(scales_fp16, np.uint16)
    z, zp = _c(qzeros, np.int32)
    im, imp = _c(idx_m, np.int64)
    inn, inp = _c(idx_n, np.int64)
    K = x.shape[1]
    N = q.shape[1]
    out = np.empty(im.size, np.float64)
    _load().orc_int4g128_asym_linear_pairs(xp, sp, qp, scp, zp, N, K, imp, inp, im.size, _p(out))
    return out


def int5g128_linear(xq, x_scale, qweight, qhigh, scales_fp16, zeros=None) -> np.ndarray:
    """int5 g128: low nibbles in qweight [K/8, N], fifth bits in qhigh [K/8, N] (bit j of byte
    (i, n) for k = 8i + j); zero point 16, or zeros [K/128, N] uint8 per (group, column)."""
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    h, hp = _c(qhigh, np.uint8)
    sc, scp = _c(scales_fp16, np.uint16)
    z, zp = (None, None) if zeros is None else _c(zeros, np.uint8)
    M, K = x.shape
    N = q.shape[1]
    out = np.empty((M, N), np.float64)
    _load().orc_int5g128_linear(xp, sp, qp, hp, scp, zp, M, N, K, _p(out))
    return out


def int5g128_linear_pairs(xq, x_scale, qweight, qhigh, scales_fp16, zeros, idx_m, idx_n) -> np.ndarray:
    x, xp = _c(xq, np.uint8)
    s, sp = _c(x_scale, np.float32)
    q, qp = _c(qweight, np.int32)
    h, hp = _c(qhigh, np.uint8)
    sc, scp = _c(scales_fp16, np.uint16)
    z, zp = (None, None) if zeros is None else _c(zeros, np.uint8)
    im, imp = _c(idx_m, np.int64)
    inn, inp = _c(idx_n, np.int64)
    K = x.shape[1]
    N = q.shape[1]
    out = np.empty(im.size, np.float64)
    _load().orc_int5g128_linear_pairs(xp, sp, qp, hp, scp, zp, N, K, imp, inp, im.size, _p(out))
    return out


def act_quant_mxfp4(x_bf16):
    """W4A4 activations: bf16 [M, K] (uint16 bits) -> (packed e2m1 [M, K/2], e8m0 [M, K/32]) by the
    OCP rule per 32 along each row."""
    x, xp = _c(x_bf16, np.uint16)
    M, K = x.shape
    out_p = np.empty((M, K // 2), np.uint8)
    out_e = np.empty((M, K // 32), np.uint8)
    _load().orc_act_quant_mxfp4(xp, M, K, _p(out_p), _p(out_e))
    return out_p, out_e


def mxfp4_a4_linear(xa, xe, w_packed, w_e8m0) -> np.ndarray:
    """W4A4: out[m, n] = sum_k dequant(xa)[m, k] * dequant(w)[n, k], fp64."""
    a, ap = _c(xa, np.uint8)
    e, ep = _c(xe, np.uint8)
    w, wp = _c(w_packed, np.uint8)
    we, wep = _c(w_e8m0, np.uint8)
    M = a.shape[0]
    K = 2 * a.shape[1]
    N = w.shape[0]
    out = np.empty((M, N), np.float64)
    _load().orc_mxfp4_a4_linear(ap, ep, wp, wep, M, N, K, _p(out))
    return out


def mxfp4_a4_linear_pairs(xa, xe, w_packed, w_e8m0, idx_m, idx_n) -> np.ndarray:
    a, ap = _c(xa, np.uint8)
    e, ep = _c(xe, np.uint8)
    w, wp = _c(w_packed, np.uint8)
    we, wep = _c(w_e8m0, np.uint8)
    im, imp = _c(idx_m, np.int64)
    inn, inp = _c(idx_n, np.int64)
    K = 2 * a.shape[1]
    out = np.empty(im.size, np.float64)
    _load().orc_mxfp4_a4_linear_pairs(ap, ep, wp, wep, K, imp, inp, im.size, _p(out))
    return out
