"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds random number generation and the workload recipes only -- none of the
quantizer's arithmetic (no fp8 / e2m1 / e8m0 encoding happens here).  It is portable across
machines: every draw comes from a counter-based splitmix64 stream keyed by (seed, tensor id),
turned into uniforms from the top 53 bits and into normals by the Box-Muller transform, in
numpy uint64 / float64 arithmetic.

Workload recipes (the served model's linear shapes: hidden 5120, MLP 17408, merged gate_up
34816 = 17408 + 17408; attention qkv 10240 x 5120):

* tiny:     x bf16 ~ N(0, 1), each element x8 with probability 0.01; W fp32 ~ N(0, 0.02).
* decode:   x bf16 ~ N(0, 1); weight bytes uniform 0..255; e8m0 uniform in {118..121}.
* prefill:  x bf16 ~ N(0, 1) * r_m, r_m ~ LogNormal(0, 1) per row; nibbles uniform;
            e8m0 uniform in {118..124}.
* int4:     qweight int32 of uniform nibbles [K/8, N]; scales fp16(|N(0, 0.003)|) [K/128, N];
            qzeros 0x77777777 [K/128, N/8]; x bf16 ~ N(0, 1).
* requant:  W fp32 ~ N(0, 0.02) [N, K], split into row partitions.
* fp8 per-channel requant source: e4m3 codes uniform over the 254 finite codes [N, K];
            row scale fp32 2^u, u uniform in [-12, -6], per row.
* bf16 requant source: bf16(N(0, 0.02)) [N, K].
* int4 asymmetric: as int4, with qzeros [K/128, ceil(N/8)] of uniform nibbles (zero points 1..16).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Tensor ids: one independent stream per tensor role.
T_X, T_OUTLIER, T_OUTLIER_PICK, T_W, T_E, T_ROWSCALE, T_QW, T_QS, T_WREQ, T_NVS, T_W8, T_W8S, T_WB, T_QZ, T_QH, T_Z5 = range(1, 17)

GATE_UP = (34816, 5120)
DOWN = (5120, 17408)
QKV = (10240, 5120)
GATE_UP_PARTITIONS = (17408, 17408)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def u64(seed: int, tensor: int, n: int, offset: int = 0) -> np.ndarray:
    """n pseudo-random uint64 from the counter-based stream (seed, tensor)."""
    key = _mix(np.array([(seed * 1000003 + tensor) & 0xFFFFFFFFFFFFFFFF], np.uint64))[0]
    ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * _GOLDEN)


def uniform(seed: int, tensor: int, n: int) -> np.ndarray:
    """Uniform float64 in [0, 1)."""
    return (u64(seed, tensor, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, tensor: int, n: int, chunk: int = 1 << 24) -> np.ndarray:
    """Standard normals; element 2j is r*cos(t) and element 2j+1 is r*sin(t) for the uniform
    pair at counters (2j, 2j+1), so the stream does not depend on the chunk size."""
    out = np.empty(n, np.float64)
    for a in range(0, n, chunk):  # chunk is even, so pairs never straddle chunks
        b = min(n, a + chunk)
        h = (b - a + 1) // 2
        u = (u64(seed, tensor, 2 * h, offset=a) >> np.uint64(11)).astype(np.float64)
        u *= 1.0 / 9007199254740992.0
        r = np.sqrt(-2.0 * np.log(1.0 - u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        z = np.empty(2 * h, np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        out[a:b] = z[: b - a]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bfloat16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations(M: int, K: int, seed: int = 0, outliers: bool = False,
                lognormal_rows: bool = False) -> np.ndarray:
    """bf16 bits [M, K]."""
    x = normal(seed, T_X, M * K).reshape(M, K)
    if outliers:
        pick = uniform(seed, T_OUTLIER_PICK, M * K).reshape(M, K) < 0.01
        x = np.where(pick, 8.0 * x, x)
    if lognormal_rows:
        r = np.exp(normal(seed, T_ROWSCALE, M))
        x = x * r[:, None]
    return to_bf16_bits(x.astype(np.float32))


def uniform_bytes(n_rows: int, n_cols: int, seed: int, tensor: int) -> np.ndarray:
    n = n_rows * n_cols
    words = u64(seed, tensor, (n + 7) // 8)
    return words.view(np.uint8)[:n].reshape(n_rows, n_cols).copy()


def uniform_ints(n: int, lo: int, hi: int, seed: int, tensor: int) -> np.ndarray:
    """Uniform integers in [lo, hi] inclusive."""
    span = np.uint64(hi - lo + 1)
    return lo + (u64(seed, tensor, n) % span).astype(np.int64)


def mxfp4_weights(N: int, K: int, seed: int = 0, e_lo: int = 118, e_hi: int = 121):
    """(packed [N, K/2] uint8 with uniform bytes, e8m0 [N, K/32] uniform in [e_lo, e_hi])."""
    packed = uniform_bytes(N, K // 2, seed, T_W)
    e8m0 = uniform_ints(N * (K // 32), e_lo, e_hi, seed, T_E).astype(np.uint8)
    return packed, e8m0.reshape(N, K // 32)


def decode_case(M: int, N: int, K: int, seed: int = 0):
    x = activations(M, K, seed)
    w, e = mxfp4_weights(N, K, seed, 118, 121)
    return x, w, e


def prefill_case(M: int, N: int, K: int, seed: int = 0):
    x = activations(M, K, seed, lognormal_rows=True)
    w, e = mxfp4_weights(N, K, seed, 118, 124)
    return x, w, e


def int4_weights(N: int, K: int, seed: int = 0):
    """(qweight int32 [K/8, N], scales fp16 bits uint16 [K/128, N], qzeros int32 [K/128, N/8])."""
    n_words = (K // 8) * N
    q = u64(seed, T_QW, (n_words + 1) // 2).view(np.uint32)[:n_words]
    qweight = q.view(np.int32).reshape(K // 8, N).copy()
    s = np.abs(normal(seed, T_QS, (K // 128) * N) * 0.003).astype(np.float16)
    scales = s.view(np.uint16).reshape(K // 128, N).copy()
    qzeros = np.full((K // 128, max(N // 8, 1)), 0x77777777, np.uint32).view(np.int32)
    return qweight, scales, qzeros


def int4_case(M: int, N: int, K: int, seed: int = 0):
    x = activations(M, K, seed)
    qw, sc, qz = int4_weights(N, K, seed)
    return x, qw, sc, qz


def nvfp4_tensor_bytes(N: int, K: int, seed: int = 0, s_lo: int = 0x28, s_hi: int = 0x50):
    """Throughput-test stand-in for an NVFP4 checkpoint tensor, in its storage layout:
    (packed [N, K/2] uniform bytes, e4m3 scale codes [N, K/16] uniform in [s_lo, s_hi] (positive
    normals, 2^-2 .. 2^3 for the defaults)).  Shapes and byte volumes match a real checkpoint;
    the values are not the output of a quantizer (parity tests use the oracle's quantizer)."""
    packed = uniform_bytes(N, K // 2, seed, T_W)
    scale = uniform_ints(N * (K // 16), s_lo, s_hi, seed, T_NVS).astype(np.uint8)
    return packed, scale.reshape(N, K // 16)


def gaussian_weights(N: int, K: int, sigma: float = 0.02, seed: int = 0,
                     row_gain=None) -> np.ndarray:
    """fp32 [N, K] ~ N(0, sigma); row_gain (optional [N]) multiplies each row."""
    w = normal(seed, T_WREQ, N * K).reshape(N, K) * sigma
    if row_gain is not None:
        w = w * np.asarray(row_gain, np.float64)[:, None]
    return w.astype(np.float32)


def fp8_channel_weights(N: int, K: int, seed: int = 0):
    """FP8 per-channel checkpoint stand-in: (codes uint8 [N, K] uniform over the finite e4m3
    codes, i.e. every byte but 0x7F and 0xFF; row scale float32 [N] = 2^u, u uniform in
    [-12, -6])."""
    idx = uniform_ints(N * K, 0, 253, seed, T_W8)
    codes = (idx + (idx >= 0x7F)).astype(np.uint8)  # skip 0x7F (and so end below 0xFF)
    u = uniform(seed, T_W8S, N) * 6.0 - 12.0
    return codes.reshape(N, K), np.exp2(u).astype(np.float32)


def bf16_weights(N: int, K: int, seed: int = 0, sigma: float = 0.02) -> np.ndarray:
    """bf16 bits [N, K] of N(0, sigma) weights."""
    return to_bf16_bits(normal(seed, T_WB, N * K).reshape(N, K) * sigma)


def int4_asym_zeros(N: int, K: int, seed: int = 0) -> np.ndarray:
    """qzeros int32 [K/128, ceil(N/8)] of uniform nibbles."""
    nz = (N + 7) // 8
    words = (u64(seed, T_QZ, (K // 128) * nz) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return words.reshape(K // 128, nz).view(np.int32)


def int5_weights(N: int, K: int, seed: int = 0):
    """int5 group-128 stand-in: uniform 5-bit codes as (qweight int32 [K/8, N] of the low
    nibbles, qhigh uint8 [K/8, N] of the fifth bits, bit j of byte (i, n) for k = 8i + j,
    scales fp16 bits uint16 [K/128, N] ~ |N(0, 0.0015)|, half the int4 spread for the doubled
    code range)."""
    n_words = (K // 8) * N
    q = u64(seed, T_QW, (n_words + 1) // 2).view(np.uint32)[:n_words]
    qweight = q.view(np.int32).reshape(K // 8, N).copy()
    qhigh = uniform_bytes(K // 8, N, seed, T_QH)
    s = np.abs(normal(seed, T_QS, (K // 128) * N) * 0.0015).astype(np.float16)
    scales = s.view(np.uint16).reshape(K // 128, N).copy()
    return qweight, qhigh, scales


def int5_zeros(N: int, K: int, seed: int = 0) -> np.ndarray:
    """Per (group, column) zero points, uint8 [K/128, N], uniform in 0..31."""
    return uniform_ints((K // 128) * N, 0, 31, seed, T_Z5).astype(np.uint8).reshape(K // 128, N)
