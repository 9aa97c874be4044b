"""Pins for the oracle's per-token activation quant ("radiance_autoround.py",
autoround_linear: dynamic per-token fp8) and its dequantize-and-matmul GEMMs ("vllm-radiance
(MXFP4)", "The W4A8 fp8-WMMA kernel"; "radiance_autoround.py", _exact_ref).

Independent references: numpy float32 division plus a brute-force e4m3 grid search for the
codes; the library fp8 dtype, numpy bit unpacking and a float64 matmul for the GEMMs; and
hand-built inputs whose outputs are known in closed form.
"""
import numpy as np
import pytest
import torch

from int4_quantized_linear_gb300 import synth
from test_oracle_codecs import brute_e4m3

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def fp8_to_f64(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def test_act_quant_vs_bruteforce(orc):
    x = synth.activations(9, 384, seed=1, outliers=True)
    xq, sc = orc.act_quant(x)
    xf = synth.bf16_bits_to_float(x)
    amax = np.max(np.abs(xf), axis=1)
    assert np.array_equal(sc, (amax / np.float32(448.0)).astype(np.float32))
    q = (xf / sc[:, None]).astype(np.float32)  # correctly rounded fp32 division
    assert np.array_equal(xq, brute_e4m3(q))
    # the amax element lands exactly on +-448
    for m in range(9):
        k = int(np.argmax(np.abs(xf[m])))
        assert xq[m, k] == (0xFE if xf[m, k] < 0 else 0x7E)


def test_act_quant_zero_row_and_exact_row(orc):
    # row 0 all zeros (one -0): scale 1, codes signed zeros
    # row 1 values j * amax / 448 for representable j: every code decodes back exactly
    K = 64
    x = np.zeros((2, K), np.float32)
    x[0, 3] = -0.0
    vals = np.array([448, 256, 1, 0.5, 3.5, 0.001953125, -224, -7, 13, 0], np.float64)
    amax = 2.0 ** -3 * 448
    x[1, :vals.size] = vals * (amax / 448.0)
    xb = synth.to_bf16_bits(x)
    xq, sc = orc.act_quant(xb)
    assert sc[0] == 1.0 and np.all(xq[0] == np.where(np.signbit(x[0]), 0x80, 0))
    assert sc[1] == np.float32(amax / 448.0)
    assert np.array_equal(fp8_to_f64(xq[1, :vals.size]) * sc[1], x[1, :vals.size].astype(np.float64))


def independent_mxfp4_ref(xq, sc, wp, we):
    N = wp.shape[0]
    codes = np.stack([wp & 0x0F, wp >> 4], -1).reshape(N, -1)
    w = GRID[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    w = w * np.repeat(2.0 ** (we.astype(np.float64) - 127.0), 32, axis=1)
    return (fp8_to_f64(xq) @ w.T) * sc.astype(np.float64)[:, None]


def independent_int4_ref(xq, sc, qw, s16):
    K8, N = qw.shape
    u = qw.view(np.uint32)
    codes = np.stack([(u >> np.uint32(4 * j)) & np.uint32(0xF) for j in range(8)], 1)  # [K/8, 8, N]
    codes = codes.reshape(8 * K8, N).astype(np.float64)
    s = np.repeat(s16.view(np.float16).astype(np.float64), 128, axis=0)
    w = (codes - 8.0) * s  # [K, N]
    return (fp8_to_f64(xq) @ w) * sc.astype(np.float64)[:, None]


def test_mxfp4_linear_vs_independent(orc):
    M, N, K = 5, 48, 320
    x, wp, we = synth.decode_case(M, N, K, seed=3)
    xq, sc = orc.act_quant(x)
    out = orc.mxfp4_linear(xq, sc, wp, we)
    ref = independent_mxfp4_ref(xq, sc, wp, we)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    im = np.array([0, 4, 2, 1]); inn = np.array([0, 47, 13, 30])
    assert np.array_equal(orc.mxfp4_linear_pairs(xq, sc, wp, we, im, inn), out[im, inn])


def test_mxfp4_linear_closed_forms(orc):
    # x codes 1.0 (0x38), W codes +1.0 (0x2) with e8m0 127: out = scale * K exactly
    M, N, K = 2, 3, 256
    xq = np.full((M, K), 0x38, np.uint8)
    sc = np.array([1.0, 0.5], np.float32)
    wp = np.full((N, K // 2), 0x22, np.uint8)
    we = np.full((N, K // 32), 127, np.uint8)
    out = orc.mxfp4_linear(xq, sc, wp, we)
    assert np.array_equal(out, np.array([[256.0] * 3, [128.0] * 3]))
    # low nibble = even k: W row 0 = +6 at even k, -0.5 at odd k (byte 0x97); e8m0 = 126 halves
    wp[0] = 0x97
    we[0] = 126
    xq[0, 1::2] = 0x40  # x = 2.0 at odd k
    out = orc.mxfp4_linear(xq, sc, wp, we)
    assert out[0, 0] == (128 * 6.0 * 1.0 + 128 * -0.5 * 2.0) * 0.5
    # all-zero e8m0-scaled rows: a zero x row gives exact zeros
    xq[1] = 0
    assert not orc.mxfp4_linear(xq, sc, wp, we)[1].any()


def test_int4_linear_vs_independent(orc):
    M, N, K = 3, 24, 384
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=5)
    xq, sc = orc.act_quant(x)
    out = orc.int4g128_linear(xq, sc, qw, s16)
    ref = independent_int4_ref(xq, sc, qw, s16)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    im = np.array([0, 2, 1]); inn = np.array([23, 0, 7])
    assert np.array_equal(orc.int4g128_linear_pairs(xq, sc, qw, s16, im, inn), out[im, inn])


def test_int4_linear_closed_forms(orc):
    # symmetric zero point 8: code 9 -> +1, code 8 -> 0, code 0 -> -8 (qzeros 0x77777777)
    M, N, K = 1, 2, 256
    xq = np.full((M, K), 0x38, np.uint8)  # x = 1
    sc = np.array([2.0], np.float32)
    qw = np.zeros((K // 8, N), np.uint32)
    qw[:, 0] = 0x99999999           # every k: +1
    qw[:, 1] = 0x08080808           # k = 8i + j: j even -> -8, j odd -> 0
    s16 = np.full((K // 128, N), 0x3C00, np.uint16)  # fp16 1.0
    s16[1, 1] = 0x3800              # second group of column 1 scaled by 0.5
    out = orc.int4g128_linear(xq, sc, qw.view(np.int32), s16)
    assert out[0, 0] == 2.0 * 256
    assert out[0, 1] == 2.0 * (64 * -8.0 * 1.0 + 64 * -8.0 * 0.5)


# --- asymmetric int4 g128 ("vllm-radiance (MXFP4)", ParoQuant: asymmetric zero point)

def independent_int4_asym_ref(xq, sc, qw, s16, qz):
    """Numpy restatement: w[k, n] = (c - (1 + z nibble)) * s, then the dot in float64."""
    K = xq.shape[1]
    N = qw.shape[1]
    words = qw.view(np.uint32)
    c = np.stack([(words >> np.uint32(4 * j)) & np.uint32(0xF) for j in range(8)], 1).reshape(K, N).astype(np.float64)
    zw = qz.view(np.uint32)
    z = np.empty((K // 128, N))
    for n in range(N):
        z[:, n] = 1 + ((zw[:, n // 8] >> np.uint32(4 * (n % 8))) & np.uint32(0xF)).astype(np.float64)
    s = torch.from_numpy(s16.view(np.float16)).to(torch.float64).numpy()
    w = (c - np.repeat(z, 128, axis=0)) * np.repeat(s, 128, axis=0)
    xv = torch.from_numpy(xq).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return sc.astype(np.float64)[:, None] * (xv @ w)


def test_int4_asym_vs_independent(orc):
    M, N, K = 3, 40, 384
    x, qw, s16, _ = synth.int4_case(M, N, K, seed=6)
    qz = synth.int4_asym_zeros(N, K, seed=6)
    xq, sc = orc.act_quant(x)
    out = orc.int4g128_asym_linear(xq, sc, qw, s16, qz)
    ref = independent_int4_asym_ref(xq, sc, qw, s16, qz)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    im = np.array([2, 0, 1]); inn = np.array([39, 8, 17])
    assert np.array_equal(orc.int4g128_asym_linear_pairs(xq, sc, qw, s16, qz, im, inn), out[im, inn])


def test_int4_asym_reduces_to_symmetric(orc):
    # qzeros 0x77777777 is the zero point 8 of the symmetric format
    M, N, K = 2, 24, 256
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=7)
    assert np.all(qz.view(np.uint32) == 0x77777777)
    xq, sc = orc.act_quant(x)
    assert np.array_equal(orc.int4g128_asym_linear(xq, sc, qw, s16, qz[:, :3]), orc.int4g128_linear(xq, sc, qw, s16))


def test_int4_asym_closed_forms(orc):
    # x = 1, scale 1: column 0 codes 5 with zero point 3 (nibble 2) -> +2 per k; column 1 codes
    # 0 with zero point 16 (nibble 15) -> -16 per k; column 9 codes 15 with zero point 1 -> +14
    M, N, K = 1, 10, 128
    xq = np.full((M, K), 0x38, np.uint8)
    sc = np.array([1.0], np.float32)
    qw = np.zeros((K // 8, N), np.uint32)
    qw[:, 0] = 0x55555555
    qw[:, 9] = 0xFFFFFFFF
    s16 = np.full((K // 128, N), 0x3C00, np.uint16)
    qz = np.zeros((1, 2), np.uint32)
    qz[0, 0] = 0x000000F2           # column 0: nibble 2, column 1: nibble 15
    qz[0, 1] = 0x00000000           # column 9 (word 1, nibble 1): nibble 0
    out = orc.int4g128_asym_linear(xq, sc, qw.view(np.int32), s16, qz.view(np.int32))
    assert out[0, 0] == 2.0 * K and out[0, 1] == -16.0 * K and out[0, 9] == 14.0 * K
