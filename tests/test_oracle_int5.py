"""Pins for the oracle's int5 group-128 GEMM ("vllm-radiance (MXFP4)", section "int5 (W5A8)":
5-bit codes c with value c - 16, the low nibbles in the int4 word layout and the fifth bit in a
plane of one byte per word; the zero point folded as for int4).

Independent checks: a numpy restatement that reads the plane with ``np.unpackbits``; exact
reductions to the int4 oracle (itself pinned in test_oracle_actquant_gemm.py) when the fifth
bits are constant; hand-built planes whose outputs are known in closed form and that tell the
two bit orders apart; and a pure-Python brute force on a tiny case.
"""
import numpy as np
import torch

from int4_quantized_linear_gb300 import synth


def fp8_to_f64(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def independent_int5_ref(xq, sc, qw, qh, s16, zeros=None):
    """Codes from numpy bit unpacking (little bit order: bit j is k = 8i + j), then a float64 dot."""
    K = xq.shape[1]
    N = qw.shape[1]
    words = qw.view(np.uint32)
    lo = np.stack([(words >> np.uint32(4 * j)) & np.uint32(0xF) for j in range(8)], 1).reshape(K, N)
    hi = np.unpackbits(qh[:, None, :], axis=1, bitorder="little").reshape(K, N)
    c = lo.astype(np.float64) + 16.0 * hi
    z = np.full((K // 128, N), 16.0) if zeros is None else zeros.astype(np.float64)
    s = s16.view(np.float16).astype(np.float64)
    w = (c - np.repeat(z, 128, axis=0)) * np.repeat(s, 128, axis=0)
    return sc.astype(np.float64)[:, None] * (fp8_to_f64(xq) @ w)


def test_int5_vs_independent(orc):
    M, N, K = 3, 40, 384
    x = synth.activations(M, K, seed=8)
    qw, qh, s16 = synth.int5_weights(N, K, seed=8)
    z = synth.int5_zeros(N, K, seed=8)
    xq, sc = orc.act_quant(x)
    for zeros in (None, z):
        out = orc.int5g128_linear(xq, sc, qw, qh, s16, zeros)
        ref = independent_int5_ref(xq, sc, qw, qh, s16, zeros)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        im = np.array([2, 0, 1, 0]); inn = np.array([39, 8, 17, 0])
        assert np.array_equal(orc.int5g128_linear_pairs(xq, sc, qw, qh, s16, zeros, im, inn), out[im, inn])


def test_int5_reduces_to_int4(orc):
    # fifth bits all 0 with zero point 8, or all 1 with zero point 24: c - z = nibble - 8, the
    # symmetric int4 value; same terms in the same order, so the results are identical
    M, N, K = 2, 24, 256
    x, qw, s16, _ = synth.int4_case(M, N, K, seed=9)
    xq, sc = orc.act_quant(x)
    ref = orc.int4g128_linear(xq, sc, qw, s16)
    qh0 = np.zeros((K // 8, N), np.uint8)
    assert np.array_equal(orc.int5g128_linear(xq, sc, qw, qh0, s16, np.full((K // 128, N), 8, np.uint8)), ref)
    qh1 = np.full((K // 8, N), 0xFF, np.uint8)
    assert np.array_equal(orc.int5g128_linear(xq, sc, qw, qh1, s16, np.full((K // 128, N), 24, np.uint8)), ref)


def test_int5_symmetric_is_zero_point_16(orc):
    M, N, K = 2, 16, 256
    x = synth.activations(M, K, seed=10)
    qw, qh, s16 = synth.int5_weights(N, K, seed=10)
    xq, sc = orc.act_quant(x)
    assert np.array_equal(orc.int5g128_linear(xq, sc, qw, qh, s16),
                          orc.int5g128_linear(xq, sc, qw, qh, s16, np.full((K // 128, N), 16, np.uint8)))


def test_int5_asym_matches_int4_asym(orc):
    # fifth bits 0 and zero points 1..16: the int4 asymmetric format holds the same weights
    # (zero point 1 + nibble of qzeros)
    M, N, K = 2, 16, 256
    x, qw, s16, _ = synth.int4_case(M, N, K, seed=11)
    z = (synth.int5_zeros(N, K, seed=11) % 16) + 1
    qz = np.zeros((K // 128, N // 8), np.uint32)
    for n in range(N):
        qz[:, n // 8] |= (z[:, n].astype(np.uint32) - 1) << np.uint32(4 * (n % 8))
    xq, sc = orc.act_quant(x)
    qh0 = np.zeros((K // 8, N), np.uint8)
    assert np.array_equal(orc.int5g128_linear(xq, sc, qw, qh0, s16, z),
                          orc.int4g128_asym_linear(xq, sc, qw, s16, qz.view(np.int32)))


def test_int5_closed_forms(orc):
    M, N, K = 2, 6, 256
    xq = np.zeros((M, K), np.uint8)
    xq[0] = 0x38                 # row 0: x = 1 at every k
    xq[1, 1::2] = 0x38           # row 1: x = 1 at odd k only
    sc = np.array([1.0, 2.0], np.float32)
    qw = np.zeros((K // 8, N), np.uint32)
    qh = np.zeros((K // 8, N), np.uint8)
    s16 = np.full((K // 128, N), 0x3C00, np.uint16)  # fp16 1.0
    qw[:, 0] = 0xFFFFFFFF; qh[:, 0] = 0xFF            # column 0: code 31 -> +15
    # column 1: codes 0 -> -16 (all zero)
    qh[:, 2] = 0x01                                    # column 2: code 16 at k % 8 == 0, else 0
    qh[:, 3] = 0x80                                    # column 3: code 16 at k % 8 == 7, else 0
    qw[:, 4] = 0x00000001; qh[:, 4] = 0x01             # column 4: code 17 at k % 8 == 0 (+1), else -16
    qh[:, 5] = 0xFF; s16[1, 5] = 0x3800                # column 5: code 16 -> 0 everywhere
    out = orc.int5g128_linear(xq, sc, qw.view(np.int32), qh, s16)
    assert out[0, 0] == 15.0 * K and out[0, 1] == -16.0 * K
    assert out[0, 2] == -16.0 * (K * 7 // 8) and out[0, 3] == -16.0 * (K * 7 // 8)
    # odd k only: k % 8 in {1, 3, 5, 7}; bit 0 never lands there, bit 7 lands on one of four
    assert out[1, 2] == 2.0 * -16.0 * (K // 2) and out[1, 3] == 2.0 * -16.0 * (K * 3 // 8)
    assert out[0, 4] == (K // 8) * 1.0 + (K * 7 // 8) * -16.0
    assert out[0, 5] == 0.0 and out[1, 5] == 0.0
    # per-column zero points: column 1 with z = 0 gives 0, column 0 with z = 31 gives 0
    z = np.full((K // 128, N), 16, np.uint8)
    z[:, 1] = 0; z[:, 0] = 31
    out = orc.int5g128_linear(xq, sc, qw.view(np.int32), qh, s16, z)
    assert out[0, 0] == 0.0 and out[0, 1] == 0.0 and out[0, 2] == -16.0 * (K * 7 // 8)


def test_int5_brute_force_tiny(orc):
    M, N, K = 2, 3, 128
    x = synth.activations(M, K, seed=12)
    qw, qh, s16 = synth.int5_weights(N, K, seed=12)
    z = synth.int5_zeros(N, K, seed=12)
    xq, sc = orc.act_quant(x)
    xv = fp8_to_f64(xq)
    s = s16.view(np.float16).astype(np.float64)
    words = qw.view(np.uint32)
    out = orc.int5g128_linear(xq, sc, qw, qh, s16, z)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                c = (int(words[k // 8, n]) >> (4 * (k % 8))) & 15
                if (int(qh[k // 8, n]) >> (k % 8)) & 1:
                    c += 16
                acc += xv[m, k] * (c - int(z[k // 128, n])) * s[k // 128, n]
            assert out[m, n] == float(sc[m]) * acc
