"""Pins for the oracle's W4A4 path ("vllm-radiance (MXFP4)", section "Native MXFP4": MXFP4
weights and activations, group 32, e8m0 scales; activations by the OCP rule that
"radiance_nvfp4.py" names ocp).

Independent checks: a brute-force nearest-grid search with ties to the even code for the
activation codes and numpy's frexp for the block exponent; an exact reduction of the GEMM to
the W4A8 oracle when every activation block of a row shares its exponent (the e2m1 values are
all e4m3 values, so the two definitions then sum the same terms); a numpy restatement; and
closed forms.
"""
import numpy as np
import torch

from int4_quantized_linear_gb300 import synth

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
# e4m3 encodings of the e2m1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 (bias 7, 3 mantissa bits)
E2M1_AS_E4M3 = np.array([0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C], np.uint8)


def e2m1_value(codes):
    codes = np.asarray(codes)
    return GRID[codes & 7] * np.where(codes & 8, -1.0, 1.0)


def unpack(packed):
    return np.stack([packed & 0x0F, packed >> 4], -1).reshape(packed.shape[0], -1)


def test_act_quant_mxfp4_bruteforce(orc):
    M, K = 3, 256
    x = synth.activations(M, K, seed=21, outliers=True)
    xa, xe = orc.act_quant_mxfp4(x)
    xf = synth.bf16_bits_to_float(x).astype(np.float64).reshape(M, K // 32, 32)
    amax = np.abs(xf).max(-1)
    _, p = np.frexp(amax)                       # amax = f * 2^p, f in [0.5, 1)
    e = np.where(amax > 0, p - 1 - 2, 0)        # floor(log2 amax) - 2
    assert np.array_equal(xe.astype(np.int64), e + 127)
    v = np.abs(xf) * np.exp2(-e)[..., None]
    d = np.abs(v[..., None] - GRID)             # distance to every grid point
    best = d.min(-1, keepdims=True)
    ties = d == best
    idx = np.where(ties[..., ::2].any(-1) & (ties.sum(-1) > 1),  # a tie: take the even index
                   np.argmax(ties & (np.arange(8) % 2 == 0), -1), np.argmax(ties, -1))
    idx = np.where(v >= 6.0, 7, idx)
    code = idx + 8 * ((xf < 0) & (idx != 0))
    assert np.array_equal(unpack(xa).reshape(M, K // 32, 32), code)


def test_a4_reduces_to_w4a8(orc):
    # rows whose activation blocks share one exponent E_m: W4A4 equals the W4A8 definition fed the
    # e4m3 encodings of the same e2m1 values and the token scale 2^(E_m - 127)
    M, N, K = 3, 40, 512
    _, wp, we = synth.decode_case(1, N, K, seed=22)
    codes = synth.uniform_bytes(M, K, 22, 91) & 0x0F
    xa = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    E = np.array([127, 120, 131])
    xe = np.repeat(E[:, None], K // 32, axis=1).astype(np.uint8)
    xq = E2M1_AS_E4M3[codes & 7] | np.where(codes & 8, 0x80, 0).astype(np.uint8)
    xs = np.exp2(E - 127.0).astype(np.float32)
    assert np.array_equal(orc.mxfp4_a4_linear(xa, xe, wp, we), orc.mxfp4_linear(xq, xs, wp, we))


def test_a4_vs_independent(orc):
    M, N, K = 4, 48, 384
    x = synth.activations(M, K, seed=23)
    xa, xe = orc.act_quant_mxfp4(x)
    _, wp, we = synth.decode_case(1, N, K, seed=23)
    out = orc.mxfp4_a4_linear(xa, xe, wp, we)
    xv = e2m1_value(unpack(xa)) * np.repeat(np.exp2(xe.astype(np.float64) - 127), 32, axis=1)
    wv = e2m1_value(unpack(wp)) * np.repeat(np.exp2(we.astype(np.float64) - 127), 32, axis=1)
    ref = xv @ wv.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    im = np.array([0, 3, 2]); inn = np.array([47, 0, 21])
    assert np.array_equal(orc.mxfp4_a4_linear_pairs(xa, xe, wp, we, im, inn), out[im, inn])


def test_a4_closed_forms(orc):
    M, N, K = 2, 2, 256
    xa = np.full((M, K // 2), 0x22, np.uint8)     # x = +1 everywhere
    xa[1] = 0xAA                                   # row 1: x = -1
    xe = np.full((M, K // 32), 127, np.uint8)
    xe[1, :4] = 128                                # row 1, first 128 k: x = -2
    wp = np.full((N, K // 2), 0x22, np.uint8)      # W = +1
    wp[1] = 0x7F                                   # column 1: -6 at even k (code 15), +6 at odd (7)
    we = np.full((N, K // 32), 127, np.uint8)
    we[1] = 126                                    # column 1 halved
    out = orc.mxfp4_a4_linear(xa, xe, wp, we)
    assert out[0, 0] == K and out[1, 0] == -2.0 * 128 - 1.0 * 128
    assert out[0, 1] == 0.0 and out[1, 1] == 0.0   # +3 and -3 alternate along k
    # a bf16 row of exact grid values times 2^-4 quantizes to those codes with e8m0 127 - 4 - ...
    x = np.zeros((1, 64), np.float32)
    x[0, :8] = np.array(GRID) * 2.0 ** -4         # block 0 amax 6 * 2^-4: e = floor(log2) - 2 = -4
    x[0, 32] = -4.0                                # block 1 amax 4: e = 0, code -4 -> 14
    xa1, xe1 = orc.act_quant_mxfp4(synth.to_bf16_bits(x))
    assert xe1[0, 0] == 127 - 4 and xe1[0, 1] == 127
    assert np.array_equal(unpack(xa1)[0, :8], np.arange(8)) and unpack(xa1)[0, 32] == 14
    assert not unpack(xa1)[0, 33:].any()
