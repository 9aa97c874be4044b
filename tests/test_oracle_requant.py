"""Pins for the oracle's NVFP4 -> MXFP4 requant ("radiance_nvfp4.py": dequant_nvfp4,
_block_exponent, e2m1_index, _encode_blocks, quant_mxfp4, process_weights_after_loading).

Each check compares the oracle with something independent of it: closed forms of the
exponent rules, a brute-force exponent search, brute-force nearest-grid encoding with exact
float64 errors, hand-built blocks whose result is known, and an independent numpy dequant.
"""
import numpy as np
import pytest
import torch

from int4_quantized_linear_gb300 import synth

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def brute_exponent(amax: float, mode: str) -> int:
    """Search e in [-127, 127]: ocp -> largest e with 4 * 2^e <= amax (floor(log2)-2);
    noclip -> smallest e with amax <= 6 * 2^e."""
    if amax == 0:
        return 0
    es = range(-127, 128)
    if mode == "ocp":
        ok = [e for e in es if 4.0 * 2.0 ** e <= amax]
        return max(ok) if ok else -127
    ok = [e for e in es if amax <= 6.0 * 2.0 ** e]
    return min(ok) if ok else 127


def brute_encode(w: np.ndarray, e: int):
    """Nearest grid magnitude to |w| / 2^e clamped to 6, ties to the even index; exact
    float64 squared error of the dequantized block against w."""
    v = np.abs(w.astype(np.float64)) / 2.0 ** e
    c = np.minimum(v, 6.0)
    d = np.abs(GRID[None, :] - c[:, None])
    idx = np.empty(len(w), np.int64)
    for i in range(len(w)):
        best = np.nonzero(d[i] == d[i].min())[0]
        idx[i] = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
    q = GRID[idx] * 2.0 ** e * np.where(np.signbit(w), -1.0, 1.0)
    err = float(np.sum((q - w.astype(np.float64)) ** 2))
    codes = (idx | np.where(np.signbit(w) & (idx != 0), 8, 0)).astype(np.uint8)
    return codes, err


def independent_dequant_nvfp4(packed, scale, div):
    """Numpy restatement of dequant_nvfp4 for the pins (library fp8 decode for the scales)."""
    lo = packed & 0x0F
    hi = packed >> 4
    codes = np.stack([lo, hi], -1).reshape(packed.shape[0], -1)
    g = GRID[codes & 7].astype(np.float32) * np.where(codes & 8, -1.0, 1.0).astype(np.float32)
    s = torch.from_numpy(scale).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    s = (s / np.float32(div)).astype(np.float32)
    return (g * np.repeat(s, 16, axis=1)).astype(np.float32)


@pytest.mark.parametrize("mode", ["ocp", "noclip"])
def test_block_exponent_vs_bruteforce(orc, mode):
    rng_vals = np.abs(synth.normal(3, 1, 400)) * 10.0 ** synth.uniform_ints(400, -12, 4, 3, 2)
    special = []
    for e in range(-30, 30):
        for base in (4.0, 6.0, 3.0, 8.0):
            x = np.float32(base * 2.0 ** e)
            special += [x, np.nextafter(x, np.float32(0)), np.nextafter(x, np.float32(np.inf))]
    for a in np.concatenate([rng_vals.astype(np.float32), np.array(special, np.float32)]):
        assert orc.block_exponent(float(a), mode) == brute_exponent(float(a), mode), (a, mode)


def test_block_exponent_landmarks(orc):
    assert orc.block_exponent(0.0, "ocp") == 0 and orc.block_exponent(0.0, "noclip") == 0
    for e in (-20, -3, 0, 5):
        assert orc.block_exponent(6.0 * 2.0 ** e, "noclip") == e          # fits without clipping
        assert orc.block_exponent(4.0 * 2.0 ** e, "ocp") == e             # amax lands on 4
        assert orc.block_exponent(7.9 * 2.0 ** e, "ocp") == e             # [4, 8) -> e
        assert orc.block_exponent(6.01 * 2.0 ** e, "noclip") == e + 1
    assert orc.block_exponent(1e38, "noclip") == 124   # 1e38 / 6 = 2^123.6
    assert orc.block_exponent(1e-45, "noclip") == -127                    # clamped


def test_quant_block_all_zero(orc):
    for mode in ("ocp", "noclip", "mse"):
        e, codes, err = orc.quant_block(np.zeros(32, np.float32), mode)
        assert e == 0 and not codes.any() and err == 0.0


def test_quant_block_exact_grid_values(orc):
    # values that sit on the grid at exponent e (amax = 6 * 2^e): zero error, e kept by mse
    for e in (-9, 0, 3):
        g = np.tile(GRID, 4)
        sgn = np.where(np.arange(32) % 3 == 0, -1.0, 1.0)
        w = (g * sgn * 2.0 ** e).astype(np.float32)
        for mode in ("noclip", "mse"):
            ee, codes, err = orc.quant_block(w, mode)
            assert ee == e and err == 0.0
            assert np.array_equal(codes & 7, np.tile(np.arange(8), 4))


def test_quant_block_clipping_pays_off(orc):
    # one element at 3.2 and 31 at 0.3: noclip puts 3.2 on the [3, 6] grid (e = 0); one binade
    # finer clips it to 3.0 but halves the step for the other 31, and the mse rule takes it.
    w = np.array([3.2] + [0.3] * 31, np.float32)
    assert orc.quant_block(w, "noclip")[0] == 0
    e, codes, err = orc.quant_block(w, "mse")
    assert e == -1
    assert codes[0] == 7  # 6.4 clamps to the top code
    _, exact = brute_encode(w, -1)
    assert abs(err - exact) <= 1e-6 * exact


def test_quant_block_sign_rule(orc):
    # -0 and negatives that round to index 0 stay code 0, never 8
    w = np.array([6.0, -0.0, -1e-3, -0.2, -0.26] + [0.0] * 27, np.float32)
    e, codes, _ = orc.quant_block(w, "noclip")
    assert e == 0
    assert list(codes[:5]) == [7, 0, 0, 0, 9]


def test_quant_block_vs_bruteforce(orc):
    n_blocks = 600
    w_all = synth.normal(11, 1, 32 * n_blocks).reshape(n_blocks, 32) * 0.02
    # heavy-tailed rows and an outlier per block in a third of the blocks
    w_all[::3, 0] *= 8.0
    w_all = w_all.astype(np.float32)
    for w in w_all:
        amax = float(np.max(np.abs(w)))
        for mode in ("ocp", "noclip"):
            e, codes, err = orc.quant_block(w, mode)
            assert e == brute_exponent(amax, mode)
            bc, berr = brute_encode(w, e)
            assert np.array_equal(codes, bc)
            assert abs(err - berr) <= 1e-5 * berr + 1e-30
        e0 = brute_exponent(amax, "noclip")
        c0, r0 = brute_encode(w, e0)
        c1, r1 = brute_encode(w, e0 - 1)
        e, codes, err = orc.quant_block(w, "mse")
        if abs(r1 - r0) > 1e-5 * max(r0, r1):  # not a near-tie that fp32 summation decides
            exp_e = e0 - 1 if r1 < r0 else e0
            assert e == exp_e
            assert np.array_equal(codes, c1 if exp_e != e0 else c0)


def _nvfp4(N, K, parts, seed=0, gain2=1.0):
    gain = np.ones(N)
    gain[parts[0]:] = gain2
    w = synth.gaussian_weights(N, K, 0.02, seed, row_gain=gain)
    return w


def test_dequant_nvfp4_power_of_two_divisor_exact(orc):
    N, K = 8, 64
    packed = synth.uniform_bytes(N, K // 2, 5, 1)
    scale = synth.uniform_ints(N * K // 16, 0x20, 0x60, 5, 2).astype(np.uint8).reshape(N, K // 16)
    div = np.array([256.0], np.float32)
    out_p, out_e, es = orc.requant(packed, scale, div, [N], "noclip")
    w = independent_dequant_nvfp4(packed, scale, 256.0)
    # with a power-of-two divisor every product is exact: the squared norm is exact too
    assert es[0, 1] == pytest.approx(float(np.sum(w.astype(np.float64) ** 2)), rel=1e-12)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
def test_requant_rows_vs_independent(orc, mode):
    N, K = 64, 256
    parts = [40, 24]
    w = _nvfp4(N, K, parts, seed=2, gain2=0.25)
    packed, scale, div = orc.nvfp4_quantize(w, parts)
    assert div[0] != div[1]
    out_p, out_e, es = orc.requant(packed, scale, div, parts, mode)
    # independent dequant, per partition with its own divisor
    wd = np.concatenate([independent_dequant_nvfp4(packed[:40], scale[:40], div[0]),
                         independent_dequant_nvfp4(packed[40:], scale[40:], div[1])])
    lo = out_p & 0x0F
    hi = out_p >> 4
    codes = np.stack([lo, hi], -1).reshape(N, K)  # low nibble = even k
    err_tot = np.zeros(2)
    for n in range(N):
        for b in range(K // 32):
            blk = wd[n, 32 * b:32 * b + 32]
            e = int(out_e[n, b]) - 127
            amax = float(np.max(np.abs(blk)))
            if mode != "mse":
                assert e == brute_exponent(amax, mode)
            else:
                assert e in (brute_exponent(amax, "noclip"), brute_exponent(amax, "noclip") - 1)
            bc, berr = brute_encode(blk, e)
            assert np.array_equal(codes[n, 32 * b:32 * b + 32], bc)
            err_tot[0 if n < 40 else 1] += berr
    ssq = [float(np.sum(wd[:40].astype(np.float64) ** 2)), float(np.sum(wd[40:].astype(np.float64) ** 2))]
    assert es[:, 0] == pytest.approx(err_tot, rel=1e-5)
    assert es[:, 1] == pytest.approx(ssq, rel=1e-9)
    # the dequantized MXFP4 reproduces the error sums
    deq = orc.dequant_mxfp4(out_p, out_e)
    assert float(np.sum((deq[:40] - wd[:40]) ** 2)) == pytest.approx(es[0, 0], rel=1e-5)


def test_requant_partitions_are_independent(orc):
    N, K = 48, 128
    parts = [16, 32]
    w = _nvfp4(N, K, parts, seed=4, gain2=3.0)
    packed, scale, div = orc.nvfp4_quantize(w, parts)
    joint = orc.requant(packed, scale, div, parts, "mse")
    a = orc.requant(packed[:16], scale[:16], div[:1], [16], "mse")
    b = orc.requant(packed[16:], scale[16:], div[1:], [32], "mse")
    assert np.array_equal(joint[0], np.concatenate([a[0], b[0]]))
    assert np.array_equal(joint[1], np.concatenate([a[1], b[1]]))
    with pytest.raises(ValueError):
        orc.requant(packed, scale, div, [16, 31], "mse")


def test_mse_never_worse_than_noclip(orc):
    N, K = 32, 512
    w = _nvfp4(N, K, [N], seed=6)
    packed, scale, div = orc.nvfp4_quantize(w, [N])
    r = {m: orc.rel_rms(orc.requant(packed, scale, div, [N], m)[2]) for m in ("ocp", "noclip", "mse")}
    assert r["mse"] <= r["noclip"] + 1e-12
    assert 0.0 < r["mse"] < 0.2


def test_nvfp4_producer_roundtrip(orc):
    N, K = 16, 128
    w = synth.gaussian_weights(N, K, 0.02, 9)
    packed, scale, div = orc.nvfp4_quantize(w, [N])
    assert div[0] == np.float32(2688.0) / np.float32(np.max(np.abs(w)))
    wd = independent_dequant_nvfp4(packed, scale, div[0])
    s = torch.from_numpy(scale).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = np.abs(w.astype(np.float64)) * float(div[0]) / np.repeat(s, 16, axis=1)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    q = np.abs(wd.astype(np.float64)) * float(div[0]) / np.repeat(s, 16, axis=1)
    assert np.all(np.abs(np.minimum(v, 6.0) - q) <= step / 2 + 1e-6)


# --- other requant sources ("radiance_nvfp4.py": RadianceFp8ChannelToMxfp4, RadianceBf16ToMxfp4)

def _fp8_checkpoint(N, K, seed):
    """An FP8 per-channel checkpoint built with torch's own e4m3 cast: scale[n] = amax_n / 448,
    codes = e4m3(w / scale)."""
    w = synth.gaussian_weights(N, K, 0.02, seed).astype(np.float32)
    s = (np.max(np.abs(w), axis=1) / np.float32(448.0)).astype(np.float32)
    q = torch.from_numpy(w / s[:, None]).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().copy(), s


def _check_against_brute(wd, out_p, out_e, es, mode):
    N, K = wd.shape
    codes = np.stack([out_p & 0x0F, out_p >> 4], -1).reshape(N, K)
    err = 0.0
    for n in range(N):
        for b in range(K // 32):
            blk = wd[n, 32 * b:32 * b + 32]
            e = int(out_e[n, b]) - 127
            amax = float(np.max(np.abs(blk)))
            if mode != "mse":
                assert e == brute_exponent(amax, mode)
            else:
                assert e in (brute_exponent(amax, "noclip"), brute_exponent(amax, "noclip") - 1)
            bc, berr = brute_encode(blk, e)
            assert np.array_equal(codes[n, 32 * b:32 * b + 32], bc)
            err += berr
    assert es[0, 0] == pytest.approx(err, rel=1e-5)
    assert es[0, 1] == pytest.approx(float(np.sum(wd.astype(np.float64) ** 2)), rel=1e-9)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
def test_requant_fp8_channel_vs_independent(orc, mode):
    N, K = 24, 256
    w8, s = _fp8_checkpoint(N, K, 11)
    out_p, out_e, es = orc.requant_fp8_channel(w8, s, mode)
    # independent dequant: torch's e4m3 decode, then one fp32 product per element
    wd = (torch.from_numpy(w8).view(torch.float8_e4m3fn).to(torch.float32).numpy() * s[:, None]).astype(np.float32)
    _check_against_brute(wd, out_p, out_e, es, mode)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
def test_requant_bf16_vs_independent(orc, mode):
    N, K = 16, 320
    wb = synth.to_bf16_bits(synth.gaussian_weights(N, K, 0.02, 12).astype(np.float64))
    out_p, out_e, es = orc.requant_bf16(wb, mode)
    wd = (wb.astype(np.uint32) << 16).view(np.float32)
    _check_against_brute(wd, out_p, out_e, es, mode)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
def test_requant_sources_agree_on_exact_weights(orc, mode):
    # NVFP4 with a power-of-two divisor dequantizes exactly to values with at most six
    # significant bits, exact in bf16: the bf16 source must give the NVFP4 result bit for bit
    N, K = 12, 128
    packed = synth.uniform_bytes(N, K // 2, 13, 1)
    scale = synth.uniform_ints(N * K // 16, 0x28, 0x48, 13, 2).astype(np.uint8).reshape(N, K // 16)
    ref = orc.requant(packed, scale, np.array([1024.0], np.float32), [N], mode)
    wd = independent_dequant_nvfp4(packed, scale, 1024.0)
    wb = ((wd.view(np.uint32) >> 16)).astype(np.uint16)
    assert np.array_equal((wb.astype(np.uint32) << 16).view(np.float32), wd)
    got = orc.requant_bf16(wb, mode)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    assert got[2][0, 0] == ref[2][0, 0] and got[2][0, 1] == ref[2][0, 1]


def test_requant_fp8_channel_closed_forms(orc):
    # codes 0x38 (1.0) and 0xB8 (-1.0) with scale 2: every block is +-2 -> noclip e = -1,
    # index 6 (value 4), no error; an all-zero row gives e = 0 and code 0
    w8 = np.full((3, 64), 0x38, np.uint8)
    w8[1, ::2] = 0xB8
    w8[2] = 0
    out_p, out_e, es = orc.requant_fp8_channel(w8, np.array([2.0, 2.0, 5.0], np.float32), "noclip")
    assert np.all(out_e[:2] == 126) and np.all(out_e[2] == 127)
    assert np.all(out_p[0] == 0x66) and np.all(out_p[1] == 0x6E) and np.all(out_p[2] == 0)
    assert es[0, 0] == 0.0 and es[0, 1] == 2 * 64 * 4.0
    with pytest.raises(ValueError):
        orc.requant_fp8_channel(np.zeros((2, 48), np.uint8), np.ones(2, np.float32), "ocp")
