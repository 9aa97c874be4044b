"""GPU parity: every kernel against the oracle, through the C ABI (via the binding).

Bit-exact: act-quant codes and scales, requant codes and e8m0 bytes.  GEMMs: the acceptance
bound of helpers.gemm_check against the oracle fed the same fp8 codes.  Sizes span several
tiles with ragged tails; the full workload sizes are checked on sampled outputs.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_to_f64, gemm_check, host, to_dev, to_dev_bf16, to_dev_fp16
from int4_quantized_linear_gb300 import synth

pytestmark = pytest.mark.gpu

GATE_UP, DOWN, QKV = synth.GATE_UP, synth.DOWN, synth.QKV


# ---------------------------------------------------------------------------- act quant

@pytest.mark.parametrize("M,K", [(1, 512), (3, 520), (64, 5120), (5, 17408), (257, 1024)])
def test_act_quant_bit_exact(lib, orc, M, K):
    x = synth.activations(M, K, seed=M + K, outliers=True, lognormal_rows=True)
    xq, xs = lib.act_quant(to_dev_bf16(x))
    rq, rs = orc.act_quant(x)
    assert np.array_equal(host(xs), rs)
    assert np.array_equal(host(xq), rq)


def test_act_quant_edge_rows(lib, orc):
    K = 256
    x = np.zeros((4, K), np.float32)
    x[0, 7] = -0.0                       # all-zero row with a signed zero
    x[1] = 1e-30 * (np.arange(K) - 100)  # tiny magnitudes, negatives that round to -0
    x[2, :] = 3.0
    x[2, 5] = -448.0 * 1024              # huge amax
    x[3] = synth.bf16_bits_to_float(synth.activations(1, K, seed=9))[0]
    xb = synth.to_bf16_bits(x)
    xq, xs = lib.act_quant(to_dev_bf16(xb))
    rq, rs = orc.act_quant(xb)
    assert np.array_equal(host(xs), rs)
    assert np.array_equal(host(xq), rq)


@pytest.mark.slow
def test_act_quant_full_prefill(lib, orc):
    M, K = 4096, 17408
    x = synth.activations(M, K, seed=1, lognormal_rows=True)
    xq, xs = lib.act_quant(to_dev_bf16(x))
    rq, rs = orc.act_quant(x)
    assert np.array_equal(host(xs), rs)
    assert np.array_equal(host(xq), rq)


def test_act_quant_rejects(lib):
    x = torch.zeros((2, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.act_quant(x)


# ---------------------------------------------------------------------------- requant

def _nvfp4_case(orc, N, K, parts, seed, gain2=1.0):
    gain = np.ones(N)
    gain[parts[0]:] = gain2
    w = synth.gaussian_weights(N, K, 0.02, seed, row_gain=gain)
    return orc.nvfp4_quantize(w, parts)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
@pytest.mark.parametrize("N,K,parts,gain2", [(96, 512, [40, 56], 0.25), (33, 160, [33], 1.0),
                                             (300, 2048, [100, 150, 50], 4.0)])
def test_requant_bit_exact(lib, orc, mode, N, K, parts, gain2):
    packed, scale, div = _nvfp4_case(orc, N, K, parts, seed=N, gain2=gain2)
    gp, ge, gs = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), parts, mode)
    rp, re_, rs = orc.requant(packed, scale, div, parts, mode)
    assert np.array_equal(host(ge), re_)
    assert np.array_equal(host(gp), rp)
    _check_err_ssq(host(gs), rs)


def _check_err_ssq(got, ref):
    """Requant error report: the error column sums the same fp32 block errors on both sides
    (fp64 across blocks, order aside); the weight-energy column is a float-precision statistic
    (fp32 per 32-block on the GPU, fp64 in the oracle), checked to 2e-6 relative -- the relRMS
    it feeds is specified to 1e-5 relative ("radiance_nvfp4.py",
    process_weights_after_loading)."""
    assert np.allclose(got[:, 0], ref[:, 0], rtol=1e-9, atol=0)
    assert np.allclose(got[:, 1], ref[:, 1], rtol=2e-6, atol=0)


def test_requant_degenerate_blocks(lib, orc):
    # all-zero blocks, one-element blocks, subnormal-scale blocks, huge divisor
    N, K = 8, 128
    packed = synth.uniform_bytes(N, K // 2, 3, 1)
    packed[0] = 0
    packed[1, :16] = 0x08                # -0 codes only
    scale = synth.uniform_ints(N * K // 16, 0, 0x7e, 3, 2).astype(np.uint8).reshape(N, K // 16)
    scale[2] = 0x01                      # subnormal e4m3 scales
    scale[3, :2] = 0
    div = np.array([1.0e6], np.float32)
    for mode in ("ocp", "noclip", "mse"):
        gp, ge, gs = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), [N], mode)
        rp, re_, rs = orc.requant(packed, scale, div, [N], mode)
        assert np.array_equal(host(ge), re_)
        assert np.array_equal(host(gp), rp)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
def test_requant_without_error_sums(lib, orc, mode):
    """Without the error report the kernel is built without the error arithmetic (outside the mse
    rule): codes and e8m0 must still match the oracle bit for bit, for every source.  The blocks
    mix large values with tiny negatives that round to a zero index (code 0, never 8)."""
    N, K = 70, 384
    packed = synth.uniform_bytes(N, K // 2, 11, 1)
    packed[3, :8] = 0x99                 # -0.5 in both nibbles next to large values
    packed[3, 8:16] = 0x77               # 6.0
    scale = synth.uniform_ints(N * K // 16, 0x30, 0x50, 11, 2).astype(np.uint8).reshape(N, K // 16)
    div = np.array([37.0, 1000.0], np.float32)
    parts = [30, 40]
    gp, ge, gs = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), parts, mode, err_ssq=False)
    assert gs is None
    rp, re_, _ = orc.requant(packed, scale, div, parts, mode)
    assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp)
    wb = synth.bf16_weights(N, K, seed=12).copy()
    wb[5, 0] = 0x4480                    # 1024
    wb[5, 1:32] = 0xB400                 # -2^-23, far below the block's smallest grid step
    gp, ge, _ = lib.requant_bf16(to_dev_bf16(wb), mode, err_ssq=False)
    rp, re_, _ = orc.requant_bf16(wb, mode)
    assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp)
    assert np.all(host(gp)[5, :16] & 0x88 == 0)  # no sign on the zero indices
    w8, sc8 = synth.fp8_channel_weights(N, K, seed=13)
    gp, ge, _ = lib.requant_fp8_channel(to_dev(w8), to_dev(sc8), mode, err_ssq=False)
    rp, re_, _ = orc.requant_fp8_channel(w8, sc8, mode)
    assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp)


@pytest.mark.slow
def test_requant_full_gate_up(lib, orc):
    N, K = GATE_UP
    parts = list(synth.GATE_UP_PARTITIONS)
    packed, scale, div = _nvfp4_case(orc, N, K, parts, seed=0, gain2=0.25)
    for mode in ("ocp", "noclip", "mse"):
        gp, ge, gs = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), parts, mode)
        rp, re_, rs = orc.requant(packed, scale, div, parts, mode)
        assert np.array_equal(host(ge), re_), mode
        assert np.array_equal(host(gp), rp), mode
        _check_err_ssq(host(gs), rs)
        rel_g = orc.rel_rms(host(gs))
        assert abs(rel_g - orc.rel_rms(rs)) <= 1e-5 * orc.rel_rms(rs)


def _page_exponent_disagreements(packed, scale, div, parts, e_exact, mode):
    """How often the page's fp32 exponent formulas ("radiance_nvfp4.py", _block_exponent:
    floor(log2(amax)) - 2 for ocp, ceil(log2(amax / 6)) for noclip, torch.log2 in fp32) differ from
    the exact rule the library and the oracle implement, on the blocks with amax > 0.  The
    dequantized weights follow dequant_nvfp4 in fp32 on the GPU."""
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device="cuda")
    N = packed.shape[0]
    pk = to_dev(packed)
    codes = torch.stack([pk & 0x0F, pk >> 4], -1).reshape(N, -1).long()
    val = grid[codes & 7] * torch.where((codes & 8) != 0, -1.0, 1.0)
    sc = to_dev(scale).view(torch.float8_e4m3fn).float()
    rows = torch.repeat_interleave(torch.arange(len(parts), device="cuda"), torch.tensor(parts, device="cuda"))
    t = sc / to_dev(div)[rows][:, None]                       # fl(s / divisor)
    w = val * torch.repeat_interleave(t, 16, dim=1)           # fl(G * t)
    amax = w.abs().reshape(N, -1, 32).amax(-1)
    pos = amax > 0
    if mode == "ocp":
        page = torch.floor(torch.log2(amax)) - 2
    else:
        page = torch.ceil(torch.log2(amax / 6.0))
    exact = (to_dev(e_exact).float() - 127.0)
    return int(((page != exact) & pos).sum()), int(pos.sum())


@pytest.mark.slow
def test_requant_gate_up_relrms_report(lib, orc):
    """Config: the merged gate_up [34816, 5120], W ~ N(0, 0.02), two 17408-row partitions each
    NVFP4-quantized with its own divisor 6*448/amax, requantized by every rule: bit-exact codes and
    e8m0, and the per-layer relRMS from the GPU's error sums ("radiance_nvfp4.py",
    process_weights_after_loading) equal to the oracle's.  Prints the figures and the direct
    bf16 -> MXFP4 relRMS of the same weights (the pages' context: 0.158 requantized, 0.112 direct,
    on real checkpoint tensors) and the page-formula exponent diagnostic."""
    import json
    N, K = GATE_UP
    parts = list(synth.GATE_UP_PARTITIONS)
    w = synth.gaussian_weights(N, K, 0.02, 0)
    packed, scale, div = orc.nvfp4_quantize(w, parts)
    report = {"divisors": [float(d) for d in div]}
    for mode in ("ocp", "noclip", "mse"):
        gp, ge, gs = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), parts, mode)
        rp, re_, rs = orc.requant(packed, scale, div, parts, mode)
        assert np.array_equal(host(ge), re_), mode
        assert np.array_equal(host(gp), rp), mode
        g = host(gs)
        rel = orc.rel_rms(g)
        assert abs(rel - orc.rel_rms(rs)) <= 1e-5 * orc.rel_rms(rs)
        report[mode] = {"relrms": rel, "per_partition": [float(np.sqrt(e / s)) for e, s in g]}
        if mode != "mse":
            bad, total = _page_exponent_disagreements(packed, scale, div, parts, re_, mode)
            report[mode]["page_formula_disagreements"] = [bad, total]
    # mse picks the lower-error exponent per block, so it can only help
    assert report["mse"]["relrms"] <= report["noclip"]["relrms"]
    wb = synth.to_bf16_bits(w)
    _, _, gs = lib.requant_bf16(to_dev_bf16(wb), "mse")
    report["direct_bf16_mse_relrms"] = orc.rel_rms(host(gs))
    print("REQUANT_REPORT " + json.dumps(report))


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
@pytest.mark.parametrize("N,K", [(1, 32), (70, 384), (257, 1024)])
def test_requant_fp8_channel_bit_exact(lib, orc, mode, N, K):
    w8, s = synth.fp8_channel_weights(N, K, seed=N)
    gp, ge, gs = lib.requant_fp8_channel(to_dev(w8), to_dev(s), mode)
    rp, re_, rs = orc.requant_fp8_channel(w8, s, mode)
    assert np.array_equal(host(ge), re_)
    assert np.array_equal(host(gp), rp)
    _check_err_ssq(host(gs), rs)


@pytest.mark.parametrize("mode", ["ocp", "noclip", "mse"])
@pytest.mark.parametrize("N,K", [(1, 32), (70, 384), (257, 1024)])
def test_requant_bf16_bit_exact(lib, orc, mode, N, K):
    wb = synth.bf16_weights(N, K, seed=N)
    gp, ge, gs = lib.requant_bf16(to_dev_bf16(wb), mode)
    rp, re_, rs = orc.requant_bf16(wb, mode)
    assert np.array_equal(host(ge), re_)
    assert np.array_equal(host(gp), rp)
    _check_err_ssq(host(gs), rs)


def test_requant_other_sources_degenerate(lib, orc):
    # zero rows, the largest and smallest e4m3 magnitudes, a zero channel scale, bf16 zeros,
    # signed zeros and values whose exponent clamps at the e8m0 range
    w8, s = synth.fp8_channel_weights(6, 64, seed=7)
    w8[0] = 0
    w8[1, :32] = 0x7E                    # 448
    w8[1, 32:] = 0x01                    # 2^-9
    w8[2] = 0x80                         # -0
    s[3] = 0.0
    s[4] = np.float32(2.0 ** -120)
    wb = synth.bf16_weights(6, 64, seed=8)
    wb[0] = 0
    wb[1] = 0x8000                       # -0
    wb[2, :32] = 0x7F7F                  # largest finite bf16
    wb[3, :32] = 0x0001                  # smallest subnormal bf16
    for mode in ("ocp", "noclip", "mse"):
        gp, ge, _ = lib.requant_fp8_channel(to_dev(w8), to_dev(s), mode)
        rp, re_, _ = orc.requant_fp8_channel(w8, s, mode)
        assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp), mode
        gp, ge, _ = lib.requant_bf16(to_dev_bf16(wb), mode)
        rp, re_, _ = orc.requant_bf16(wb, mode)
        assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp), mode


@pytest.mark.slow
def test_requant_other_sources_full_gate_up(lib, orc):
    N, K = GATE_UP
    w8, s = synth.fp8_channel_weights(N, K, seed=1)
    gp, ge, gs = lib.requant_fp8_channel(to_dev(w8), to_dev(s), "mse")
    rp, re_, rs = orc.requant_fp8_channel(w8, s, "mse")
    assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp)
    _check_err_ssq(host(gs), rs)
    del w8, gp, ge
    wb = synth.bf16_weights(N, K, seed=2)
    gp, ge, gs = lib.requant_bf16(to_dev_bf16(wb), "mse")
    rp, re_, rs = orc.requant_bf16(wb, "mse")
    assert np.array_equal(host(ge), re_) and np.array_equal(host(gp), rp)
    _check_err_ssq(host(gs), rs)


def test_requant_other_sources_reject(lib):
    w = torch.zeros((4, 48), dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.requant_fp8_channel(w, torch.ones(4, dtype=torch.float32, device="cuda"), "mse")  # K % 32
    wb = torch.zeros((4, 40), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.requant_bf16(wb, "ocp")


def test_requant_rejects(lib):
    p = torch.zeros((4, 16), dtype=torch.uint8, device="cuda")
    s = torch.zeros((4, 2), dtype=torch.uint8, device="cuda")
    d = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.requant(p, s, d, [2, 1], "mse")  # rows do not sum to N


# ---------------------------------------------------------------------------- GEMMs

POLICIES = [1, 2]  # CUDA-core kernels, tensor-core kernels where the shape allows


@pytest.fixture(params=POLICIES, ids=["simt", "tc"])
def policy(request, lib):
    lib.set_gemm_policy(request.param)
    yield request.param
    lib.set_gemm_policy(0)


def _mx_gemm(lib, orc, x, w, e, pairs=None):
    xq, xs = lib.act_quant(to_dev_bf16(x))
    out = lib.mxfp4_linear(xq, xs, to_dev(w), to_dev(e))
    lib.check_device_status()
    hq, hs = host(xq), host(xs)
    got = bf16_to_f64(out)
    if pairs is None:
        return got, orc.mxfp4_linear(hq, hs, w, e)
    im, inn = pairs
    return got[im, inn], orc.mxfp4_linear_pairs(hq, hs, w, e, im, inn)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (4, 256, 512), (7, 384, 640), (33, 200, 256),
                                   (64, 1024, 1024), (65, 256, 384), (130, 520, 1152),
                                   (300, 384, 256), (3, 96, 96),
                                   # K a multiple of 512: the tensor-core path (stream-K splits,
                                   # ragged token and weight-row tails, every token tile width)
                                   (1, 128, 512), (5, 384, 1024), (17, 200, 512), (33, 520, 1536),
                                   (64, 1000, 2048), (65, 256, 512), (130, 520, 1024),
                                   (257, 384, 512), (300, 640, 1536), (16, 4096, 512)])
def test_mxfp4_linear_small(lib, orc, policy, M, N, K):
    x, w, e = synth.prefill_case(M, N, K, seed=M * 7 + N)
    got, ref = _mx_gemm(lib, orc, x, w, e)
    gemm_check(got, ref, f"mxfp4 M={M} N={N} K={K} policy={policy}")


def _sample_pairs(M, N, n_cols=192, seed=0):
    cols = np.unique(np.concatenate([[0, N - 1, 127, 128, N // 2],
                                     synth.uniform_ints(n_cols, 0, N - 1, seed, 77)]))
    im = np.repeat(np.arange(M), cols.size)
    inn = np.tile(cols, M)
    return im, inn


@pytest.mark.parametrize("shape", [GATE_UP, DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_mxfp4_decode_full_sampled(lib, orc, shape, M):
    N, K = shape
    x, w, e = synth.decode_case(M, N, K, seed=0)
    got, ref = _mx_gemm(lib, orc, x, w, e, pairs=_sample_pairs(M, N))
    gemm_check(got, ref, f"decode M={M} N={N} K={K}")


@pytest.mark.slow
@pytest.mark.parametrize("shape", [GATE_UP, DOWN, QKV], ids=["gate_up", "down", "qkv"])
@pytest.mark.parametrize("M", [512, 4096])
def test_mxfp4_prefill_full_sampled(lib, orc, shape, M):
    N, K = shape
    x, w, e = synth.prefill_case(M, N, K, seed=0)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], synth.uniform_ints(12, 0, M - 1, 1, 5)]))
    cols = np.unique(np.concatenate([[0, 255, 256, N - 1], synth.uniform_ints(48, 0, N - 1, 1, 6)]))
    im = np.repeat(rows, cols.size)
    inn = np.tile(cols, rows.size)
    got, ref = _mx_gemm(lib, orc, x, w, e, pairs=(im, inn))
    gemm_check(got, ref, f"prefill M={M} N={N} K={K}")


def test_mxfp4_tiny_config_end_to_end(lib, orc):
    """M=4, N=256, K=512: W ~ N(0, 0.02) -> NVFP4 -> requant (mse) -> W4A8 GEMM."""
    M, N, K = 4, 256, 512
    x = synth.activations(M, K, seed=0, outliers=True)
    w32 = synth.gaussian_weights(N, K, 0.02, seed=0)
    packed, scale, div = orc.nvfp4_quantize(w32, [N])
    gp, ge, _ = lib.requant(to_dev(packed), to_dev(scale), to_dev(div), [N], "mse")
    rp, re_, _ = orc.requant(packed, scale, div, [N], "mse")
    assert np.array_equal(host(gp), rp) and np.array_equal(host(ge), re_)
    xq, xs = lib.act_quant(to_dev_bf16(x))
    out = lib.mxfp4_linear(xq, xs, gp, ge)
    gemm_check(bf16_to_f64(out), orc.mxfp4_linear(host(xq), host(xs), rp, re_), "tiny")


def test_mxfp4_rejects(lib):
    xq = torch.zeros((2, 48), dtype=torch.uint8, device="cuda")
    xs = torch.ones(2, dtype=torch.float32, device="cuda")
    w = torch.zeros((8, 24), dtype=torch.uint8, device="cuda")
    e = torch.zeros((8, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises((lib.W4A8Error, ValueError)):
        lib.mxfp4_linear(xq, xs, w, e)  # K = 48 is not a multiple of 32


# ------------------------------------------------------- fused act quant + GEMM (one call)

@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (7, 384, 640), (1, 128, 512), (5, 384, 1024),
                                   (33, 520, 1536), (64, 1000, 2048), (130, 520, 1024)])
def test_linear_fused_matches_two_calls(lib, orc, policy, M, N, K):
    """w4a8_mxfp4_linear_bf16 is bit-identical to act quant + w4a8_mxfp4_linear, and within the
    GEMM bound of the oracle."""
    x, w, e = synth.prefill_case(M, N, K, seed=M * 11 + N)
    xd, wd, ed = to_dev_bf16(x), to_dev(w), to_dev(e)
    fused = lib.linear(xd, wd, ed)
    xq, xs = lib.act_quant(xd)
    two = lib.mxfp4_linear(xq, xs, wd, ed)
    lib.check_device_status()
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
    gemm_check(bf16_to_f64(fused), orc.mxfp4_linear(host(xq), host(xs), w, e), f"fused M={M} N={N} K={K}")


# The one-launch form (w4a8_mxfp4_linear_bf16_single): every CTA takes the rows' amax from L2 and
# writes its fills' e4m3 tiles into shared memory itself.  It must give the bytes of the two-kernel
# chain, for 1 or 2 tokens and up to 96 KB of bf16 activations; past that it refuses the shape.
@pytest.mark.parametrize("M,N,K", [(1, 520, 512), (2, 256, 1024), (1, 1000, 2048), (2, 4096, 5120),
                                   (1, 384, 5120), (2, 256, 10240), (1, 5120, 17408),
                                   (2, 34816, 5120), (1, 160, 49152)])
def test_linear_fused_quant_in_gemm(lib, orc, M, N, K):
    x, w, e = synth.decode_case(M, N, K, seed=M * 5 + N)
    x = x.copy()
    x[0, :7] = 0x8000                      # -0 values
    if M > 1:
        x[1, 3::5] = 0                     # zeros inside a row
    xd, wd, ed = to_dev_bf16(x), to_dev(w), to_dev(e)
    one = lib.linear(xd, wd, ed, single_kernel=True)
    two = lib.linear(xd, wd, ed)
    lib.check_device_status()
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
    hq, hs = orc.act_quant(x)
    im, inn = _sample_pairs(M, N, seed=M)
    gemm_check(bf16_to_f64(one)[im, inn], orc.mxfp4_linear_pairs(hq, hs, w, e, im, inn),
               f"one-launch linear M={M} N={N} K={K}")


def test_linear_single_all_zero_row(lib):
    """An all-zero token gets scale 1 and zero codes, so its output row is exactly zero."""
    x, w, e = synth.decode_case(2, 512, 2048, seed=3)
    x = x.copy()
    x[1, :] = 0
    one = lib.linear(to_dev_bf16(x), to_dev(w), to_dev(e), single_kernel=True)
    lib.check_device_status()
    assert np.all(bf16_to_f64(one)[1] == 0.0)


@pytest.mark.parametrize("M,N,K", [(3, 256, 1024), (1, 256, 1000 * 32), (1, 256, 49152 + 512), (1, 256, 992)])
def test_linear_single_rejects_shapes(lib, M, N, K):
    """More than 2 tokens, more than 96 KB of activations, or K not a multiple of 512: refused."""
    xd = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    ed = torch.full((N, K // 32), 127, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.W4A8Error) as ei:
        lib.linear(xd, wd, ed, single_kernel=True)
    assert ei.value.status == 2


@pytest.mark.parametrize("shape", [GATE_UP, DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 64])
def test_linear_fused_decode_full_sampled(lib, orc, shape, M):
    N, K = shape
    x, w, e = synth.decode_case(M, N, K, seed=3)
    out = lib.linear(to_dev_bf16(x), to_dev(w), to_dev(e))
    lib.check_device_status()
    hq, hs = orc.act_quant(x)
    im, inn = _sample_pairs(M, N, seed=4)
    gemm_check(bf16_to_f64(out)[im, inn], orc.mxfp4_linear_pairs(hq, hs, w, e, im, inn),
               f"fused decode M={M} N={N} K={K}")


def test_linear_fused_chained_layers(lib, orc):
    """Layer 2 quantizes layer 1's output: the activation quant must wait for the GEMM before
    it on the stream (both launched with programmatic dependent launch).  One workspace per
    layer, reused over repeated passes."""
    M, K1, N1, N2 = 8, 512, 1536, 1024
    x, w1, e1 = synth.prefill_case(M, N1, K1, seed=21)
    _, w2, e2 = synth.prefill_case(M, N2, N1, seed=22)
    xd = to_dev_bf16(x)
    w1d, e1d, w2d, e2d = to_dev(w1), to_dev(e1), to_dev(w2), to_dev(e2)
    ws1 = lib.make_linear_workspace(M, N1, K1, "cuda")
    ws2 = lib.make_linear_workspace(M, N2, N1, "cuda")
    outs = []
    for _ in range(3):
        h = lib.linear(xd, w1d, e1d, workspace=ws1)
        outs.append(lib.linear(h, w2d, e2d, workspace=ws2))
    lib.check_device_status()
    h_ref = lib.linear(xd, w1d, e1d)
    torch.cuda.synchronize()
    hq, hs = lib.act_quant(h_ref)
    ref2 = lib.mxfp4_linear(hq, hs, w2d, e2d)
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref2.view(torch.int16))
    gemm_check(bf16_to_f64(ref2), orc.mxfp4_linear(host(hq), host(hs), w2, e2), "layer 2")


def test_workspace_shared_across_shapes(lib):
    """One workspace buffer, sized for the largest need, serves a sequence of shapes and entry
    points: the arrival counters sit at a fixed offset that no partial tile ever reaches, so a
    wide decode tile's partials cannot leave garbage where a narrower one counts.  Every output
    must equal the same call with a fresh workspace, bit for bit."""
    N, K = 1024, 2048  # 8 weight tiles of 4 units: every tile split over 4 CTAs
    cases = [64, 1, 300, 8, 1, 32, 1]
    need = max(max(lib.workspace_bytes(M, N, K), lib.int4_workspace_bytes(M, N, K),
                   lib.linear_workspace_bytes(M, N, K)) for M in cases)
    ws = lib.make_workspace(need + 256, "cuda")
    ws = ws[(-ws.data_ptr()) % 256:][:need]
    _, w, e = synth.prefill_case(1, N, K, seed=31)
    wd, ed = to_dev(w), to_dev(e)
    _, qw, s16, _ = synth.int4_case(1, N, K, seed=32)
    qwd, s16d = to_dev(qw), to_dev_fp16(s16)
    for M in cases:
        xd = to_dev_bf16(synth.activations(M, K, seed=M))
        xq, xs = lib.act_quant(xd)
        got = [lib.mxfp4_linear(xq, xs, wd, ed, workspace=ws), lib.int4g128_linear(xq, xs, qwd, s16d, workspace=ws),
               lib.linear(xd, wd, ed, workspace=ws)]
        ref = [lib.mxfp4_linear(xq, xs, wd, ed), lib.int4g128_linear(xq, xs, qwd, s16d), lib.linear(xd, wd, ed)]
        lib.check_device_status()
        for g, r, what in zip(got, ref, ("mxfp4", "int4", "bf16 linear")):
            assert torch.equal(g.view(torch.int16), r.view(torch.int16)), f"{what} M={M}"


def test_linear_fused_rejects(lib):
    M, N, K = 2, 128, 512
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    e = torch.zeros((N, K // 32), dtype=torch.uint8, device="cuda")
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.linear(x, w, e, workspace=small)
    ws = lib.make_linear_workspace(M, N, K, "cuda")
    big = torch.zeros(ws.numel() + 512, dtype=torch.uint8, device="cuda")
    off = (-big.data_ptr()) % 256 + 16  # 16-byte but not 256-byte aligned
    with pytest.raises(lib.W4A8Error):
        lib.linear(x, w, e, workspace=big[off:off + ws.numel()])


def _i4_gemm(lib, orc, x, qw, s16, qz, pairs=None):
    xq, xs = lib.act_quant(to_dev_bf16(x))
    out = lib.int4g128_linear(xq, xs, to_dev(qw), to_dev_fp16(s16), qzeros=to_dev(qz))
    lib.check_device_status()
    hq, hs = host(xq), host(xs)
    got = bf16_to_f64(out)
    if pairs is None:
        return got, orc.int4g128_linear(hq, hs, qw, s16)
    im, inn = pairs
    return got[im, inn], orc.int4g128_linear_pairs(hq, hs, qw, s16, im, inn)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (8, 256, 512), (33, 136, 384), (64, 512, 1024),
                                   (100, 264, 256), (200, 128, 640),
                                   # K a multiple of 512: the tensor-core path (stream-K splits,
                                   # ragged token and column tails, every token tile width)
                                   (1, 132, 512), (5, 384, 1024), (17, 200, 1536), (33, 520, 2048),
                                   (64, 1000, 512), (65, 260, 1024), (130, 384, 512), (300, 640, 1536)])
def test_int4_linear_small(lib, orc, policy, M, N, K):
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=M + N)
    got, ref = _i4_gemm(lib, orc, x, qw, s16, qz)
    gemm_check(got, ref, f"int4 M={M} N={N} K={K} policy={policy}")


@pytest.mark.parametrize("shape", [GATE_UP, DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 8, 64, 4096])
def test_int4_full_sampled(lib, orc, shape, M):
    N, K = shape
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=0)
    if M > 64:
        rows = np.unique(np.concatenate([[0, 127, 128, M - 1], synth.uniform_ints(6, 0, M - 1, 2, 5)]))
        cols = np.unique(np.concatenate([[0, 255, 256, N - 1], synth.uniform_ints(32, 0, N - 1, 2, 6)]))
        pairs = (np.repeat(rows, cols.size), np.tile(cols, rows.size))
    else:
        pairs = _sample_pairs(M, N, 96)
    got, ref = _i4_gemm(lib, orc, x, qw, s16, qz, pairs=pairs)
    gemm_check(got, ref, f"int4 M={M} N={N} K={K}")


# M > 128 without zero points takes the 256-token prefill tiling (signed operand codes, no
# zero-point MMAs): several token tiles with a ragged last one, ragged column tiles, N % 8 != 0
# (plain output stores), split tiles only (small shapes) and whole tiles beside stream-K splits
# (192 tiles on the GPU's SMs).
PREFILL_I4 = [(129, 132, 512), (256, 256, 512), (300, 1004, 1024), (513, 392, 2048), (600, 640, 1536),
              (512, 12288, 512)]


def _prefill_pairs(M, N, seed):
    edges = [r for r in (0, 95, 96, 127, 128, 191, 192, 255, 256, 383, 384) if r < M] + [M - 1]
    rows = np.unique(np.concatenate([edges, synth.uniform_ints(24, 0, M - 1, seed, 5)]))
    cols = np.unique(np.concatenate([[0, 127, 128, N - 1], synth.uniform_ints(48, 0, N - 1, seed, 6)]))
    return np.repeat(rows, cols.size), np.tile(cols, rows.size)


@pytest.mark.parametrize("M,N,K", PREFILL_I4)
def test_int4_prefill_tiling(lib, orc, M, N, K):
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=M + 7)
    pairs = _prefill_pairs(M, N, 7) if M * N > 1 << 20 else None
    got, ref = _i4_gemm(lib, orc, x, qw, s16, qz, pairs=pairs)
    gemm_check(got, ref, f"int4 prefill M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(129, 144, 512), (256, 256, 512), (300, 1008, 1024), (513, 400, 2048),
                                   (512, 12288, 512)])
def test_int5_prefill_tiling(lib, orc, M, N, K):
    x = synth.activations(M, K, seed=M + 8)
    qw, qh, s16 = synth.int5_weights(N, K, seed=M + 8)
    pairs = _prefill_pairs(M, N, 8) if M * N > 1 << 20 else None
    got, ref = _i5_gemm(lib, orc, x, qw, qh, s16, pairs=pairs)
    gemm_check(got, ref, f"int5 prefill M={M} N={N} K={K}")


def test_int4_prefill_extreme_codes(lib, orc):
    # every code 0 (value -8) and every code 15 (value 7), and an all-zero activation row: the
    # signed operand bytes at both ends and a row whose output must be exactly zero
    M, N, K = 260, 256, 1024
    x, _, s16, qz = synth.int4_case(M, N, K, seed=21)
    x[3, :] = 0
    for word in (0x00000000, 0xFFFFFFFF, 0x0F0F0F0F):
        qw = np.full((K // 8, N), word, np.uint32).view(np.int32)
        got, ref = _i4_gemm(lib, orc, x, qw, s16, qz)
        gemm_check(got, ref, f"int4 prefill codes {word:#x}")
        assert np.all(got[3] == 0.0)


@pytest.mark.parametrize("M", [1, 16])
def test_int4_decode_extreme_codes(lib, orc, M):
    # decode tiles (1 and 16 tokens): every code 0 (value -8, the output is the zero point's
    # term alone), every code 15 (value 7), alternating 15 / 0, and an all-zero activation row
    # whose output must be exactly zero
    N, K = 384, 1536
    x, _, s16, qz = synth.int4_case(M, N, K, seed=22 + M)
    live = M - 1 if M > 1 else M  # rows checked against the oracle; the last one is zero if M > 1
    if M > 1:
        x[M - 1, :] = 0
    for word in (0x00000000, 0xFFFFFFFF, 0x0F0F0F0F):
        qw = np.full((K // 8, N), word, np.uint32).view(np.int32)
        got, ref = _i4_gemm(lib, orc, x, qw, s16, qz)
        gemm_check(got[:live], ref[:live], f"int4 decode M={M} codes {word:#x}")
        if M > 1:
            assert np.all(got[M - 1] == 0.0)


def _i4_asym_gemm(lib, orc, x, qw, s16, qz, pairs=None):
    xq, xs = lib.act_quant(to_dev_bf16(x))
    out = lib.int4g128_asym_linear(xq, xs, to_dev(qw), to_dev_fp16(s16), to_dev(qz))
    lib.check_device_status()
    hq, hs = host(xq), host(xs)
    got = bf16_to_f64(out)
    if pairs is None:
        return got, orc.int4g128_asym_linear(hq, hs, qw, s16, qz)
    im, inn = pairs
    return got[im, inn], orc.int4g128_asym_linear_pairs(hq, hs, qw, s16, qz, im, inn)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (8, 260, 512), (33, 136, 384), (100, 264, 256),
                                   (1, 132, 512), (5, 384, 1024), (17, 200, 1536), (33, 520, 2048),
                                   (64, 1000, 512), (65, 260, 1024), (130, 384, 512)])
def test_int4_asym_linear_small(lib, orc, policy, M, N, K):
    x, qw, s16, _ = synth.int4_case(M, N, K, seed=M + N + 1)
    qz = synth.int4_asym_zeros(N, K, seed=M + N + 1)
    got, ref = _i4_asym_gemm(lib, orc, x, qw, s16, qz)
    gemm_check(got, ref, f"int4 asym M={M} N={N} K={K} policy={policy}")


@pytest.mark.parametrize("M", [1, 64])
def test_int4_asym_full_sampled(lib, orc, M):
    N, K = GATE_UP
    x, qw, s16, _ = synth.int4_case(M, N, K, seed=3)
    qz = synth.int4_asym_zeros(N, K, seed=3)
    got, ref = _i4_asym_gemm(lib, orc, x, qw, s16, qz, pairs=_sample_pairs(M, N, 96))
    gemm_check(got, ref, f"int4 asym M={M} N={N} K={K}")


def test_int4_asym_symmetric_zeros_match(lib, orc):
    # qzeros 0x77777777 through the asymmetric entry reproduces the symmetric definition
    M, N, K = 4, 256, 1024
    x, qw, s16, qz = synth.int4_case(M, N, K, seed=9)
    got, ref = _i4_asym_gemm(lib, orc, x, qw, s16, qz[:, :N // 8])
    gemm_check(got, orc.int4g128_linear(*[host(t) for t in lib.act_quant(to_dev_bf16(x))], qw, s16),
               "int4 asym with symmetric zeros")


def test_int4_rejects_asymmetric(lib):
    xq = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    xs = torch.ones(1, dtype=torch.float32, device="cuda")
    qw = torch.zeros((16, 8), dtype=torch.int32, device="cuda")
    s = torch.ones((1, 8), dtype=torch.float16, device="cuda")
    qz = torch.full((1, 1), 0x77777776, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        lib.int4g128_linear(xq, xs, qw, s, qzeros=qz)


# --- int5 g128 ("vllm-radiance (MXFP4)", section "int5 (W5A8)")

def _i5_gemm(lib, orc, x, qw, qh, s16, z=None, pairs=None):
    xq, xs = lib.act_quant(to_dev_bf16(x))
    out = lib.int5g128_linear(xq, xs, to_dev(qw), to_dev(qh), to_dev_fp16(s16),
                              None if z is None else to_dev(z))
    lib.check_device_status()
    hq, hs = host(xq), host(xs)
    got = bf16_to_f64(out)
    if pairs is None:
        return got, orc.int5g128_linear(hq, hs, qw, qh, s16, z)
    im, inn = pairs
    return got[im, inn], orc.int5g128_linear_pairs(hq, hs, qw, qh, s16, z, im, inn)


@pytest.mark.parametrize("asym", [False, True], ids=["sym", "asym"])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (8, 256, 512), (33, 144, 384), (100, 264, 256),
                                   # N % 16 == 0 and K % 512 == 0: the tensor-core path (stream-K
                                   # splits, ragged token and column tails, every token tile width)
                                   (1, 144, 512), (5, 384, 1024), (17, 208, 1536), (33, 528, 2048),
                                   (64, 1008, 512), (65, 272, 1024), (130, 384, 512), (300, 640, 1536),
                                   # N % 16 != 0: CUDA-core kernel under every policy
                                   (3, 200, 1024)])
def test_int5_linear_small(lib, orc, policy, asym, M, N, K):
    x = synth.activations(M, K, seed=M + N + 2)
    qw, qh, s16 = synth.int5_weights(N, K, seed=M + N + 2)
    z = synth.int5_zeros(N, K, seed=M + N + 2) if asym else None
    got, ref = _i5_gemm(lib, orc, x, qw, qh, s16, z)
    gemm_check(got, ref, f"int5 asym={asym} M={M} N={N} K={K} policy={policy}")


@pytest.mark.parametrize("asym", [False, True], ids=["sym", "asym"])
@pytest.mark.parametrize("shape", [GATE_UP, DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 64, 4096])
def test_int5_full_sampled(lib, orc, shape, M, asym):
    N, K = shape
    x = synth.activations(M, K, seed=4)
    qw, qh, s16 = synth.int5_weights(N, K, seed=4)
    z = synth.int5_zeros(N, K, seed=4) if asym else None
    if M > 64:
        rows = np.unique(np.concatenate([[0, 63, 64, M - 1], synth.uniform_ints(6, 0, M - 1, 4, 5)]))
        cols = np.unique(np.concatenate([[0, 127, 128, N - 1], synth.uniform_ints(32, 0, N - 1, 4, 6)]))
        pairs = (np.repeat(rows, cols.size), np.tile(cols, rows.size))
    else:
        pairs = _sample_pairs(M, N, 96)
    got, ref = _i5_gemm(lib, orc, x, qw, qh, s16, z, pairs=pairs)
    gemm_check(got, ref, f"int5 asym={asym} M={M} N={N} K={K}")


def test_int5_degenerate_codes(lib, orc):
    # every fifth bit set with zero point 16 (values = nibbles), none set (nibble - 16), and
    # zero points at both ends of 0..31
    M, N, K = 4, 256, 1024
    x = synth.activations(M, K, seed=13)
    qw, _, s16 = synth.int5_weights(N, K, seed=13)
    for qh in (np.full((K // 8, N), 0xFF, np.uint8), np.zeros((K // 8, N), np.uint8)):
        got, ref = _i5_gemm(lib, orc, x, qw, qh, s16)
        gemm_check(got, ref, "int5 constant fifth bits")
    _, qh, _ = synth.int5_weights(N, K, seed=14)
    z = np.zeros((K // 128, N), np.uint8)
    z[:, 1::2] = 31
    got, ref = _i5_gemm(lib, orc, x, qw, qh, s16, z)
    gemm_check(got, ref, "int5 zero points 0 and 31")


def test_int5_rejects(lib):
    xq = torch.zeros((1, 128), dtype=torch.uint8, device="cuda")
    xs = torch.ones(1, dtype=torch.float32, device="cuda")
    qw = torch.zeros((16, 16), dtype=torch.int32, device="cuda")
    qh = torch.zeros((16, 16), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        lib.int5g128_linear(xq, xs, qw, qh[:8], s)
    with pytest.raises(ValueError):
        lib.int5g128_linear(xq, xs, qw, qh, s, torch.zeros((2, 16), dtype=torch.uint8, device="cuda"))
    out = torch.empty((1, 16), dtype=torch.bfloat16, device="cuda")
    st = lib.load().w4a8_int5g128_linear(xq.data_ptr(), xs.data_ptr(), qw.data_ptr(), None, s.data_ptr(), None,
                                         out.data_ptr(), 1, 16, 128, None, 0, None)
    assert st == 1  # W4A8_ERR_INVALID_ARG: no fifth-bit plane


# --- W4A4 ("vllm-radiance (MXFP4)", section "Native MXFP4": MXFP4 activations)

def _a4_gemm(lib, orc, x, w, e, pairs=None):
    xa, xe = lib.act_quant_mxfp4(to_dev_bf16(x))
    out = lib.mxfp4_a4_linear(xa, xe, to_dev(w), to_dev(e))
    lib.check_device_status()
    ha, he = host(xa), host(xe)
    oa, oe = orc.act_quant_mxfp4(x)
    assert np.array_equal(ha, oa) and np.array_equal(he, oe), "W4A4 activation codes or scales differ"
    got = bf16_to_f64(out)
    if pairs is None:
        return got, orc.mxfp4_a4_linear(ha, he, w, e)
    im, inn = pairs
    return got[im, inn], orc.mxfp4_a4_linear_pairs(ha, he, w, e, im, inn)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (9, 5120), (64, 17408), (130, 1024)])
def test_w4a4_act_quant_bit_exact(lib, orc, M, K):
    x = synth.activations(M, K, seed=M + K, outliers=True)
    x[0, :min(K, 64)] = 0  # an all-zero block (and for K <= 64 an all-zero row)
    xa, xe = lib.act_quant_mxfp4(to_dev_bf16(x))
    torch.cuda.synchronize()
    oa, oe = orc.act_quant_mxfp4(x)
    assert np.array_equal(host(xa), oa) and np.array_equal(host(xe), oe)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (4, 256, 512), (33, 200, 256), (65, 256, 384), (3, 96, 96),
                                   # K a multiple of 512: the tensor-core path (stream-K splits,
                                   # ragged token and weight-row tails, every token tile width)
                                   (1, 128, 512), (5, 384, 1024), (17, 200, 512), (33, 520, 1536),
                                   (64, 1000, 2048), (65, 256, 512), (130, 520, 1024),
                                   (257, 384, 512), (300, 640, 1536), (16, 4096, 512)])
def test_w4a4_linear_small(lib, orc, policy, M, N, K):
    # prefill recipe: per-token magnitudes spread by a log-normal factor, so every token of a
    # tile has its own block exponents
    x, w, e = synth.prefill_case(M, N, K, seed=M * 5 + N)
    got, ref = _a4_gemm(lib, orc, x, w, e)
    gemm_check(got, ref, f"w4a4 M={M} N={N} K={K} policy={policy}")


@pytest.mark.parametrize("shape", [GATE_UP, DOWN], ids=["gate_up", "down"])
@pytest.mark.parametrize("M", [1, 8, 32, 64, 4096])
def test_w4a4_full_sampled(lib, orc, shape, M):
    N, K = shape
    x, w, e = synth.prefill_case(M, N, K, seed=1)
    if M > 64:
        rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], synth.uniform_ints(8, 0, M - 1, 1, 5)]))
        cols = np.unique(np.concatenate([[0, 127, 128, N - 1], synth.uniform_ints(32, 0, N - 1, 1, 6)]))
        pairs = (np.repeat(rows, cols.size), np.tile(cols, rows.size))
    else:
        pairs = _sample_pairs(M, N, 96)
    got, ref = _a4_gemm(lib, orc, x, w, e, pairs=pairs)
    gemm_check(got, ref, f"w4a4 M={M} N={N} K={K}")


def test_w4a4_less_accurate_than_w4a8(lib, orc):
    # the pages' numerics claim: fp8 activations are more accurate than MXFP4 ones.  Both paths
    # against the exact product of the bf16 activations and the dequantized weights.
    M, N, K = 16, 512, 2048
    x = synth.activations(M, K, seed=31)
    _, w, e = synth.decode_case(1, N, K, seed=31)
    exact = synth.bf16_bits_to_float(x).astype(np.float64) @ orc.dequant_mxfp4(w, e).T
    xd = to_dev_bf16(x)
    xq, xs = lib.act_quant(xd)
    o8 = bf16_to_f64(lib.mxfp4_linear(xq, xs, to_dev(w), to_dev(e)))
    xa, xe = lib.act_quant_mxfp4(xd)
    o4 = bf16_to_f64(lib.mxfp4_a4_linear(xa, xe, to_dev(w), to_dev(e)))
    rel = lambda o: np.linalg.norm(o - exact) / np.linalg.norm(exact)
    r8, r4 = rel(o8), rel(o4)
    assert r8 < 0.05 and r4 < 0.25 and r4 > 2.0 * r8, (r8, r4)


def test_w4a4_rejects(lib):
    xa = torch.zeros((1, 64), dtype=torch.uint8, device="cuda")
    xe = torch.zeros((1, 4), dtype=torch.uint8, device="cuda")
    w = torch.zeros((16, 64), dtype=torch.uint8, device="cuda")
    we = torch.zeros((16, 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        lib.mxfp4_a4_linear(xa, xe[:, :2], w, we)
    out = torch.empty((1, 16), dtype=torch.bfloat16, device="cuda")
    st = lib.load().w4a4_mxfp4_linear(xa.data_ptr(), xe.data_ptr(), w.data_ptr(), we.data_ptr(), out.data_ptr(),
                                      1, 16, 120, None, 0, None)
    assert st == 2  # W4A8_ERR_UNSUPPORTED_SHAPE: K % 32


@pytest.mark.parametrize("a4", [False, True], ids=["w4a8", "w4a4"])
def test_mxfp4_prefill_224_token_tiles(lib, orc, a4):
    # M = 3100, K = 1024: fourteen 224-token tiles per weight tile (the last one 188 tokens) --
    # the two-accumulator tiling for large M and shorter K, with a ragged token tail
    M, N, K = 3100, 1152, 1024
    x, w, e = synth.prefill_case(M, N, K, seed=78)
    rows = np.array([0, 1, 223, 224, 447, 448, 2911, 2912, 3098, 3099])
    cols = np.unique(np.concatenate([[0, 127, 128, N - 1], synth.uniform_ints(40, 0, N - 1, 78, 6)]))
    pairs = (np.repeat(rows, cols.size), np.tile(cols, rows.size))
    got, ref = (_a4_gemm if a4 else _mx_gemm)(lib, orc, x, w, e, pairs=pairs)
    gemm_check(got, ref, f"224-token tiles a4={a4}")


@pytest.mark.parametrize("a4", [False, True], ids=["w4a8", "w4a4"])
def test_mxfp4_prefill_192_token_tiles(lib, orc, a4):
    # M = 1000, 127 weight tiles, K = 512: six 192-token tiles per weight tile (the last one 40
    # tokens), five per CTA -- the two-accumulator prefill tiling with a ragged token tail
    M, N, K = 1000, 16256, 512
    x, w, e = synth.prefill_case(M, N, K, seed=77)
    rows = np.array([0, 1, 191, 192, 383, 384, 959, 960, 998, 999])
    cols = np.unique(np.concatenate([[0, 127, 128, N - 1], synth.uniform_ints(40, 0, N - 1, 77, 6)]))
    pairs = (np.repeat(rows, cols.size), np.tile(cols, rows.size))
    got, ref = (_a4_gemm if a4 else _mx_gemm)(lib, orc, x, w, e, pairs=pairs)
    gemm_check(got, ref, f"192-token tiles a4={a4}")
