"""Pins for the oracle's number formats, each against something other than the oracle.

* e4m3 decode: the format's landmark values and the library's float8_e4m3fn dtype.
* e4m3 encode: a brute-force nearest-of-grid search with ties to the even code over dense
  sweeps of fp32 bit patterns, all grid midpoints and their neighbours, and
  decode(encode(v)) == v on every finite code.
* e2m1_index ("radiance_nvfp4.py", e2m1_index docstring): the grid itself, the tie table
  implied by "ties to the EVEN code" (tests/golden/e2m1_grid.json), and an argmin search.
* fp16 decode: numpy's float16 over all 65536 patterns.
"""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _grid_e4m3():
    """All finite non-negative e4m3 values, enumerated through the library's fp8 dtype."""
    codes = torch.arange(0, 127, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes.numpy(), vals


def brute_e4m3(y: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 magnitude by search over the sorted grid; ties to the even code;
    saturating at 448; sign bit copied from the input."""
    codes, vals = _grid_e4m3()
    a = np.minimum(np.abs(y.astype(np.float64)), 448.0)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    c = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    c = np.where(a == vals[hi], codes[hi], c).astype(np.uint8)
    return c | (np.signbit(y).astype(np.uint8) << 7)


def test_e4m3_decode_matches_library_dtype(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode_many(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_landmarks(orc):
    assert orc.e4m3_decode(0x00) == 0.0
    assert np.signbit(orc.e4m3_decode(0x80))
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x3F) == 1.875
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0xFE) == -448.0
    assert np.isnan(orc.e4m3_decode(0x7F)) and np.isnan(orc.e4m3_decode(0xFF))


def test_e4m3_encode_roundtrip_all_codes(orc):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c, hex(c)


def test_e4m3_encode_bruteforce_sweep(orc):
    pieces = []
    for lo_exp, hi_exp in [(-11, -5), (6, 9)]:
        lo = np.float32(2.0 ** lo_exp).view(np.uint32)
        hi = np.float32(2.0 ** hi_exp).view(np.uint32)
        pieces.append(np.arange(lo, hi, 31, dtype=np.uint32))
    pieces.append(np.arange(0, 0x7F800000, 10007, dtype=np.uint32))
    y = np.concatenate(pieces).view(np.float32)
    y = np.concatenate([y, -y])
    got = orc.e4m3_encode_many(y)
    exp = brute_e4m3(y)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, [(float(y[i]), hex(got[i]), hex(exp[i])) for i in bad[:10]]


def test_e4m3_encode_midpoints_and_saturation(orc):
    codes, vals = _grid_e4m3()
    mids = ((vals[:-1] + vals[1:]) / 2.0).astype(np.float32)  # exact for this grid
    y = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(1e9))]).astype(np.float32)
    y = np.concatenate([y, -y])
    assert np.array_equal(orc.e4m3_encode_many(y), brute_e4m3(y))
    assert orc.e4m3_encode(1.0625) == 0x38   # tie between 1.0 (0x38) and 1.125 -> even
    assert orc.e4m3_encode(1.1875) == 0x3A   # tie between 1.125 and 1.25 (0x3A) -> even
    assert orc.e4m3_encode(448.0) == 0x7E
    assert orc.e4m3_encode(470.0) == 0x7E
    assert orc.e4m3_encode(1e30) == 0x7E
    assert orc.e4m3_encode(-1e30) == 0xFE
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-1e-30) == 0x80  # a negative that rounds to zero keeps its sign


def test_fp16_decode_matches_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.fp16_decode_many(bits)
    assert np.all((np.isnan(got) & np.isnan(ref)) | (got == ref))


def test_e2m1_grid_and_tie_table_golden(orc):
    with open(os.path.join(GOLDEN, "e2m1_grid.json")) as fh:
        g = json.load(fh)
    for i, v in enumerate(g["grid"]):
        assert orc.e2m1_index(v) == i
    for a, idx in g["ties"]:
        assert orc.e2m1_index(a) == idx, (a, idx)
    for a, idx in g["clamp"]:
        assert orc.e2m1_index(a) == idx, (a, idx)


def test_e2m1_index_bruteforce_argmin(orc):
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    near = [np.nextafter(np.float32(t), np.float32(d))
            for t in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) for d in (0, 100)]
    a = np.concatenate([np.arange(0, 12.0, 1.0 / 256), near]).astype(np.float32)
    for v in a:
        c = min(float(v), 6.0)
        d = np.abs(grid - c)
        best = np.nonzero(d == d.min())[0]
        exp = int(best[0]) if best.size == 1 else int([b for b in best if b % 2 == 0][0])
        assert orc.e2m1_index(float(v)) == exp, float(v)
