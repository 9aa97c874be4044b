"""The C-ABI library builds for sm_103a, loads without a GPU, exports every entry point that
include/w4a8.h declares, and validates arguments on the host (these calls return an error
before any CUDA call, so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

from int4_quantized_linear_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "w4a8.h")) as fh:
        src = fh.read()
    return sorted(set(re.findall(r"^W4A8_API\s+[^;(]*?\b(\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def clib():
    return binding.load()


def test_header_declares_the_four_operations():
    names = declared_entry_points()
    for n in ("w4a8_act_quant", "w4a8_mxfp4_linear", "nvfp4_to_mxfp4_requant",
              "w4a8_int4g128_linear"):
        assert n in names


def test_library_exports_every_declared_symbol(clib):
    names = declared_entry_points()
    assert len(names) >= 10
    for n in names:
        assert hasattr(clib, n), n
    assert set(binding.EXPORTS) <= set(names)


def test_status_strings(clib):
    for code, name in binding.STATUS.items():
        assert clib.w4a8_status_string(code).decode() == name
    assert clib.w4a8_decode_max_m() == 64


NULL = None


def test_host_validation_without_gpu(clib):
    # errors are returned before anything touches the device
    assert clib.w4a8_act_quant(NULL, NULL, NULL, -1, 16, NULL) == 1
    assert clib.w4a8_act_quant(NULL, NULL, NULL, 0, 16, NULL) == 0          # M = 0: no-op
    assert clib.w4a8_act_quant(NULL, NULL, NULL, 2, 16, NULL) == 1          # null pointers
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1001)
    assert clib.w4a8_act_quant(fake, fake, fake, 2, 12, NULL) == 2          # K % 8
    assert clib.w4a8_act_quant(odd, fake, fake, 2, 16, NULL) == 3           # misaligned x
    assert clib.w4a8_mxfp4_linear(fake, fake, fake, fake, fake, 2, 8, 48, NULL, 0, NULL) == 2
    assert clib.w4a8_mxfp4_linear(odd, fake, fake, fake, fake, 2, 8, 64, NULL, 0, NULL) == 3
    assert clib.w4a8_mxfp4_linear(NULL, NULL, NULL, NULL, NULL, 0, 8, 64, NULL, 0, NULL) == 0
    assert clib.w4a8_int4g128_linear(fake, fake, fake, fake, fake, 2, 8, 64, NULL, 0, NULL) == 2
    rows = (ctypes.c_int64 * 2)(3, 4)
    r = ctypes.cast(rows, ctypes.c_void_p)
    assert clib.nvfp4_to_mxfp4_requant(fake, fake, fake, r, 2, 8, 64, 2, fake, fake, NULL, NULL) == 1
    assert clib.nvfp4_to_mxfp4_requant(fake, fake, fake, r, 2, 7, 64, 3, fake, fake, NULL, NULL) == 1
    assert clib.nvfp4_to_mxfp4_requant(fake, fake, fake, r, 2, 7, 48, 2, fake, fake, NULL, NULL) == 2
    assert clib.nvfp4_to_mxfp4_requant(fake, fake, fake, r, 0, 7, 64, 2, fake, fake, NULL, NULL) == 1
    assert clib.w4a8_workspace_bytes(0, 8, 64) == 0
    # asymmetric int4, int5, the other requant sources and W4A4: the same host-side checks
    assert clib.w4a8_int4g128_asym_linear(fake, fake, fake, fake, NULL, fake, 2, 8, 128, NULL, 0, NULL) == 1
    assert clib.w4a8_int4g128_asym_linear(fake, fake, fake, fake, fake, fake, 2, 8, 64, NULL, 0, NULL) == 2
    assert clib.w4a8_int5g128_linear(fake, fake, fake, NULL, fake, NULL, fake, 2, 16, 128, NULL, 0, NULL) == 1
    assert clib.w4a8_int5g128_linear(fake, fake, fake, fake, fake, NULL, fake, 2, 16, 192, NULL, 0, NULL) == 2
    assert clib.w4a8_int5g128_linear(odd, fake, fake, fake, fake, NULL, fake, 2, 16, 128, NULL, 0, NULL) == 3
    assert clib.w4a8_int5g128_linear(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 16, 128, NULL, 0, NULL) == 0
    assert clib.fp8_channel_to_mxfp4_requant(fake, fake, 4, 48, 0, fake, fake, NULL, NULL) == 2
    assert clib.fp8_channel_to_mxfp4_requant(fake, fake, 4, 64, 3, fake, fake, NULL, NULL) == 1
    assert clib.bf16_to_mxfp4_requant(fake, 4, 48, 0, fake, fake, NULL, NULL) == 2
    assert clib.bf16_to_mxfp4_requant(odd, 4, 64, 0, fake, fake, NULL, NULL) == 3
    assert clib.w4a4_act_quant(fake, fake, fake, 2, 48, NULL) == 2
    assert clib.w4a4_act_quant(fake, fake, fake, 0, 64, NULL) == 0
    assert clib.w4a4_mxfp4_linear(fake, fake, fake, fake, fake, 2, 8, 48, NULL, 0, NULL) == 2
    assert clib.w4a4_mxfp4_linear(fake, NULL, fake, fake, fake, 2, 8, 64, NULL, 0, NULL) == 1
    assert clib.w4a4_mxfp4_linear(odd, fake, fake, fake, fake, 2, 8, 64, NULL, 0, NULL) == 3
    assert clib.w4a8_int5g128_workspace_bytes(0, 8, 128) == 0
    # the one-launch bf16 linear: 1 or 2 tokens only, same pointer and alignment checks
    single = clib.w4a8_mxfp4_linear_bf16_single
    assert single(fake, fake, fake, fake, 3, 8, 512, fake, 1 << 20, NULL) == 2
    assert single(fake, fake, fake, fake, 1, 8, 49152 + 512, fake, 1 << 20, NULL) == 2
    assert single(odd, fake, fake, fake, 1, 8, 512, fake, 1 << 20, NULL) == 3
    assert single(NULL, fake, fake, fake, 1, 8, 512, fake, 1 << 20, NULL) == 1
    assert single(NULL, NULL, NULL, NULL, 0, 8, 512, NULL, 0, NULL) == 0


def test_symmetric_zero_point_check():
    import torch
    binding.check_symmetric_qzeros(torch.full((2, 4), 0x77777777, dtype=torch.int32))
    with pytest.raises(ValueError):
        binding.check_symmetric_qzeros(torch.full((2, 4), 0x77777778, dtype=torch.int32))
    binding.check_autoround_config(4, 128, True)
    for bad in ((8, 128, True), (4, 64, True), (4, 128, False)):
        with pytest.raises(ValueError):
            binding.check_autoround_config(*bad)


def test_path_queries_without_gpu(clib):
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1001)
    # invalid arguments: the entry point would reject them
    assert clib.w4a8_mxfp4_path(fake, fake, fake, fake, 2, 8, 48) == 0     # K % 32
    assert clib.w4a8_mxfp4_path(odd, fake, fake, fake, 2, 8, 64) == 0      # misaligned xq
    assert clib.w4a8_mxfp4_path(NULL, fake, fake, fake, 2, 8, 64) == 0
    assert clib.w4a8_int4g128_path(fake, fake, fake, fake, 2, 8, 64) == 0  # K % 128
    assert clib.w4a8_int5g128_path(fake, fake, NULL, fake, fake, 2, 8, 128) == 0
    assert clib.w4a4_mxfp4_path(fake, fake, fake, fake, fake, 0, 8, 512) == 0
    # valid, but K % 512 != 0: only the CUDA-core kernels take it
    assert clib.w4a8_mxfp4_path(fake, fake, fake, fake, 2, 8, 96) == 2
    assert clib.w4a8_int4g128_path(fake, fake, fake, fake, 2, 8, 384) == 2
    assert clib.w4a8_int5g128_path(fake, fake, fake, fake, fake, 2, 16, 384) == 2
    assert clib.w4a4_mxfp4_path(fake, fake, fake, fake, fake, 2, 8, 96) == 2


def test_workspace_sizes_do_not_depend_on_policy(clib):
    shapes = [(1, 34816, 5120), (64, 5120, 17408), (4096, 10240, 5120)]
    sizes = {}
    for policy in (0, 1, 2):
        clib.w4a8_set_gemm_policy(policy)
        sizes[policy] = [(clib.w4a8_workspace_bytes(*s), clib.w4a8_int4g128_workspace_bytes(*s)) for s in shapes]
    clib.w4a8_set_gemm_policy(0)
    assert sizes[0] == sizes[1] == sizes[2]
    assert all(a > 0 and b > 0 for a, b in sizes[0])


def test_workspace_sizes_hold_the_counter_region(clib):
    # Every GEMM workspace opens with 16 KiB of arrival counters (the same place for every shape,
    # so one buffer serves any sequence of shapes), and the bf16 linear's workspace keeps that
    # region in front of the quantized activations even where the GEMM itself needs no scratch.
    counters = 16384
    for M, N, K in [(1, 34816, 5120), (8, 5120, 17408), (64, 5120, 17408), (300, 1024, 2048),
                    (4096, 10240, 5120), (1, 128, 512)]:
        g = clib.w4a8_workspace_bytes(M, N, K)
        assert g >= counters
        assert clib.w4a8_int4g128_workspace_bytes(M, N, K) >= counters
        lin = clib.w4a8_mxfp4_linear_bf16_workspace_bytes(M, N, K)
        assert lin >= g + M * K + 4 * M
    # K not a multiple of 512: no tensor-core scratch, but the linear keeps the counter region
    assert clib.w4a8_workspace_bytes(2, 96, 96) == 0
    assert clib.w4a8_mxfp4_linear_bf16_workspace_bytes(2, 96, 96) >= counters + 2 * 96 + 8
