"""The allocation-free MXFP4 entry point (w4a8_mxfp4_linear_noalloc), called through the C ABI.

Some callers of this library cannot hand it a workspace: serving engines that reserve all device
memory for their own pool and treat any other allocation as an error, and plugin interfaces that
pass a kernel only its inputs and outputs.  For them the no-alloc entry point keeps the split-K
scratch in a fixed array inside the library.  These tests check that two calls in a row through it
give the regular entry point's result and the oracle's (on sampled outputs), and that sizes beyond
the array are refused.  The file is named so pytest collects it last: a run that stops at the first
failure has then run every other test.  It also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bf16_to_f64, gemm_check, to_dev, to_dev_bf16
from int4_quantized_linear_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(8, 5120, 17408), (64, 4096, 5120), (1, 34816, 5120)])
def test_noalloc_matches_workspace_entry_point(lib, orc, M, N, K):
    clib = lib.load()
    assert clib.w4a8_noalloc_scratch_bytes() == 12 << 20
    # these shapes use the tensor-core path with stream-K scratch
    assert 0 < lib.workspace_bytes(M, N, K) <= clib.w4a8_noalloc_scratch_bytes()
    x, w, e = synth.decode_case(M, N, K, seed=M + 3)
    xq, xs = lib.act_quant(to_dev_bf16(x))
    wd, ed = to_dev(w), to_dev(e)
    ref = lib.mxfp4_linear(xq, xs, wd, ed)  # the workspace entry point
    lib.check_device_status()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # two calls in a row share (and reuse) the fixed scratch
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = clib.w4a8_mxfp4_linear_noalloc(xq.data_ptr(), xs.data_ptr(), wd.data_ptr(), ed.data_ptr(),
                                            out.data_ptr(), M, N, K, ctypes.c_void_p(stream))
        assert st == 0, lib.STATUS.get(st, st)
        lib.check_device_status()
        gemm_check(bf16_to_f64(out), bf16_to_f64(ref), f"noalloc M={M} N={N} K={K}")
        # and against the oracle, fed the same fp8 codes, on outputs sampled across every tile
        rng = np.random.default_rng(M)
        im = rng.integers(0, M, 512)
        inn = rng.integers(0, N, 512)
        o_ref = orc.mxfp4_linear_pairs(xq.cpu().numpy(), xs.cpu().numpy(), w, e, im, inn)
        gemm_check(bf16_to_f64(out)[im, inn], o_ref, f"noalloc vs oracle M={M} N={N} K={K}")


def test_noalloc_rejects_oversized(lib):
    clib = lib.load()
    M, N, K = 4096, 34816, 5120  # prefill-sized scratch does not fit the fixed array
    assert lib.workspace_bytes(M, N, K) > clib.w4a8_noalloc_scratch_bytes()
    xq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    xs = torch.ones(M, dtype=torch.float32, device="cuda")
    w = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    e = torch.zeros((N, K // 32), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = clib.w4a8_mxfp4_linear_noalloc(xq.data_ptr(), xs.data_ptr(), w.data_ptr(), e.data_ptr(), out.data_ptr(),
                                        M, N, K, None)
    assert st == 4  # W4A8_ERR_WORKSPACE, nothing launched
