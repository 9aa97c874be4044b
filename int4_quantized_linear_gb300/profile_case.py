"""One small, self-checking invocation of one hot-path kernel, for profilers.

    python -m int4_quantized_linear_gb300.profile_case --m 1 --n 34816 --k 5120 --calls 3

Builds synthetic inputs of the given shape (the same recipe as the benchmark), runs the
per-token activation quant once and the MXFP4 GEMM ``--calls`` times on ``cuda:0``, then checks
the library's device status word; exits non-zero if a bounded wait ran out.  Meant as the
target of ``ncu -k regex:mxfp4_tc -c <calls>`` (``regex:int4_tc`` with ``--int4`` or ``--int5`` up to
128 tokens, ``regex:int4_pf`` above;
``--w4a4`` runs the MXFP4-activation path, whose GEMM is also ``mxfp4_tc``): it launches nothing
else of note.  ``--act-quant`` runs only the per-token activation quant of x [M, K]
(``regex:act_quant``) and ``--requant MODE`` the NVFP4 -> MXFP4 requant of an [N, K] merged
weight of two equal partitions (``regex:requant``), each ``--calls`` times.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import binding as lib
from . import synth


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--n", type=int, default=synth.GATE_UP[0])
    ap.add_argument("--k", type=int, default=synth.GATE_UP[1])
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--int4", action="store_true", help="the AutoRound int4 g128 GEMM instead of MXFP4")
    ap.add_argument("--int5", action="store_true", help="the int5 g128 GEMM (zero point 16) instead of MXFP4")
    ap.add_argument("--w4a4", action="store_true", help="MXFP4 activations (W4A4) instead of fp8 ones")
    ap.add_argument("--act-quant", action="store_true", help="only the per-token activation quant")
    ap.add_argument("--fused", action="store_true",
                    help="the whole linear from bf16 x (w4a8_mxfp4_linear_bf16: activation quant, then the GEMM)")
    ap.add_argument("--single", action="store_true",
                    help="the whole linear from bf16 x as one kernel (w4a8_mxfp4_linear_bf16_single, 1-2 tokens)")
    ap.add_argument("--requant", choices=["ocp", "noclip", "mse"], help="only the NVFP4 -> MXFP4 requant")
    args = ap.parse_args(argv)
    M, N, K = args.m, args.n, args.k
    lib.load()
    dev = torch.device("cuda", 0)
    if args.requant:
        nv_p, nv_s = synth.nvfp4_tensor_bytes(N, K, 0)
        nvp, nvs = torch.from_numpy(nv_p).to(dev), torch.from_numpy(nv_s).to(dev)
        div = torch.tensor([2688.0, 10752.0], dtype=torch.float32, device=dev)
        parts = [N // 2, N - N // 2]
        for _ in range(args.calls):
            lib.requant(nvp, nvs, div, parts, args.requant, err_ssq=True)
        torch.cuda.synchronize()
        print(f"ok requant {args.requant} N={N} K={K} calls={args.calls}")
        return 0
    x = torch.from_numpy(np.ascontiguousarray(synth.activations(M, K, seed=M)).view(np.int16)).to(dev)
    xq, xs = lib.act_quant(x.view(torch.bfloat16))
    if args.act_quant:
        for _ in range(args.calls - 1):
            lib.act_quant(x.view(torch.bfloat16), xq, xs)
        torch.cuda.synchronize()
        print(f"ok act_quant M={M} K={K} calls={args.calls}")
        return 0
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if args.int5:
        qw, qh, sc = synth.int5_weights(N, K, 0)
        qd, hd = torch.from_numpy(qw).to(dev), torch.from_numpy(qh).to(dev)
        sd = torch.from_numpy(sc).to(dev).view(torch.float16)
        ws = lib.make_workspace(lib.int5_workspace_bytes(M, N, K), dev)
        for _ in range(args.calls):
            lib.int5g128_linear(xq, xs, qd, hd, sd, out=out, workspace=ws)
    elif args.w4a4:
        w, e = synth.mxfp4_weights(N, K, 0, 118, 121)
        wd, ed = torch.from_numpy(w).to(dev), torch.from_numpy(e).to(dev)
        xa, xe = lib.act_quant_mxfp4(x.view(torch.bfloat16))
        ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
        for _ in range(args.calls):
            lib.mxfp4_a4_linear(xa, xe, wd, ed, out=out, workspace=ws)
    elif args.fused or args.single:
        w, e = synth.mxfp4_weights(N, K, 0, 118, 121)
        wd, ed = torch.from_numpy(w).to(dev), torch.from_numpy(e).to(dev)
        lws = lib.make_linear_workspace(M, N, K, dev)
        for _ in range(args.calls):
            lib.linear(x.view(torch.bfloat16), wd, ed, out=out, workspace=lws, single_kernel=args.single)
    elif args.int4:
        qw, sc, _ = synth.int4_weights(N, K, 0)
        qd = torch.from_numpy(qw).to(dev)
        sd = torch.from_numpy(sc).to(dev).view(torch.float16)
        ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
        for _ in range(args.calls):
            lib.int4g128_linear(xq, xs, qd, sd, out=out, workspace=ws)
    else:
        w, e = synth.mxfp4_weights(N, K, 0, 118, 121)
        wd = torch.from_numpy(w).to(dev)
        ed = torch.from_numpy(e).to(dev)
        ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
        for _ in range(args.calls):
            lib.mxfp4_linear(xq, xs, wd, ed, out=out, workspace=ws)
    torch.cuda.synchronize()
    lib.check_device_status()
    kind = "int5" if args.int5 else "w4a4" if args.w4a4 else "int4" if args.int4 else "single" if args.single else "fused" if args.fused else "mxfp4"
    print(f"ok {kind} M={M} N={N} K={K} calls={args.calls}")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
