"""W4A8 quantized-linear benchmark (decode band, MXFP4).

Workload (one step): for each of the two served shapes -- gate_up N=34816 K=5120 and down
N=5120 K=17408 -- and each decode batch M in {1, 8, 32, 64}: per-token fp8 activation quant
of x [M, K] followed by the MXFP4 W4A8 GEMM (one w4a8_mxfp4_linear_bf16 call, two kernels
chained by programmatic dependent launch), 16 kernel launches in all.  Each (shape, M)
pair owns its own weight copy, so one step streams 568 MB of weights (more than the 129 MB
L2): every GEMM reads its weights from HBM.  The step is captured once in a CUDA graph and
replayed.

Metric: decode weight GB/s = weight bytes (N*K*(1/2 + 1/32) per GEMM) per step / step time.

Also reported on the same line:
  roofline      the decode GEMM kernel's achieved weight GB/s against the measured HBM copy
                bandwidth, from CUDA events around each GEMM in a graph replay pass;
  e2e           the same metric through the public Python API with host buffers: pinned host
                x -> device, act quant + GEMM, bf16 output -> host, every step;
  cpu_baseline  the CPU oracle on a bounded sample of the same workload;
  prefill / int4 / requant   the other hot-path kernels on their workloads (--extras).

--impl reference times the CPU oracle (the only reference implementation this project has)
on the same workload, as a bounded sample per step.
Multi-GPU (torchrun): independent replicas, one per GPU; value = all ranks' bytes / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from int4_quantized_linear_gb300 import synth  # noqa: E402

SHAPES = [("gate_up", synth.GATE_UP), ("down", synth.DOWN)]
DECODE_M = [1, 8, 32, 64]
METRIC = "W4A8 GEMM: decode weight GB/s and prefill TFLOP/s, % of GB300 roofline"
WORKLOAD = ("decode band MXFP4 W4A8: M in {1,8,32,64} x {gate_up N=34816 K=5120, down N=5120 "
            "K=17408}; act quant + GEMM per (shape, M), one w4a8_mxfp4_linear_bf16 call each")


def weight_bytes(N, K):
    return N * K // 2 + N * K // 32


def decode_traffic():
    """DRAM bytes per decode-GEMM launch (mean over the step's 8 launches) from the committed ncu
    capture, or None when the kernel's sources changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "decode_gemm_traffic.json")) as fh:
            rec = json.load(fh)
        h = hashlib.sha256()
        for s in rec["sources"]:
            with open(os.path.join(ROOT, s), "rb") as fh:
                h.update(fh.read())
        return rec["dram_bytes_per_launch_mean"] if h.hexdigest() == rec["sources_sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for t, r in self.rows if t0 <= t <= t1]
        window = "timed region"
        if len(rows) < 3:  # short timed region: widen to the surrounding load phase
            mid = 0.5 * (t0 + t1)
            rows = [r for t, r in self.rows if abs(t - mid) <= max(1.0, 0.5 * (t1 - t0))]
            window = "timed region +-1 s"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        smax = None
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


# ---------------------------------------------------------------------------------- CPU side

def aggregate(elapsed_ms, step_bytes, steps, world, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: every rank did step_bytes per step; the
    job time is the slowest rank's (max over ranks).  Returns (GB/s, max elapsed ms)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return world * step_bytes * steps / (elapsed_ms * 1e-3) / 1e9, elapsed_ms


def oracle_sample(orc, cases, budget_s):
    """Time the oracle GEMM (act quant of the sample rows + dequantize-and-matmul) over a
    column sample of every (shape, M) case; returns (weight bytes processed, seconds)."""
    done_bytes = 0
    total_t = 0.0
    per_case = budget_s / len(cases)
    for (name, (N, K), M, x, w, e) in cases:
        # calibrate columns so this case costs about per_case seconds
        cols = 8
        t_start = time.perf_counter()
        xq, xs = orc.act_quant(x)
        while True:
            n_idx = np.arange(cols) % N
            im = np.repeat(np.arange(M), cols)
            inn = np.tile(n_idx, M)
            t0 = time.perf_counter()
            orc.mxfp4_linear_pairs(xq, xs, w, e, im, inn)
            dt = time.perf_counter() - t0
            if dt >= per_case * 0.5 or cols >= N:
                break
            cols = min(N, int(cols * max(2.0, per_case / max(dt, 1e-4))))
        total_t += time.perf_counter() - t_start
        done_bytes += cols * (K // 2 + K // 32)
    return done_bytes, total_t


def make_host_cases(seed=0):
    cases = []
    for name, (N, K) in SHAPES:
        w, e = synth.mxfp4_weights(N, K, seed, 118, 121)
        for M in DECODE_M:
            cases.append((name, (N, K), M, synth.activations(M, K, seed + M), w, e))
    return cases


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    cases = make_host_cases()
    budget = float(os.environ.get("W4A8_REF_STEP_S", "1.0"))
    for _ in range(args.warmup):
        oracle_sample(orc, cases, budget * 0.25)
    tot_b, tot_t = 0, 0.0
    for _ in range(args.steps):
        b, t = oracle_sample(orc, cases, budget)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    cores = orc.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle: e4m3 x e2m1 dequantized exactly, fp64 accumulate)",
        "data": "synthetic", "config": {"workload": WORKLOAD, "parallelism": "cpu oracle",
                                        "sample": "output-column sample per (shape, M)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"~{budget:.1f} s of oracle GEMM per step over column samples of all 8 (shape, M) cases"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- GPU side

def run_ours(args, rank, world, local_rank):
    import torch
    from int4_quantized_linear_gb300 import binding as lib

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib.load()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def to_dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- workload: one weight copy per (shape, M), inputs resident in HBM
    calls = []
    for name, (N, K) in SHAPES:
        w_host, e_host = synth.mxfp4_weights(N, K, 0, 118, 121)
        w0, e0 = to_dev(w_host), to_dev(e_host)
        for i, M in enumerate(DECODE_M):
            w = w0 if i == 0 else w0.clone()
            e = e0 if i == 0 else e0.clone()
            x_host = synth.activations(M, K, seed=M)
            x = to_dev_bf16(x_host)
            xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
            xs = torch.empty((M,), dtype=torch.float32, device=dev)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
            lws = lib.make_linear_workspace(M, N, K, dev)
            calls.append(dict(name=name, N=N, K=K, M=M, w=w, e=e, x=x, x_host=x_host, xq=xq, xs=xs,
                              out=out, ws=ws, lws=lws, bytes=weight_bytes(N, K)))
    step_bytes = sum(c["bytes"] for c in calls)
    clib = lib.load()
    stream = torch.cuda.Stream(device=dev)

    def launch(c, s):
        # one native call per (shape, M): activation quant, then the GEMM (chained on the stream)
        lws = c["lws"]
        st = clib.w4a8_mxfp4_linear_bf16(c["x"].data_ptr(), c["w"].data_ptr(), c["e"].data_ptr(),
                                         c["out"].data_ptr(), c["M"], c["N"], c["K"], lws.data_ptr(),
                                         lws.numel(), s)
        if st:
            raise lib.W4A8Error("w4a8_mxfp4_linear_bf16", st)

    # eager warm-up (also makes the library's lazy per-device set-up happen outside capture)
    with torch.cuda.stream(stream):
        for c in calls:
            launch(c, stream.cuda_stream)
    stream.synchronize()
    lib.check_device_status(stream)  # a bounded wait that ran out means the kernels are broken

    # ---- step graph, and a second graph with timing events around every GEMM
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for c in calls:
            launch(c, stream.cuda_stream)
    ev_graph = None
    evs = None
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in calls]
        ev_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ev_graph, stream=stream):
            for c, (a, b) in zip(calls, evs):
                st = clib.w4a8_act_quant(c["x"].data_ptr(), c["xq"].data_ptr(), c["xs"].data_ptr(),
                                         c["M"], c["K"], stream.cuda_stream)
                a.record(stream)
                ws = c["ws"]
                clib.w4a8_mxfp4_linear(c["xq"].data_ptr(), c["xs"].data_ptr(), c["w"].data_ptr(),
                                       c["e"].data_ptr(), c["out"].data_ptr(), c["M"], c["N"], c["K"],
                                       None if ws is None else ws.data_ptr(),
                                       0 if ws is None else ws.numel(), stream.cuda_stream)
                b.record(stream)
    except (TypeError, RuntimeError):
        ev_graph = None

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    # keep the GPU busy for a moment so the clock samples see the load
    t_load = time.time()
    while time.time() - t_load < 0.5:
        graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    value, elapsed_ms = aggregate(e0.elapsed_time(e1), step_bytes, args.steps, world, dist, dev)
    ms_per_step = elapsed_ms / args.steps

    # ---- per-kernel durations of the decode GEMM (same graph, event-bracketed GEMMs)
    gemm_ms = [0.0] * len(calls)
    reps = max(3, min(args.steps, 50))
    if ev_graph is not None:
        for _ in range(reps):
            ev_graph.replay()
            torch.cuda.synchronize()
            for i, (a, b) in enumerate(evs):
                gemm_ms[i] += a.elapsed_time(b) / reps
    # ---- the same 8 GEMMs back to back (one graph, chained by programmatic dependent launch,
    # activations already quantized by the runs above): the kernels' sustained rate in a chain
    chain_us = None
    try:
        cgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cgraph, stream=stream):
            for c in calls:
                ws = c["ws"]
                clib.w4a8_mxfp4_linear(c["xq"].data_ptr(), c["xs"].data_ptr(), c["w"].data_ptr(),
                                       c["e"].data_ptr(), c["out"].data_ptr(), c["M"], c["N"], c["K"],
                                       None if ws is None else ws.data_ptr(),
                                       0 if ws is None else ws.numel(), stream.cuda_stream)
        for _ in range(3):
            cgraph.replay()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                cgraph.replay()
        c1.record(stream)
        torch.cuda.synchronize()
        chain_us = 1e3 * c0.elapsed_time(c1) / reps
    except (TypeError, RuntimeError):
        chain_us = None
    t_kern_end = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    peaks, peak_src = load_peaks()
    traffic = decode_traffic()
    roofline = None
    if ev_graph is not None:
        ach = sum(c["bytes"] for c in calls) / (sum(gemm_ms) * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"], "traffic": traffic,
                    "algorithmic_bytes_per_launch": sum(c["bytes"] for c in calls) / len(calls),
                    "kernel": "decode-band MXFP4 GEMM (w4a8_mxfp4_linear, M<=64)",
                    "peak_source": peak_src,
                    "per_case_us": {f"{c['name']}_M{c['M']}": round(1e3 * g, 2) for c, g in zip(calls, gemm_ms)},
                    "timing": "each GEMM bracketed by CUDA events in a replica of the step graph (so "
                              "it starts cold, without programmatic overlap with its neighbours)"}
        if chain_us:
            roofline["gemm_chain"] = {"us_per_step": round(chain_us, 2),
                                      "GB/s": round(step_bytes / (chain_us * 1e-6) / 1e9, 1),
                                      "note": "the 8 GEMMs back to back in one graph, no activation quant"}

    # ---- e2e through the public API with host buffers
    h2d = sum(c["M"] * c["K"] * 2 for c in calls)
    d2h = sum(c["M"] * c["N"] * 2 for c in calls)
    pinned_x = [torch.from_numpy(c["x_host"].view(np.int16)).view(torch.bfloat16).pin_memory() for c in calls]
    pinned_o = [torch.empty((c["M"], c["N"]), dtype=torch.bfloat16).pin_memory() for c in calls]
    dev_x = [torch.empty((c["M"], c["K"]), dtype=torch.bfloat16, device=dev) for c in calls]
    dev_o = [torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device=dev) for c in calls]
    e2e_steps = max(3, min(args.steps, 20))

    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        # per call: pinned host x -> device, the public linear(), device out -> pinned host.  The
        # copies run on a second stream (inputs first, each output as soon as its GEMM is done),
        # so they overlap the other calls' kernels, as a serving loop would pipeline them.
        copy_stream.wait_stream(stream)
        x_ready, o_ready = [], []
        with torch.cuda.stream(copy_stream):
            for hx, xd in zip(pinned_x, dev_x):
                xd.copy_(hx, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                x_ready.append(ev)
        with torch.cuda.stream(stream):
            for c, xd, od, ev in zip(calls, dev_x, dev_o, x_ready):
                stream.wait_event(ev)
                lib.linear(xd, c["w"], c["e"], out=od, workspace=c["lws"], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                o_ready.append(done)
        with torch.cuda.stream(copy_stream):
            for ho, od, done in zip(pinned_o, dev_o, o_ready):
                copy_stream.wait_event(done)
                ho.copy_(od, non_blocking=True)
        stream.wait_stream(copy_stream)

    def wall(fn, n):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    e2e_eager_s = wall(e2e_step, e2e_steps)
    # the same calls and copies captured once in a CUDA graph, as a serving loop replays a decode
    # step: every replay still copies x in from pinned host memory and the outputs back out
    g_e2e = torch.cuda.CUDAGraph()
    e2e_step()
    stream.synchronize()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_step()
    e2e_s = wall(lambda: g_e2e.replay(), e2e_steps)
    if not all(torch.equal(ho, od.cpu()) for ho, od in zip(pinned_o, dev_o)):
        raise RuntimeError("end-to-end outputs copied back do not match the device outputs")
    e2e_val = step_bytes * e2e_steps / e2e_s / 1e9
    e2e_eager_val = step_bytes * e2e_steps / e2e_eager_s / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e2m1 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "weight_bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2: 8 distinct weight copies, 568 MB per step",
                   "graph": "step captured in a CUDA graph", "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "per (shape, M): pinned host x -> device, binding.linear, device out -> pinned host, "
                        "copies on a second stream overlapping the kernels; the step captured in a CUDA "
                        "graph and replayed, wall-clock timed",
                "eager_value": e2e_eager_val},
        "gpu_launches": 2 * len(calls) * args.steps,
    }
    if not args.no_extras and rank == 0:
        line["extras"] = run_extras(lib, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        b, t = oracle_sample(orc, make_host_cases(), float(os.environ.get("W4A8_CPU_BASELINE_S", "12")))
        line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s", "cores": orc.num_threads(),
                                "kind": "oracle",
                                "sample": f"oracle act quant + GEMM on output-column samples of all 8 (shape, M) cases, {t:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_extras(lib, dev, peaks):
    """Prefill, int4 and requant kernels on their workloads (event-timed, inputs > L2)."""
    import torch
    out = {}

    def timeit(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def to_dev(arr):
        return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)

    def timeit_rot(fns, reps=24):
        """Average time of one call, cycling over calls that touch different buffers (so the
        working set exceeds L2); the calls are captured in a CUDA graph, so host-side launch
        cost does not enter the figure."""
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            for f in fns:
                f()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(reps):
                fns[i % len(fns)]()
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        with torch.cuda.stream(s):
            g.replay()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    fp8_peak = 2.0 * peaks.get("bf16_tflops", 1900.0)
    pf = {}
    for name, (N, K) in SHAPES + [("qkv", synth.QKV)]:
        w, e = synth.mxfp4_weights(N, K, 0, 118, 124)
        # three weight copies in rotation, so weights + activations exceed L2 between calls
        wds = [to_dev(w) for _ in range(3)]
        eds = [to_dev(e) for _ in range(3)]
        for M in (512, 2048, 4096):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.mxfp4_linear(xq, xs, a, b, out=o, workspace=ws) for a, b in zip(wds, eds)]
            ms = timeit_rot(fns, reps=12)
            tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            pf[f"{name}_M{M}"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                  "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        del wds, eds
    out["prefill"] = {"fp8_peak_tflops": fp8_peak,
                      "peak_note": "2 x measured bf16 burst (fp8 dense rate is twice bf16)",
                      "timing": "CUDA graph of 12 calls over 3 weight copies, persistent workspace", "cases": pf}
    hbm = peaks["hbm_gbs"]


    # ---- per-token activation quant: 2MK bytes read, MK + 4M written
    aq = {}
    for M, K in ((1, 17408), (64, 17408), (4096, 5120), (4096, 17408)):
        n_copies = max(2, int(3 * 129e6 // (3 * M * K)) + 1) if M * K * 3 > 4e6 else 8
        xs_ = [torch.randn((M, K), device=dev).to(torch.bfloat16) for _ in range(min(n_copies, 8))]
        qs_ = [(torch.empty((M, K), dtype=torch.uint8, device=dev), torch.empty((M,), dtype=torch.float32, device=dev))
               for _ in xs_]
        fns = [lambda x=x, q=q: lib.act_quant(x, q[0], q[1]) for x, q in zip(xs_, qs_)]
        ms = timeit_rot(fns)
        gbs = (3 * M * K + 4 * M) / (ms * 1e-3) / 1e9
        aq[f"M{M}_K{K}"] = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4)}
        del xs_, qs_
    out["act_quant"] = {"bound": "hbm", "peak_gbs": hbm, "cases": aq}

    # ---- NVFP4 -> MXFP4 requant of the merged gate_up weight (two partitions)
    N, K = synth.GATE_UP
    nv_p, nv_s = synth.nvfp4_tensor_bytes(N, K, 0)
    nvp, nvs = to_dev(nv_p), to_dev(nv_s)
    div = torch.tensor([2688.0, 10752.0], dtype=torch.float32, device=dev)
    o_p = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    o_e = torch.empty((N, K // 32), dtype=torch.uint8, device=dev)
    rq_bytes = N * K // 2 + N * K // 16 + N * K // 2 + N * K // 32
    rq = {}
    for mode in ("ocp", "noclip", "mse"):
        ms = timeit(lambda: lib.requant(nvp, nvs, div, list(synth.GATE_UP_PARTITIONS), mode, o_p, o_e, err_ssq=True))
        gbs = rq_bytes / (ms * 1e-3) / 1e9
        rq[mode] = {"us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4)}
    out["requant"] = {"bound": "hbm", "peak_gbs": hbm, "bytes": rq_bytes,
                      "config": "gate_up N=34816 K=5120, partitions 17408+17408, with per-partition error sums",
                      "cases": rq}
    del nvp, nvs

    # ---- FP8-per-channel and bf16 -> MXFP4 requant, same shape, mse rule, with error sums
    w8_h, s8_h = synth.fp8_channel_weights(N, K, 0)
    w8, s8 = to_dev(w8_h), to_dev(s8_h)
    ms = timeit(lambda: lib.requant_fp8_channel(w8, s8, "mse", o_p, o_e, err_ssq=True))
    by = N * K + 4 * N + N * K // 2 + N * K // 32
    gbs = by / (ms * 1e-3) / 1e9
    other = {"fp8_channel_mse": {"us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                                 "bytes": by}}
    del w8, s8, w8_h
    wb = torch.from_numpy(synth.bf16_weights(N, K, 0).view(np.int16)).to(dev).view(torch.bfloat16)
    ms = timeit(lambda: lib.requant_bf16(wb, "mse", o_p, o_e, err_ssq=True))
    by = 2 * N * K + N * K // 2 + N * K // 32
    gbs = by / (ms * 1e-3) / 1e9
    other["bf16_mse"] = {"us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4), "bytes": by}
    out["requant_other_sources"] = {"bound": "alu (as the NVFP4 requant)", "peak_gbs": hbm,
                                    "config": "gate_up N=34816 K=5120, one partition, mse rule, with error sums",
                                    "cases": other}
    del wb, o_p, o_e

    # ---- AutoRound int4 g128: decode weight GB/s, prefill TFLOP/s
    i4 = {}
    for name, (N, K) in SHAPES:
        qw, sc, _ = synth.int4_weights(N, K, 0)
        wb = N * K // 2 + N * K // 64
        n_copies = 3
        qws = [to_dev(qw) for _ in range(n_copies)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(n_copies)]
        for M in (1, 8, 64):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.int4g128_linear(xq, xs, a, b, out=o, workspace=ws) for a, b in zip(qws, scs)]
            ms = timeit_rot(fns)
            gbs = wb / (ms * 1e-3) / 1e9
            i4[f"{name}_M{M}"] = {"us": round(ms * 1e3, 2), "weight GB/s": round(gbs, 1),
                                  "frac_of_hbm": round(gbs / hbm, 4)}
        M = 4096
        x = torch.randn((M, K), device=dev).to(torch.bfloat16)
        xq, xs = lib.act_quant(x)
        o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
        ms = timeit(lambda: lib.int4g128_linear(xq, xs, qws[0], scs[0], out=o, workspace=ws), reps=2)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        i4[f"{name}_M{M}"] = {"ms": round(ms, 3), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        del qws, scs
    out["int4g128"] = {"decode_bound": "hbm", "prefill_bound": "tensor (fp8 peak)", "cases": i4}

    # ---- asymmetric int4 g128 (per-group, per-column zero points): decode GB/s, M = 1 and 64
    i4a = {}
    for name, (N, K) in SHAPES:
        qw, sc, _ = synth.int4_weights(N, K, 0)
        qz = to_dev(synth.int4_asym_zeros(N, K, 0))
        wb = N * K // 2 + N * K // 64 + (K // 128) * ((N + 7) // 8) * 4
        qws = [to_dev(qw) for _ in range(3)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(3)]
        for M in (1, 64):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.int4g128_asym_linear(xq, xs, a, b, qz, out=o, workspace=ws)
                   for a, b in zip(qws, scs)]
            ms = timeit_rot(fns)
            gbs = wb / (ms * 1e-3) / 1e9
            i4a[f"{name}_M{M}"] = {"us": round(ms * 1e3, 2), "weight GB/s": round(gbs, 1),
                                   "frac_of_hbm": round(gbs / hbm, 4)}
        del qws, scs, qz
    out["int4g128_asym"] = {"decode_bound": "hbm", "cases": i4a}

    # ---- int5 g128 (fifth-bit plane; zero point 16, or a byte per group and column): decode
    # weight GB/s at M = 1 and 64, prefill TFLOP/s at M = 4096
    i5 = {}
    for name, (N, K) in SHAPES:
        qw, qh, sc = synth.int5_weights(N, K, 0)
        z5 = to_dev(synth.int5_zeros(N, K, 0))
        wb = N * K // 2 + N * K // 8 + N * K // 64
        qws = [to_dev(qw) for _ in range(3)]
        qhs = [to_dev(qh) for _ in range(3)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(3)]
        for M in (1, 64):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int5_workspace_bytes(M, N, K), dev)
            for tag, z in (("", None), ("_asym", z5)):
                fns = [lambda a=a, h=h, b=b, z=z: lib.int5g128_linear(xq, xs, a, h, b, z, out=o, workspace=ws)
                       for a, h, b in zip(qws, qhs, scs)]
                ms = timeit_rot(fns)
                by = wb + (0 if z is None else (K // 128) * N)
                gbs = by / (ms * 1e-3) / 1e9
                i5[f"{name}_M{M}{tag}"] = {"us": round(ms * 1e3, 2), "weight GB/s": round(gbs, 1),
                                           "frac_of_hbm": round(gbs / hbm, 4)}
        M = 4096
        x = torch.randn((M, K), device=dev).to(torch.bfloat16)
        xq, xs = lib.act_quant(x)
        o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = lib.make_workspace(lib.int5_workspace_bytes(M, N, K), dev)
        ms = timeit(lambda: lib.int5g128_linear(xq, xs, qws[0], qhs[0], scs[0], out=o, workspace=ws), reps=2)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        i5[f"{name}_M{M}"] = {"ms": round(ms, 3), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        del qws, qhs, scs, z5
    # ---- W4A4 (MXFP4 activations by the OCP rule): GEMM decode weight GB/s, prefill TFLOP/s,
    # activation quant latency, and the relative error of W4A4 and W4A8 against the exact product
    a4 = {}
    for name, (N, K) in SHAPES:
        _, wp, we = synth.decode_case(1, N, K, 0)
        wb = N * K // 2 + N * K // 32
        wps = [to_dev(wp) for _ in range(3)]
        wes = [to_dev(we) for _ in range(3)]
        for M in (1, 64, 4096):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xa, xe = lib.act_quant_mxfp4(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
            if M < 4096:
                fns = [lambda a=a, b=b: lib.mxfp4_a4_linear(xa, xe, a, b, out=o, workspace=ws) for a, b in zip(wps, wes)]
                ms = timeit_rot(fns)
                gbs = wb / (ms * 1e-3) / 1e9
                a4[f"{name}_M{M}"] = {"us": round(ms * 1e3, 2), "weight GB/s": round(gbs, 1),
                                      "frac_of_hbm": round(gbs / hbm, 4)}
                ms = timeit_rot([lambda: lib.act_quant_mxfp4(x, xa, xe)], reps=24)
                a4[f"act_quant_{name}_M{M}"] = {"us": round(ms * 1e3, 2)}
            else:
                ms = timeit(lambda: lib.mxfp4_a4_linear(xa, xe, wps[0], wes[0], out=o, workspace=ws), reps=2)
                tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
                a4[f"{name}_M{M}"] = {"ms": round(ms, 3), "tflops": round(tf, 1),
                                      "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        del wps, wes
    M, N, K = 16, 4096, 5120
    x = torch.randn((M, K), device=dev).to(torch.bfloat16)
    _, wp, we = synth.decode_case(1, N, K, 1)
    wpd, wed = to_dev(wp), to_dev(we)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = np.stack([wp & 0x0F, wp >> 4], -1).reshape(N, K)
    wv = grid[codes & 7] * np.where(codes & 8, -1.0, 1.0) * np.repeat(np.exp2(we.astype(np.float64) - 127), 32, 1)
    wf = torch.from_numpy(wv).to(dev)  # the MXFP4 weights' exact values
    exact = x.double() @ wf.T
    xq, xs = lib.act_quant(x)
    xa, xe = lib.act_quant_mxfp4(x)
    rel = lambda o: float(torch.linalg.norm(o.double() - exact) / torch.linalg.norm(exact))
    a4["rel_error_vs_exact"] = {"w4a8": round(rel(lib.mxfp4_linear(xq, xs, wpd, wed)), 5),
                                "w4a4": round(rel(lib.mxfp4_a4_linear(xa, xe, wpd, wed)), 5),
                                "case": f"M={M} N={N} K={K}, x ~ N(0,1) bf16, uniform MXFP4 weights"}
    out["w4a4"] = {"decode_bound": "hbm", "prefill_bound": "tensor (fp8 rate: e2m1 x e2m1 in kind::mxf8f6f4)",
                   "cases": a4}

    out["int5g128"] = {"decode_bound": "hbm", "prefill_bound": "tensor (fp8 peak)",
                       "weight_bytes": "N*K*(1/2 + 1/8 + 2/128) (+ K/128*N zero bytes for asym)", "cases": i5}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other hot-path kernels (prefill, act quant, requant, int4)")
    ap.add_argument("--extras", action="store_true", help="(default) kept for compatibility")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
