"""W4A8 quantized-linear benchmark (decode band, MXFP4).

Workload (one step): for each of the two served shapes -- gate_up N=34816 K=5120 and down
N=5120 K=17408 -- and each decode batch M in {1, 8, 32, 64}: per-token fp8 activation quant
of x [M, K] followed by the MXFP4 W4A8 GEMM (one w4a8_mxfp4_linear_bf16 call).  Each (shape, M)
pair owns its own weight copy, so one step streams 568 MB of weights (more than the 129 MB L2):
every GEMM reads its weights from HBM.  The step is captured once in a CUDA graph and replayed.

Metric: decode weight GB/s = weight bytes (N*K*(1/2 + 1/32) per GEMM) per step / step time.

Also reported on the same line:
  roofline          the decode GEMM kernel against the measured HBM copy bandwidth: the step's
                    eight GEMMs back to back in one graph (the kernel as it runs inside the step);
                    the cold, event-bracketed per-GEMM figure is kept as frac_cold;
  decode_cases      every decode-band GEMM format (W4A8, W4A4, int4, int5) per (shape, M) under
                    one protocol: a graph of back-to-back calls cycling over weight copies > L2;
  prefill_roofline  the M=4096 prefill GEMMs against the dense fp8 peak measured in the same run;
  e2e               the same metric through the public Python API with host buffers: pinned host
                    x -> device, act quant + GEMM, bf16 output -> host, every step;
  cpu_baseline      the CPU oracle on a fixed sample of the same workload (the same sample, per
                    pass, that --impl reference times);
  extras            the other hot-path kernels (act quant, requant, asymmetric int4, ...).

--impl reference times the CPU oracle (the only reference implementation this project has) on
the same workload: one pass of the fixed sample per step.
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
# Oracle sample: per (shape, M) case, every token row and SAMPLE_COLS output columns spread
# over N by stride; one pass = activation quant of the rows + the sampled GEMM outputs.
SAMPLE_COLS = 64
# Decode-band per-case protocol shared by every format: a graph of CHAIN_REPS back-to-back calls
# of one (shape, M) case cycling over weight copies whose total exceeds L2.
CHAIN_REPS = 24


def weight_bytes(N, K):
    return N * K // 2 + N * K // 32


STEP_BYTES = sum(weight_bytes(N, K) for _, (N, K) in SHAPES for _ in DECODE_M)


def bench_config(world):
    """The workload description shared by both arms (the driver compares them)."""
    return {"workload": WORKLOAD, "weight_bytes_per_step": STEP_BYTES,
            "l2": "inputs larger than L2: 8 distinct weight copies, 568 MB per step",
            "parallelism": f"replicas x{world}"}


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


def make_oracle_sample(seed=0):
    """The fixed oracle sample: per (shape, M) case of the step, the case's activations (the same
    seeded x the GPU arm uses), its weights, and SAMPLE_COLS output columns spread over N."""
    sample = []
    for name, (N, K) in SHAPES:
        w, e = synth.mxfp4_weights(N, K, seed, 118, 121)
        cols = (np.arange(SAMPLE_COLS, dtype=np.int64) * N) // SAMPLE_COLS
        for M in DECODE_M:
            x = synth.activations(M, K, seed=seed + M)
            im = np.repeat(np.arange(M, dtype=np.int64), SAMPLE_COLS)
            inn = np.tile(cols, M)
            sample.append((x, w, e, im, inn, SAMPLE_COLS * (K // 2 + K // 32)))
    return sample


SAMPLE_NOTE = (f"one pass = oracle act quant of every token row + {SAMPLE_COLS} output columns (spread over N "
               f"by stride) of each of the 8 (shape, M) cases; weight GB/s = sampled weight bytes / time")


def oracle_pass(orc, sample):
    """One pass of the oracle over the fixed sample; returns the weight bytes it covered."""
    done = 0
    for x, w, e, im, inn, nbytes in sample:
        xq, xs = orc.act_quant(x)
        orc.mxfp4_linear_pairs(xq, xs, w, e, im, inn)
        done += nbytes
    return done


def oracle_timed(orc, sample, budget_s):
    """Whole passes until budget_s has elapsed (at least one); every timed pass is counted."""
    oracle_pass(orc, sample)  # warm-up: page in the weights
    done, t0 = 0, time.perf_counter()
    while True:
        done += oracle_pass(orc, sample)
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            return done, dt


def oracle_other(orc, budget_s=1.5):
    """The oracle's other hot-path steps on bounded samples of their workloads: activation quant
    (M=64, K=17408), NVFP4 -> MXFP4 requant (2048 rows of gate_up, mse), and a prefill GEMM sample
    (gate_up, M=4096, 16 output columns)."""
    out = {}

    def rep(fn):
        fn()
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                return n, dt

    M, K = 64, 17408
    x = synth.activations(M, K, seed=M)
    n, dt = rep(lambda: orc.act_quant(x))
    out["act_quant_M64_K17408"] = {"GB/s": round(n * (3 * M * K + 4 * M) / dt / 1e9, 4),
                                   "us_per_pass": round(1e6 * dt / n, 1)}
    R, K = 2048, synth.GATE_UP[1]
    nv_p, nv_s = synth.nvfp4_tensor_bytes(R, K, 0)
    div = np.array([2688.0], np.float32)
    pr = np.array([R], np.int64)
    n, dt = rep(lambda: orc.requant(nv_p, nv_s, div, pr, "mse"))
    by = R * K // 2 + R * K // 16 + R * K // 2 + R * K // 32
    out["requant_mse_2048_rows"] = {"GB/s": round(n * by / dt / 1e9, 4), "ms_per_pass": round(1e3 * dt / n, 1)}
    (N, K), M, C = synth.GATE_UP, 4096, 16
    x, wp, we = synth.prefill_case(M, N, K, 0)
    xq, xs = orc.act_quant(x)
    cols = (np.arange(C, dtype=np.int64) * N) // C
    im = np.repeat(np.arange(M, dtype=np.int64), C)
    inn = np.tile(cols, M)
    n, dt = rep(lambda: orc.mxfp4_linear_pairs(xq, xs, wp, we, im, inn))
    out["prefill_gate_up_M4096_16cols"] = {"TFLOP/s": round(n * 2.0 * M * C * K / dt / 1e12, 6),
                                           "ms_per_pass": round(1e3 * dt / n, 1)}
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, one pass of the fixed sample per step."""
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    sample = make_oracle_sample()
    for _ in range(args.warmup):
        oracle_pass(orc, sample)
    done, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        done += oracle_pass(orc, sample)
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    cores = orc.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle: e4m3 x e2m1 dequantized exactly, fp64 accumulate)",
        "data": "synthetic", "config": bench_config(1),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": SAMPLE_NOTE + "; one pass per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- GPU side

def chain_time(torch, dev, fns, reps=CHAIN_REPS):
    """Mean time (ms) of one call when `reps` calls run back to back, cycling over `fns` (calls
    on different weight copies, so the working set exceeds L2): the calls are captured in one
    CUDA graph, so consecutive library kernels overlap their set-up through programmatic
    dependent launch exactly as they do inside a decode step, and host launch cost is excluded."""
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
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (2 * reps)


def measure_fp8_peak(torch, dev):
    """Dense fp8 (e4m3) GEMM rate of this GPU: torch._scaled_mm (cuBLASLt) on 8192^3, best of 10
    event-timed calls after warm-up.  Returns TFLOP/s, or None if the call is not available."""
    try:
        n = 8192
        a = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev).to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.ones((), device=dev, dtype=torch.float32)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None


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
    assert step_bytes == STEP_BYTES
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

    def gemm(c, s, w=None, e=None):
        ws = c["ws"]
        st = clib.w4a8_mxfp4_linear(c["xq"].data_ptr(), c["xs"].data_ptr(), (c["w"] if w is None else w).data_ptr(),
                                    (c["e"] if e is None else e).data_ptr(), c["out"].data_ptr(), c["M"], c["N"],
                                    c["K"], None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(), s)
        if st:
            raise lib.W4A8Error("w4a8_mxfp4_linear", st)

    # eager warm-up (also makes the library's lazy per-device set-up happen outside capture)
    with torch.cuda.stream(stream):
        for c in calls:
            launch(c, stream.cuda_stream)
            clib.w4a8_act_quant(c["x"].data_ptr(), c["xq"].data_ptr(), c["xs"].data_ptr(), c["M"], c["K"],
                                stream.cuda_stream)
    stream.synchronize()
    lib.check_device_status(stream)  # a bounded wait that ran out means the kernels are broken

    # ---- step graph, and a second graph with timing events around every GEMM
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for c in calls:
            launch(c, stream.cuda_stream)
    evs = [(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in calls]
    ev_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ev_graph, stream=stream):
        for c, (a, b) in zip(calls, evs):
            clib.w4a8_act_quant(c["x"].data_ptr(), c["xq"].data_ptr(), c["xs"].data_ptr(), c["M"], c["K"],
                                stream.cuda_stream)
            a.record(stream)
            gemm(c, stream.cuda_stream)
            b.record(stream)
    # the step's eight GEMMs back to back (activations already quantized): the kernel's rate
    # as it runs inside the step
    cgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cgraph, stream=stream):
        for c in calls:
            gemm(c, stream.cuda_stream)

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

    # ---- the GEMM inside the step: the eight GEMMs chained in one graph
    reps = max(5, min(args.steps, 50))
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
    # ---- each GEMM bracketed by events (starts cold, without overlap with its neighbours)
    gemm_ms = [0.0] * len(calls)
    for _ in range(reps):
        ev_graph.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            gemm_ms[i] += a.elapsed_time(b) / reps
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    traffic = decode_traffic()
    step_us = 1e3 * ms_per_step
    # The GEMMs' time per step cannot exceed the step (which adds the activation quant); if the
    # separate chain measurement ever did, the whole step is charged to the GEMM instead.
    consistent = chain_us <= step_us
    gemm_us = chain_us if consistent else step_us
    ach = step_bytes / (gemm_us * 1e-6) / 1e9
    ach_cold = step_bytes / (sum(gemm_ms) * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": traffic, "algorithmic_bytes_per_launch": step_bytes / len(calls),
                "kernel": "decode-band MXFP4 GEMM (w4a8_mxfp4_linear, M<=64)", "peak_source": peak_src,
                "gemm_us_per_step": round(gemm_us, 2), "step_us": round(step_us, 2),
                "gemm_within_step": consistent,
                "timing": "the step's 8 GEMMs back to back in one CUDA graph (programmatic dependent launch "
                          "between them, as inside the step), CUDA events on the launching stream",
                "frac_cold": ach_cold / hbm,
                "cold_per_case_us": {f"{c['name']}_M{c['M']}": round(1e3 * g, 2) for c, g in zip(calls, gemm_ms)}}

    # ---- W4A8 decode per case, in the shared per-case protocol (the other formats: extras)
    decode_cases = {"protocol": f"graph of {CHAIN_REPS} back-to-back calls of one (shape, M) case cycling over "
                                "weight copies (> L2); per-call mean",
                    "w4a8": {}}
    for name, _ in SHAPES:
        cs = [c for c in calls if c["name"] == name]
        for c in cs:
            fns = [lambda c=c, o=o, s=stream: gemm(c, torch.cuda.current_stream().cuda_stream, o["w"], o["e"])
                   for o in cs]
            us = 1e3 * chain_time(torch, dev, fns)
            decode_cases["w4a8"][f"{name}_M{c['M']}"] = {"us": round(us, 2), "frac_of_hbm": round(
                c["bytes"] / (us * 1e-6) / 1e9 / hbm, 4)}

    # ---- e2e through the public API with host buffers
    h2d = sum(c["M"] * c["K"] * 2 for c in calls)
    d2h = sum(c["M"] * c["N"] * 2 for c in calls)
    pinned_x = [torch.from_numpy(c["x_host"].view(np.int16)).view(torch.bfloat16).pin_memory() for c in calls]
    pinned_o = [torch.empty((c["M"], c["N"]), dtype=torch.bfloat16).pin_memory() for c in calls]
    dev_x = [torch.empty((c["M"], c["K"]), dtype=torch.bfloat16, device=dev) for c in calls]
    dev_o = [torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device=dev) for c in calls]
    e2e_steps = max(3, min(args.steps, 20))

    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)

    # Before call i the compute stream waits for the input copies up to call E2E_WAITS[i]: the first
    # two calls' inputs, then (before the third call, long after they landed) all the others.  Every
    # wait on another stream breaks the programmatic-dependent-launch overlap between the two
    # kernels around it (~4 us), and every copy costs ~5 us of latency, so one wait per call
    # (241.6 us per step) and one wait for all inputs up front (261 us) both lose to this
    # (221-227 us; 200 us without any copies).
    E2E_WAITS = {0: 1, 2: len(calls) - 1}

    def e2e_step():
        # per call: pinned host x -> device, the public linear(), device out -> pinned host.  The
        # copies run on two more streams, one per direction (inputs first, in call order; each
        # output as soon as its GEMM is done), so they overlap the other calls' kernels and each
        # other, as a serving loop would pipeline them.
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        x_ready, o_ready = [], []
        with torch.cuda.stream(h2d_stream):
            for hx, xd in zip(pinned_x, dev_x):
                xd.copy_(hx, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d_stream)
                x_ready.append(ev)
        with torch.cuda.stream(stream):
            for i, (c, xd, od) in enumerate(zip(calls, dev_x, dev_o)):
                if i in E2E_WAITS:
                    stream.wait_event(x_ready[E2E_WAITS[i]])
                lib.linear(xd, c["w"], c["e"], out=od, workspace=c["lws"], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                o_ready.append(done)
        with torch.cuda.stream(d2h_stream):
            for ho, od, done in zip(pinned_o, dev_o, o_ready):
                d2h_stream.wait_event(done)
                ho.copy_(od, non_blocking=True)
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)

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
        "data": "synthetic", "config": bench_config(world),
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "per (shape, M): pinned host x -> device, binding.linear, device out -> pinned host, "
                        "copies on one stream per direction overlapping the kernels (the compute stream "
                        "waits for the first two inputs before the first call and for the rest before the "
                        "third); the step captured in a CUDA graph and replayed, wall-clock timed",
                "eager_value": e2e_eager_val},
        "gpu_launches": 2 * len(calls) * args.steps,
        "decode_cases": decode_cases,
    }
    del calls, graph, ev_graph, cgraph, g_e2e
    torch.cuda.empty_cache()
    if not args.no_extras and rank == 0:
        extras, prefill_roofline = run_extras(lib, dev, peaks)
        line["prefill_roofline"] = prefill_roofline
        for k in ("w4a4", "int4", "int5"):
            line["decode_cases"][k] = extras.pop("decode_" + k)
        line["extras"] = extras
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        sample = make_oracle_sample()
        b, t = oracle_timed(orc, sample, float(os.environ.get("W4A8_CPU_BASELINE_S", "10")))
        line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                                "sample": SAMPLE_NOTE + f"; whole passes for {t:.1f} s",
                                "other_steps": oracle_other(orc)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_extras(lib, dev, peaks):
    """The other hot-path kernels on their workloads (event-timed, working sets > L2).  Returns
    (extras, prefill_roofline); extras holds decode_w4a4 / decode_int4 / decode_int5 per-case
    figures in the shared decode protocol, lifted to the line's decode_cases by the caller."""
    import torch
    out = {}
    hbm = peaks["hbm_gbs"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def copies(nbytes):
        return max(3, -(-2 * l2 // nbytes))

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

    def dec_entry(us, nbytes):
        return {"us": round(us, 2), "frac_of_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4)}

    # ---- dense fp8 peak, measured now (the prefill roofline's denominator)
    fp8_meas = measure_fp8_peak(torch, dev)
    fp8_peak = fp8_meas if fp8_meas else 2.0 * peaks.get("bf16_tflops", 1900.0)
    fp8_src = ("measured: torch._scaled_mm e4m3 8192^3 (cuBLASLt), best of 10" if fp8_meas else
               "fallback: 2 x measured bf16 burst")

    # ---- MXFP4 prefill: TFLOP/s against the fp8 peak
    pf = {}
    for name, (N, K) in SHAPES + [("qkv", synth.QKV)]:
        w, e = synth.mxfp4_weights(N, K, 0, 118, 124)
        wds = [to_dev(w) for _ in range(3)]
        eds = [to_dev(e) for _ in range(3)]
        for M in (512, 2048, 4096):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.mxfp4_linear(xq, xs, a, b, out=o, workspace=ws) for a, b in zip(wds, eds)]
            ms = chain_time(torch, dev, fns, reps=12)
            tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            pf[f"{name}_M{M}"] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / fp8_peak, 4)}
        del wds, eds
    prefill_roofline = {"bound": "tensor", "unit": "TFLOP/s", "peak": round(fp8_peak, 1), "peak_source": fp8_src,
                        "kernel": "MXFP4 W4A8 GEMM, kind::mxf8f6f4 (fp8 rate)",
                        "timing": "graph of 12 calls over 3 weight copies, per-call mean",
                        "cases": {k: v for k, v in pf.items() if k.endswith("M4096")}}
    out["prefill"] = {"fp8_peak_tflops": fp8_peak, "peak_source": fp8_src, "cases": pf}

    # ---- per-token activation quant: 2MK bytes read, MK + 4M written
    aq = {}
    for M, K in ((1, 17408), (64, 17408), (4096, 5120), (4096, 17408)):
        n_copies = max(2, int(3 * 129e6 // (3 * M * K)) + 1) if M * K * 3 > 4e6 else 8
        xs_ = [torch.randn((M, K), device=dev).to(torch.bfloat16) for _ in range(min(n_copies, 8))]
        qs_ = [(torch.empty((M, K), dtype=torch.uint8, device=dev), torch.empty((M,), dtype=torch.float32, device=dev))
               for _ in xs_]
        fns = [lambda x=x, q=q: lib.act_quant(x, q[0], q[1]) for x, q in zip(xs_, qs_)]
        ms = chain_time(torch, dev, fns)
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
    out["requant_other_sources"] = {"bound": "hbm", "peak_gbs": hbm,
                                    "config": "gate_up N=34816 K=5120, one partition, mse rule, with error sums",
                                    "cases": other}
    del wb, o_p, o_e

    # ---- AutoRound int4 g128: decode (shared protocol), prefill TFLOP/s at M=4096
    dec_i4, i4 = {}, {}
    for name, (N, K) in SHAPES:
        qw, sc, _ = synth.int4_weights(N, K, 0)
        wb = N * K // 2 + N * K // 64
        nc = copies(wb)
        qws = [to_dev(qw) for _ in range(nc)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(nc)]
        for M in DECODE_M:
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.int4g128_linear(xq, xs, a, b, out=o, workspace=ws) for a, b in zip(qws, scs)]
            dec_i4[f"{name}_M{M}"] = dec_entry(1e3 * chain_time(torch, dev, fns), wb)
        M = 4096
        x = torch.randn((M, K), device=dev).to(torch.bfloat16)
        xq, xs = lib.act_quant(x)
        o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
        fns = [lambda a=a, b=b: lib.int4g128_linear(xq, xs, a, b, out=o, workspace=ws) for a, b in zip(qws[:3], scs[:3])]
        ms = chain_time(torch, dev, fns, reps=6)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        i4[f"{name}_M{M}"] = {"ms": round(ms, 3), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        prefill_roofline["cases"][f"int4_{name}_M{M}"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                                          "frac": round(tf / fp8_peak, 4)}
        del qws, scs
    out["decode_int4"] = dec_i4
    out["int4g128_prefill"] = {"bound": "tensor (fp8 peak)", "cases": i4}

    # ---- asymmetric int4 g128 (per-group, per-column zero points): decode GB/s, M = 1 and 64
    i4a = {}
    for name, (N, K) in SHAPES:
        qw, sc, _ = synth.int4_weights(N, K, 0)
        qz = to_dev(synth.int4_asym_zeros(N, K, 0))
        wb = N * K // 2 + N * K // 64 + (K // 128) * ((N + 7) // 8) * 4
        nc = copies(wb)
        qws = [to_dev(qw) for _ in range(nc)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(nc)]
        for M in (1, 64):
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int4_workspace_bytes(M, N, K), dev)
            fns = [lambda a=a, b=b: lib.int4g128_asym_linear(xq, xs, a, b, qz, out=o, workspace=ws)
                   for a, b in zip(qws, scs)]
            i4a[f"{name}_M{M}"] = dec_entry(1e3 * chain_time(torch, dev, fns), wb)
        del qws, scs, qz
    out["int4g128_asym_decode"] = {"bound": "hbm", "cases": i4a}

    # ---- int5 g128 (fifth-bit plane; zero point 16, or a byte per group and column): decode in
    # the shared protocol (zero point 16), with zero points at M = 1 and 64, prefill at M = 4096
    dec_i5, i5 = {}, {}
    for name, (N, K) in SHAPES:
        qw, qh, sc = synth.int5_weights(N, K, 0)
        z5 = to_dev(synth.int5_zeros(N, K, 0))
        wb = N * K // 2 + N * K // 8 + N * K // 64
        nc = copies(wb)
        qws = [to_dev(qw) for _ in range(nc)]
        qhs = [to_dev(qh) for _ in range(nc)]
        scs = [to_dev(sc).view(torch.float16) for _ in range(nc)]
        for M in DECODE_M:
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xq, xs = lib.act_quant(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.int5_workspace_bytes(M, N, K), dev)
            for tag, z in (("", None), ("_asym", z5)):
                if z is not None and M not in (1, 64):
                    continue
                fns = [lambda a=a, h=h, b=b, z=z: lib.int5g128_linear(xq, xs, a, h, b, z, out=o, workspace=ws)
                       for a, h, b in zip(qws, qhs, scs)]
                e = dec_entry(1e3 * chain_time(torch, dev, fns), wb + (0 if z is None else (K // 128) * N))
                if z is None:
                    dec_i5[f"{name}_M{M}"] = e
                else:
                    i5[f"{name}_M{M}_asym"] = e
        M = 4096
        x = torch.randn((M, K), device=dev).to(torch.bfloat16)
        xq, xs = lib.act_quant(x)
        o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = lib.make_workspace(lib.int5_workspace_bytes(M, N, K), dev)
        fns = [lambda a=a, h=h, b=b: lib.int5g128_linear(xq, xs, a, h, b, out=o, workspace=ws)
               for a, h, b in zip(qws[:3], qhs[:3], scs[:3])]
        ms = chain_time(torch, dev, fns, reps=6)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        i5[f"{name}_M{M}"] = {"ms": round(ms, 3), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / fp8_peak, 4)}
        prefill_roofline["cases"][f"int5_{name}_M{M}"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                                          "frac": round(tf / fp8_peak, 4)}
        del qws, qhs, scs, z5
    out["decode_int5"] = dec_i5
    out["int5g128"] = {"weight_bytes": "N*K*(1/2 + 1/8 + 2/128) (+ K/128*N zero bytes with zero points)",
                       "cases": i5}

    # ---- W4A4 (MXFP4 activations by the OCP rule): decode GEMM in the shared protocol, prefill
    # TFLOP/s, activation quant latency, and the relative error of W4A4 and W4A8 against the exact
    # product
    dec_a4, a4 = {}, {}
    for name, (N, K) in SHAPES:
        _, wp, we = synth.decode_case(1, N, K, 0)
        wb = N * K // 2 + N * K // 32
        nc = copies(wb)
        wps = [to_dev(wp) for _ in range(nc)]
        wes = [to_dev(we) for _ in range(nc)]
        for M in DECODE_M + [4096]:
            x = torch.randn((M, K), device=dev).to(torch.bfloat16)
            xa, xe = lib.act_quant_mxfp4(x)
            o = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = lib.make_workspace(lib.workspace_bytes(M, N, K), dev)
            if M < 4096:
                fns = [lambda a=a, b=b: lib.mxfp4_a4_linear(xa, xe, a, b, out=o, workspace=ws) for a, b in zip(wps, wes)]
                dec_a4[f"{name}_M{M}"] = dec_entry(1e3 * chain_time(torch, dev, fns), wb)
                if M in (1, 64):
                    ms = chain_time(torch, dev, [lambda: lib.act_quant_mxfp4(x, xa, xe)])
                    a4[f"act_quant_{name}_M{M}"] = {"us": round(ms * 1e3, 2)}
            else:
                fns = [lambda a=a, b=b: lib.mxfp4_a4_linear(xa, xe, a, b, out=o, workspace=ws)
                       for a, b in zip(wps[:3], wes[:3])]
                ms = chain_time(torch, dev, fns, reps=6)
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
    out["decode_w4a4"] = dec_a4
    out["w4a4"] = {"prefill_bound": "tensor (fp8 rate: e2m1 x e2m1 in kind::mxf8f6f4)", "cases": a4}
    return out, prefill_roofline


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other hot-path kernels (prefill, act quant, requant, int4, int5, W4A4)")
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
