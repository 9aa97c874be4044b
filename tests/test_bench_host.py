"""Host-side logic of bench.py, on CPU: the multi-rank aggregation (gloo, world size 2) and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    value, ms = bench.aggregate(elapsed[rank], 1000, 4, world, dist, "cpu")
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    world, port = 2, _free_port()
    elapsed = [10.0, 12.5]  # ms per rank for 4 steps of 1000 bytes each
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, elapsed, out), nprocs=world, join=True)
    for r in range(world):
        value, ms = out[r]
        assert ms == 12.5                      # the slowest rank sets the job time
        assert value == pytest.approx(2 * 1000 * 4 / 12.5e-3 / 1e9)  # all ranks' bytes


def test_aggregate_single_rank():
    import bench
    value, ms = bench.aggregate(20.0, 500, 2, 1)
    assert ms == 20.0 and value == pytest.approx(500 * 2 / 20e-3 / 1e9)


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == "GB/s"
    import bench
    # the same workload description as the GPU arm's line, so the two lines compare
    assert line["config"] == bench.bench_config(1)


def test_oracle_sample_is_fixed():
    """Both arms time the same fixed sample: its bytes per pass do not depend on timing."""
    import bench
    import oracle as orc
    orc.build()
    sample = bench.make_oracle_sample()
    assert len(sample) == 8
    per_pass = sum(s[-1] for s in sample)
    assert per_pass == bench.SAMPLE_COLS * sum(K // 2 + K // 32 for _, (N, K) in bench.SHAPES for _ in bench.DECODE_M)
    assert bench.oracle_pass(orc, sample) == per_pass
