"""The bench's multi-rank host logic on CPU: the max-over-ranks reduction of the timed
region over a two-rank gloo group, and the reference arm under torchrun (rank 0 prints
the one JSON line, the other rank exits without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms, value = bench.reduce_over_ranks(10.0 + 5.0 * rank, 1000, 4, world, "cpu")
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_takes_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got["ms"] == 15.0
        assert got["value"] == pytest.approx(world * 1000 * 4 / 0.015)


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.reduce_over_ranks(20.0, 500, 2, 1, "cpu")
    assert ms == 20.0 and value == pytest.approx(500 * 2 / 0.02)


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "0", "--workload", "fp32_tiny", "--ref-tokens", "64"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
