"""The bench's host-side arithmetic and its oracle arms, on CPU: the algorithmic bytes each roofline
divides by (written out from the tensors a step must move), the gate and normalization workload's input
recipe, and the reference arm of that workload printing one well-formed line."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_norm_inputs  # noqa: E402


def test_forward_algorithmic_bytes():
    # x in and y out (bf16), B and C (bf16), dt (fp32), A and D (fp32), the final state (fp32)
    w = WORKLOADS["long_n128"]
    T, H, P, N = 16384, 80, 64, 128
    expect = 2 * T * H * P * 2 + 2 * T * N * 2 + 4 * T * H + 8 * H + H * P * N * 4
    assert expect == 351_797_888
    assert bench.algorithmic_bytes(w, T, 1) == expect
    # with an initial state the state is read as well as written
    w2 = WORKLOADS["m2_2p7b"]
    rows = w2.batch * w2.seqlen
    assert bench.algorithmic_bytes(w2, rows, w2.batch) - bench.algorithmic_bytes(w2.with_(init_state=False), rows, w2.batch) \
        == w2.batch * w2.nheads * w2.headdim * w2.dstate * 4


def test_recurrent_step_algorithmic_bytes():
    # the carried state in and out, plus one token's x, y, B, C, dt and the per-head A, D
    b, H, P, N = 64, 80, 64, 128
    rest = 2 * b * H * P * 2 + 2 * b * N * 2 + 4 * b * H + 8 * H
    assert bench.decode_algorithmic_bytes(WORKLOADS["decode_2p7b"]) == 2 * b * H * P * N * 4 + rest
    assert bench.decode_algorithmic_bytes(WORKLOADS["decode_2p7b_bf16state"]) == 2 * b * H * P * N * 2 + rest


def test_gate_and_normalization_bytes_and_inputs():
    w = WORKLOADS["gated_norm_long"]
    C = w.nheads * w.headdim
    # y and z in, out back (bf16), the fp32 weight once
    assert bench.norm_algorithmic_bytes(w) == 3 * 16384 * C * 2 + C * 4 == 503_336_960
    d = make_norm_inputs(w, rows=64)
    assert d["y"].shape == d["z"].shape == (1, 64, 80, 64) and d["weight"].shape == (C,)
    # bf16-representable values (the low 16 bits of each fp32 are zero), the weight within [0.5, 1.5)
    for k in ("y", "z"):
        assert not (d[k].view(np.uint32) & 0xFFFF).any()
    assert d["weight"].min() >= 0.5 and d["weight"].max() < 1.5
    # the same seed draws the same values
    assert np.array_equal(make_norm_inputs(w, rows=64)["y"], d["y"])


def test_gate_and_normalization_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "gated_norm_long",
                        "--steps", "1", "--warmup", "0", "--ref-tokens", "2048"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["config"]["workload"] == "gated_norm_long" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
