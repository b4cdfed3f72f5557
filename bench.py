"""Benchmark of the SSD layer forward on GB300.

One step = one full SSD forward (chunk cumsums, diagonal blocks, chunk states, inter-chunk
state pass, off-diagonal outputs and the D skip) over the long-sequence workload b=1,
T=16384, H=80, P=64, N=128, G=1, chunk 256, bf16 x/B/C with fp32 dt/A/D. Prints ONE JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Other workloads (--workload): the forward on the other layer shapes (long_n64, long_n256, m2_130m,
m2_2p7b, varlen, long_n128_dtscaled), the one-token recurrent step (decode_2p7b,
decode_2p7b_bf16state) and the block's output gate and normalization (gated_norm_long).

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of
the same workload (the slow baseline the GPU path is checked against).
Multi-GPU (torchrun): every rank runs its own copy of the workload (independent
problems, no collective on the data path); value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSD fwd tokens/s and % of bf16 tensor/HBM roofline, T=2K–16K, N=128"
DECODE_METRIC = "SSD recurrent step tokens/s (one token per carried state) and % of HBM roofline"
NORM_METRIC = "output gate and RMSNorm tokens/s (y * silu(z), normalized per group, scaled) and % of HBM roofline"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# seconds of untimed steps before the timed loop, with the clock sampler running
CLOCK_SOAK_S = 1.2

# DRAM bytes (read + write) per launch of the dominant kernel from one ncu capture, keyed by
# workload, with a stamp of the kernel's sources at capture time. A stamp that no longer
# matches the sources means the kernel changed since: the traffic is then reported as null.
KERNEL_SOURCES = {
    "ssd_fused_kernel": ("mamba_ssd_layer_gb300/csrc/ssd_fused.cu", "mamba_ssd_layer_gb300/csrc/ptx.cuh",
                         "mamba_ssd_layer_gb300/csrc/ssd_internal.cuh"),
    "ssd_decode_kernel": ("mamba_ssd_layer_gb300/csrc/ssd_decode.cu",),
    "gated_rmsnorm_kernel": ("mamba_ssd_layer_gb300/csrc/ssd_norm.cu", "mamba_ssd_layer_gb300/csrc/ssd_norm.cuh",
                             "mamba_ssd_layer_gb300/csrc/ptx.cuh"),
}
NCU_TRAFFIC = {
    "long_n128": {"kernel": "ssd_fused_kernel", "bytes": 216363008 + 147446528, "stamp": "20624a49ebfbc082"},
    "long_n64": {"kernel": "ssd_fused_kernel", "bytes": 201585920 + 138726144, "stamp": "20624a49ebfbc082"},
    # N = 256: the mean of the two launches of one pass (one per 128-column half of the state)
    "long_n256": {"kernel": "ssd_fused_kernel", "bytes": 294373376 + 143089792, "stamp": "20624a49ebfbc082"},
    "long_n128_dtscaled": {"kernel": "ssd_fused_kernel", "bytes": 207358208 + 147891200, "stamp": "20624a49ebfbc082"},
    # y (50 MB) largely still in L2 when the launch ends
    "m2_130m": {"kernel": "ssd_fused_kernel", "bytes": 60483328 + 12647936, "stamp": "20624a49ebfbc082"},
    "m2_2p7b": {"kernel": "ssd_fused_kernel", "bytes": 214793216 + 152965376, "stamp": "20624a49ebfbc082"},
    "varlen": {"kernel": "ssd_fused_kernel", "bytes": 178148096 + 120641024, "stamp": "20624a49ebfbc082"},
    # recurrent step: part of the state's write-back is still in L2 when the launch ends
    "decode_2p7b": {"kernel": "ssd_decode_kernel", "bytes": 168496384 + 117444864, "stamp": "e82f933ea29a60b6"},
    "decode_2p7b_bf16state": {"kernel": "ssd_decode_kernel", "bytes": 84610304 + 34867712,
                              "stamp": "e82f933ea29a60b6"},
    # gate and normalization: part of out is still in L2 when the launch ends
    "gated_norm_long": {"kernel": "gated_rmsnorm_kernel", "bytes": 335803392 + 133026048, "stamp": "ec00523922835394"},
}


def kernel_source_stamp(kernel: str = "ssd_fused_kernel") -> str:
    """Hash of the kernel's code: comments and blank lines are left out, so that only a change of the
    code itself invalidates a recorded measurement."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None or rec["kernel"] != kernel or rec["stamp"] != kernel_source_stamp(kernel):
        return None
    return rec["bytes"]


def reduce_over_ranks(ms: float, tokens_per_rank: int, steps: int, world: int, device):
    """Slowest rank's timed region (max over ranks) and the whole-job tokens/s it gives."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_rank * steps / (ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(PEAKS_FALLBACK), "fallback"


def algorithmic_bytes(w, batch_rows, nseq) -> int:
    """Bytes the forward must move at minimum: x in, y out (bf16), B, C in (bf16), dt in (fp32),
    A, D, and the initial/final states when used (fp32)."""
    T, H, P, N, G = batch_rows, w.nheads, w.headdim, w.dstate, w.ngroups
    e = 2 if w.dtype == "bf16" else 4
    by = 2 * T * H * P * e + 2 * T * G * N * e + 4 * T * H + 8 * H
    by += nseq * H * P * N * 4 * (2 if w.init_state else 1)
    return int(by)


def decode_algorithmic_bytes(w) -> int:
    """Bytes one recurrent step must move: the state in and out (fp32 or bf16), x in and y out, B and
    C, dt, A and D."""
    b, H, P, N, G = w.batch, w.nheads, w.headdim, w.dstate, w.ngroups
    e = 2 if w.dtype == "bf16" else 4
    es = 2 if w.state_dtype == "bf16" else 4
    return int(2 * b * H * P * N * es + 2 * b * H * P * e + 2 * b * G * N * e + 4 * b * H + 8 * H)


def norm_algorithmic_bytes(w) -> int:
    """Bytes the gate and normalization must move: y and z in, out back (bf16), the fp32 weight."""
    C = w.nheads * w.headdim
    return int(3 * w.batch * w.seqlen * C * 2 + C * 4)


def algorithmic_flops(w, batch_rows) -> int:
    """Useful FLOPs of the chunked algorithm per the pages' cost model: causal C B^T per group
    (Q+1)N/2 MACs per token, masked (L o CB^T) X per head (Q+1)P/2 MACs, chunk state and
    C.state per head N*P MACs each -> 2 FLOP per MAC."""
    Q, H, P, N, G = w.chunk, w.nheads, w.headdim, w.dstate, w.ngroups
    macs_per_token = G * (Q + 1) * N / 2 + H * ((Q + 1) * P / 2 + 2 * N * P)
    return int(2 * macs_per_token * batch_rows)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""
        else:
            self.out = ""

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen; with (t0, t1) (time.time() around the
        timed region) only the samples taken inside it count, when there are any."""
        import datetime
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        if t0 is not None and any(t0 <= r[0] <= t1 for r in rows):
            rows = [r for r in rows if t0 <= r[0] <= t1]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, s, m, flags in rows:
            sm.append(s)
            mx.append(m)
            for nm, v in zip(names, flags):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def soak(step, torch, seconds: float = None) -> float:
    """Run the step, untimed, for at least `seconds` (CLOCK_SOAK_S): the clock record then covers the
    GPU under this load (the sampler polls every 100 ms), however short the timed loop. Returns the
    wall time it started."""
    seconds = CLOCK_SOAK_S if seconds is None else seconds
    t0 = time.time()
    i = 0
    while time.time() - t0 < seconds:
        for _ in range(16):
            step(i)
            i += 1
        torch.cuda.synchronize()
    return t0


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def decode_sample(w, rows: int):
    """The first `rows` carried states of a recurrent-step workload, as (state, x, dt, A, B, C, D)."""
    from mamba_ssd_layer_gb300.inputs import make_inputs
    d = make_inputs(w)
    r = slice(0, min(rows, w.batch))
    return (d["initial_state"][r], d["x"][r, 0], d["dt"][r, 0], d["A"], d["B"][r, 0], d["C"][r, 0], d["D"])


def run_reference_decode(args, w):
    """The oracle's recurrent step on the host, bounded: each step runs a sample of the carried states."""
    import oracle
    rows = max(1, min(w.batch, args.ref_tokens // 1024))
    smp = decode_sample(w, rows)
    oracle.ssd_decode_step(*smp)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ssd_decode_step(*smp)
        times.append(time.perf_counter() - t0)
    tot = float(np.sum(times))
    val = rows * args.steps / tot
    sample = f"{rows} of {w.batch} carried states, all {w.nheads} heads, per step"
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": decode_config(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def decode_config(w):
    sb = w.batch * w.nheads * w.headdim * w.dstate * (2 if w.state_dtype == "bf16" else 4)
    return {"workload": w.name, "batch": w.batch, "nheads": w.nheads, "headdim": w.headdim, "dstate": w.dstate,
            "ngroups": w.ngroups, "state_dtype": w.state_dtype, "parallelism": "replicas",
            "l2": f"inputs larger than L2 (two {w.state_dtype} state buffers of ~{sb / 1e6:.0f} MB each, "
                  "read and written in turn)"}


def decode_cpu_baseline(w, min_seconds: float = 10.0, max_runs: int = 5000):
    """The oracle's recurrent step as it stands (numpy, one core), on 8 of the carried states,
    repeated for about `min_seconds`."""
    import oracle
    rows = min(8, w.batch)
    smp = decode_sample(w, rows)
    runs, t0 = 0, time.perf_counter()
    while runs < max_runs and (runs == 0 or time.perf_counter() - t0 < min_seconds):
        oracle.ssd_decode_step(*smp)
        runs += 1
    dt = time.perf_counter() - t0
    return {"value": rows * runs / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {w.batch} carried states (all {w.nheads} heads), {runs} runs in {dt:.1f} s"}


def run_decode(args, w):
    """Recurrent steps on the GPU: each step advances every carried state by one token."""
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from mamba_ssd_layer_gb300 import binding as bd
    from mamba_ssd_layer_gb300 import ssd_decode_step, ssd_decode_step_host
    from mamba_ssd_layer_gb300.inputs import make_inputs

    d = make_inputs(w)
    host = {"x": d["x"][:, 0], "dt": d["dt"][:, 0], "A": d["A"], "B": d["B"][:, 0], "C": d["C"][:, 0], "D": d["D"],
            "state": d["initial_state"]}
    t = {k: torch.from_numpy(np.ascontiguousarray(host[k])).to(dev, torch.bfloat16) for k in ("x", "B", "C")}
    for k in ("dt", "A", "D"):
        t[k] = torch.from_numpy(np.ascontiguousarray(host[k])).to(dev, torch.float32)
    sdt = torch.bfloat16 if w.state_dtype == "bf16" else torch.float32
    states = [torch.from_numpy(host["state"]).to(dev, sdt), torch.empty(host["state"].shape, dtype=sdt, device=dev)]
    y = torch.empty_like(t["x"])
    stream = torch.cuda.current_stream(dev)

    def step(i):
        ssd_decode_step(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], states[i % 2], states[(i + 1) % 2], y,
                        stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        soak0 = soak(step, torch)
        bd.profile_enable(True)
        wall0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        wall1 = time.time()
    bd.profile_enable(False)
    kern_ms, kern_n = bd.profile_read()
    launches = bd.profile_kernel_launches()
    kernel = bd.profile_kernel_name()
    ms = ev0.elapsed_time(ev1)
    ms, value = reduce_over_ranks(ms, w.batch, args.steps, world, dev)
    ms_per_step = ms / args.steps

    # end to end through the host entry point: pinned inputs and state in, y and the state out
    hx = {k: torch.from_numpy(np.ascontiguousarray(host[k])).to(torch.bfloat16).pin_memory() for k in ("x", "B", "C")}
    hf = {k: torch.from_numpy(np.ascontiguousarray(host[k])).pin_memory() for k in ("dt", "A", "D")}
    hf["state"] = torch.from_numpy(np.ascontiguousarray(host["state"])).to(sdt).pin_memory()
    hy = torch.empty_like(hx["x"]).pin_memory()
    devbuf = torch.empty(int(bd.load_library().ssd_decode_host_buffer_size(
        bd._shape(w.batch, 1, w.nheads, w.headdim, w.dstate, w.ngroups), bd.SSD_BF16)), dtype=torch.uint8, device=dev)

    def e2e_step():
        ssd_decode_step_host(hx["x"], hf["dt"], hf["A"], hx["B"], hx["C"], hf["D"], hf["state"], hf["state"], hy,
                             device_buffer=devbuf, stream=stream)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    h2d = sum(v.numel() * v.element_size() for v in list(hx.values()) + list(hf.values()))
    d2h = hy.numel() * 2 + hf["state"].numel() * hf["state"].element_size()

    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    alg_bytes = decode_algorithmic_bytes(w)
    kern_avg_ms = kern_ms / max(kern_n, 1)
    achieved = alg_bytes / (kern_avg_ms / 1e3) / 1e9 if kern_n else None
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": decode_config(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if achieved else None,
                     "traffic": measured_traffic(w.name, kernel), "peak_source": src, "kernel": kernel,
                     "kernel_ms": kern_avg_ms, "alg_bytes_per_launch": alg_bytes, "launches_per_step": 1.0,
                     "step_frac": alg_bytes / (ms_per_step / 1e3) / 1e9 / hbm},
        "e2e": {"value": world * w.batch * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches,
        "clocks": clk.summary(soak0, wall1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def norm_config(w):
    mb = w.batch * w.seqlen * w.nheads * w.headdim * 2 / 1e6
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "groups": w.norm_groups, "gated": True, "parallelism": "replicas",
            "l2": f"inputs larger than L2 (two rotating sets of y, z and out, ~{3 * mb:.0f} MB each)",
            "clock_soak_s": CLOCK_SOAK_S}


def norm_sample_rows(budget_tokens: int) -> int:
    return max(1, min(2048, budget_tokens // 8))


def norm_cpu_baseline(w, budget_tokens: int, min_seconds: float = 10.0, max_runs: int = 500):
    """The oracle's gate and normalization as it stands (numpy, one core) on a sample of tokens of the
    workload's shape, repeated for about `min_seconds`."""
    import oracle
    from mamba_ssd_layer_gb300.inputs import make_norm_inputs
    rows = norm_sample_rows(budget_tokens)
    d = make_norm_inputs(w, rows=rows)
    runs, t0 = 0, time.perf_counter()
    while runs < max_runs and (runs == 0 or time.perf_counter() - t0 < min_seconds):
        oracle.gated_rmsnorm(d["y"], d["z"], d["weight"], eps=1e-5, groups=w.norm_groups)
        runs += 1
    dt = time.perf_counter() - t0
    return {"value": rows * runs / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {w.batch * w.seqlen} tokens (all {w.nheads * w.headdim} channels), "
                      f"{runs} runs in {dt:.1f} s"}


def run_reference_norm(args, w):
    """The oracle's gate and normalization on the host, bounded: each step runs a sample of the tokens."""
    import oracle
    from mamba_ssd_layer_gb300.inputs import make_norm_inputs
    rows = norm_sample_rows(args.ref_tokens)
    d = make_norm_inputs(w, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.gated_rmsnorm(d["y"], d["z"], d["weight"], eps=1e-5, groups=w.norm_groups)
        times.append(time.perf_counter() - t0)
    tot = float(np.sum(times))
    val = rows * args.steps / tot
    sample = f"{rows} of {w.batch * w.seqlen} tokens, all {w.nheads * w.headdim} channels, per step"
    line = {"impl": "reference", "metric": NORM_METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": norm_config(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_norm(args, w):
    """The output gate and normalization on the GPU: each step normalizes every token of the workload."""
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    from mamba_ssd_layer_gb300 import binding as bd
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm, ssd_gated_rmsnorm_host
    from mamba_ssd_layer_gb300.inputs import make_norm_inputs

    d = make_norm_inputs(w)
    rows = w.batch * w.seqlen
    hy = torch.from_numpy(d["y"]).to(torch.bfloat16).pin_memory()
    hz = torch.from_numpy(d["z"]).to(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(d["weight"]).pin_memory()
    wt = hw.to(dev)
    # two rotating sets of y, z and out: the previous step's data is out of L2
    sets = [(hy.to(dev), hz.to(dev), torch.empty(hy.shape, dtype=torch.bfloat16, device=dev)) for _ in range(2)]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        y, z, out = sets[i % 2]
        ssd_gated_rmsnorm(y, z, wt, eps=1e-5, groups=w.norm_groups, out=out, stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        soak0 = soak(step, torch)
        bd.profile_enable(True)
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        wall1 = time.time()
    bd.profile_enable(False)
    kern_ms, kern_n = bd.profile_read()
    launches = bd.profile_kernel_launches()
    kernel = bd.profile_kernel_name()
    ms = ev0.elapsed_time(ev1)
    ms, value = reduce_over_ranks(ms, rows, args.steps, world, dev)
    ms_per_step = ms / args.steps

    # end to end through the host entry point: pinned y, z and weight in, out back
    hout = torch.empty_like(hy).pin_memory()
    import ctypes
    need = int(bd.load_library().ssd_gated_rmsnorm_host_buffer_size(
        ctypes.byref(bd._shape(w.batch, w.seqlen, w.nheads, w.headdim, 1, 1)), 1))
    devbuf = torch.empty(need, dtype=torch.uint8, device=dev)

    def e2e_step():
        ssd_gated_rmsnorm_host(hy, hz, hw, eps=1e-5, groups=w.norm_groups, out=hout, device_buffer=devbuf,
                               stream=stream)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    h2d = hy.numel() * 2 + hz.numel() * 2 + hw.numel() * 4
    d2h = hout.numel() * 2

    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    alg_bytes = norm_algorithmic_bytes(w)
    kern_avg_ms = kern_ms / max(kern_n, 1)
    achieved = alg_bytes / (kern_avg_ms / 1e3) / 1e9 if kern_n else None
    line = {
        "metric": NORM_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": norm_config(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if achieved else None,
                     "traffic": measured_traffic(w.name, kernel), "peak_source": src, "kernel": kernel,
                     "kernel_ms": kern_avg_ms, "alg_bytes_per_launch": alg_bytes, "launches_per_step": 1.0,
                     "step_frac": alg_bytes / (ms_per_step / 1e3) / 1e9 / hbm},
        "e2e": {"value": world * rows * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches,
        "clocks": clk.summary(soak0, wall1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = norm_cpu_baseline(w, args.ref_tokens)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, w):
    """The oracle on the host cores, bounded: each step runs a sample of the workload."""
    import oracle
    from mamba_ssd_layer_gb300.inputs import make_inputs, small_variant
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    if w.norm_groups:
        run_reference_norm(args, w)
        return
    if w.seqlen == 1:
        run_reference_decode(args, w)
        return
    # sample: every head, the first `tokens` tokens of the sequence (~several seconds per step)
    tokens = min(w.seqlen, args.ref_tokens)
    ws = small_variant(w, seqlen=tokens, nheads=w.nheads, batch=1) if not w.varlen_total else \
        small_variant(w, seqlen=tokens, nheads=w.nheads)
    d = make_inputs(ws)
    threads = oracle.default_threads()
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle.ssd_recurrence(d["x"][:, :64], d["dt"][:, :64], d["A"], d["B"][:, :64], d["C"][:, :64], d["D"])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ssd_recurrence(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_state"],
                              d["cu_seqlens"], nthreads=threads, scale_x_by_dt=w.scale_x_by_dt)
        times.append(time.perf_counter() - t0)
    tot = float(np.sum(times))
    val = tokens * args.steps / tot
    sample = f"{tokens} of {w.seqlen} tokens, all {w.nheads} heads, per step"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w):
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk, "scale_x_by_dt": w.scale_x_by_dt,
            # the bf16 path works on 128-token tiles whatever `chunk` is (the result does not depend on it)
            "kernel_tile": 128,
            "parallelism": "replicas",
            "l2": "inputs larger than L2 (2 rotating input sets of ~350 MB each)",
            "clock_soak_s": CLOCK_SOAK_S}


def cpu_baseline(w, budget_tokens: int, min_seconds: float = 10.0, max_runs: int = 50):
    """The oracle as it stands on the host cores: one sequence of the workload (all heads),
    run repeatedly until about `min_seconds` of CPU work has been timed."""
    import oracle
    from mamba_ssd_layer_gb300.inputs import make_inputs, small_variant
    tokens = min(w.seqlen, budget_tokens)
    d = make_inputs(small_variant(w, seqlen=tokens, nheads=w.nheads, batch=1))
    threads = oracle.default_threads()
    runs, t0 = 0, time.perf_counter()
    while runs < max_runs and (runs == 0 or time.perf_counter() - t0 < min_seconds):
        oracle.ssd_recurrence(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_state"],
                              d["cu_seqlens"], nthreads=threads, scale_x_by_dt=w.scale_x_by_dt)
        runs += 1
    dt = time.perf_counter() - t0
    return {"value": tokens * runs / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{tokens} of {w.seqlen * w.batch} tokens (one sequence, all {w.nheads} heads), "
                      f"{runs} runs in {dt:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_n128")
    ap.add_argument("--ref-tokens", type=int, default=16384)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return
    if w.seqlen == 1:
        run_decode(args, w)
        return
    if w.norm_groups:
        run_norm(args, w)
        return

    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    from mamba_ssd_layer_gb300 import binding as bd
    from mamba_ssd_layer_gb300 import ssd_forward, ssd_forward_host

    d = make_inputs(w)
    rows = d["x"].shape[0] * d["x"].shape[1]
    nseq = (len(d["cu_seqlens"]) - 1) if d["cu_seqlens"] is not None else d["x"].shape[0]

    def dev_inputs():
        t = {}
        for k in ("x", "B", "C"):
            t[k] = torch.from_numpy(d[k]).to(dev, torch.bfloat16)
        for k in ("dt", "A", "D"):
            t[k] = torch.from_numpy(d[k]).to(dev, torch.float32)
        t["init"] = None if d["initial_state"] is None else torch.from_numpy(d["initial_state"]).to(dev)
        t["cu"] = None if d["cu_seqlens"] is None else torch.from_numpy(d["cu_seqlens"]).to(dev)
        t["y"] = torch.empty_like(t["x"])
        t["final"] = torch.empty((nseq, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
        return t

    sets = [dev_inputs(), dev_inputs()]          # two rotating sets: the previous step's data is out of L2
    ws_bytes = bd.ssd_workspace_size(1 if d["cu_seqlens"] is not None else d["x"].shape[0], d["x"].shape[1],
                                     w.nheads, w.headdim, w.dstate, w.ngroups, bd.SSD_BF16, w.chunk,
                                     nseq if d["cu_seqlens"] is not None else 0)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        t = sets[i % 2]
        ssd_forward(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=w.chunk, initial_state=t["init"],
                    cu_seqlens=t["cu"], y=t["y"], final_state=t["final"], workspace=workspace, stream=stream,
                    scale_x_by_dt=w.scale_x_by_dt)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    status = bd.ssd_status(workspace)
    if status != bd.SSD_OK:
        raise RuntimeError(f"device status after warm-up: {bd.ssd_status_string(status)}")

    if world > 1:
        torch.distributed.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        soak0 = soak(step, torch)
        bd.profile_enable(True)
        wall0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        wall1 = time.time()
    bd.profile_enable(False)
    kern_ms, kern_n = bd.profile_read()
    ms = ev0.elapsed_time(ev1)
    status = bd.ssd_status(workspace)
    if status != bd.SSD_OK:
        raise RuntimeError(f"device status after timing: {bd.ssd_status_string(status)}")
    launches = bd.profile_kernel_launches()
    kernel = bd.profile_kernel_name()
    ms, value = reduce_over_ranks(ms, rows, args.steps, world, dev)
    ms_per_step = ms / args.steps

    # end to end through the host entry point: pinned inputs in, y and final states out
    hx = {k: torch.from_numpy(d[k]).to(torch.bfloat16).pin_memory() for k in ("x", "B", "C")}
    hf = {k: torch.from_numpy(d[k]).pin_memory() for k in ("dt", "A", "D")}
    hinit = None if d["initial_state"] is None else torch.from_numpy(d["initial_state"]).pin_memory()
    hcu = None if d["cu_seqlens"] is None else torch.from_numpy(d["cu_seqlens"])
    hy = torch.empty_like(hx["x"]).pin_memory()
    hfin = torch.empty((nseq, w.nheads, w.headdim, w.dstate), dtype=torch.float32).pin_memory()
    need = bd.load_library().ssd_host_buffer_size
    devbuf = None

    def e2e_step():
        nonlocal devbuf
        _, _ = ssd_forward_host(hx["x"], hf["dt"], hf["A"], hx["B"], hx["C"], hf["D"], chunk=w.chunk,
                                initial_state=hinit, cu_seqlens=hcu, y=hy, final_state=hfin,
                                device_buffer=devbuf, stream=stream, scale_x_by_dt=w.scale_x_by_dt)

    import ctypes
    shp = bd._shape(1 if hcu is not None else d["x"].shape[0], d["x"].shape[1], w.nheads, w.headdim, w.dstate,
                    w.ngroups)
    devbuf = torch.empty(int(need(ctypes.byref(shp), bd.SSD_BF16, w.chunk, nseq if hcu is not None else 0)),
                         dtype=torch.uint8, device=dev)
    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    h2d = sum(t.numel() * t.element_size() for t in (hx["x"], hx["B"], hx["C"], hf["dt"], hf["A"], hf["D"]))
    h2d += 0 if hinit is None else hinit.numel() * 4
    h2d += 0 if hcu is None else hcu.numel() * 4
    d2h = hy.numel() * 2 + hfin.numel() * 4

    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    alg_bytes = algorithmic_bytes(w, rows, nseq)
    alg_flops = algorithmic_flops(w, rows)
    kern_avg_ms = kern_ms / max(kern_n, 1)
    # roofline of the dominant kernel: the algorithmic bytes of the whole pass over the time of its
    # launches in one pass (N = 256 takes two launches, one per 128-column half of the state, and
    # each is charged half of the pass's bytes)
    launches_per_step = kern_n / args.steps if kern_n else 1
    alg_bytes_launch = alg_bytes / launches_per_step
    achieved = alg_bytes_launch / (kern_avg_ms / 1e3) / 1e9 if kern_n else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(w),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if achieved else None,
                     "traffic": measured_traffic(w.name, kernel),
                     "peak_source": src, "kernel": kernel, "kernel_ms": kern_avg_ms,
                     "alg_bytes_per_launch": int(alg_bytes_launch), "launches_per_step": launches_per_step,
                     "step_frac": alg_bytes / (ms_per_step / 1e3) / 1e9 / hbm},
        "tflops": alg_flops / (ms_per_step / 1e3) / 1e12,
        "e2e": {"value": world * rows * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches,
        "clocks": clk.summary(soak0, wall1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.ref_tokens)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
