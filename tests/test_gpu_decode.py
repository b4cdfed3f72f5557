"""GPU parity of the one-token recurrent step (ssd_decode_step, through the C ABI) against
the oracle's step on the same seeded inputs. Tolerances (normwise max|out - ref| / max|ref|):
1e-4 for fp32 storage, 1e-2 for bf16 storage; the state is fp32 on both paths."""
import numpy as np
import pytest

import oracle
from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs
from ssd_util import TOL, normwise, run_gpu

pytestmark = pytest.mark.gpu


def decode_inputs(batch, H, P, N, G, dtype, seed):
    w = WORKLOADS["decode_2p7b"].with_(batch=batch, nheads=H, headdim=P, dstate=N, ngroups=G, dtype=dtype, seed=seed)
    d = make_inputs(w)
    return dict(x=d["x"][:, 0], dt=d["dt"][:, 0], A=d["A"], B=d["B"][:, 0], C=d["C"][:, 0], D=d["D"],
                state=d["initial_state"])


def to_dev(d, dtype):
    import torch
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda().to(tdt) for k in ("x", "B", "C")}
    for k in ("dt", "A", "D", "state"):
        if k in d:
            t[k] = torch.from_numpy(np.ascontiguousarray(d[k])).cuda().float()
    return t


def gpu_step(d, dtype, use_D=True, in_place=False, scale_x_by_dt=False):
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step
    t = to_dev(d, dtype)
    new = t["state"] if in_place else torch.empty_like(t["state"])
    y, s = ssd_decode_step(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"] if use_D else None, t["state"], new,
                           scale_x_by_dt=scale_x_by_dt)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), s.cpu().numpy().astype(np.float64)


CASES = [  # batch, H, P, N, G, dtype
    (3, 4, 64, 128, 1, "bf16"), (5, 6, 64, 256, 2, "bf16"), (2, 4, 64, 64, 1, "bf16"),
    (3, 2, 16, 16, 1, "f32"), (2, 6, 12, 20, 3, "f32"), (1, 2, 256, 256, 1, "f32"),
    (7, 3, 33, 36, 3, "f32"), (2, 2, 5, 132, 1, "f32"), (4, 8, 64, 128, 4, "bf16"), (1, 1, 1, 4, 1, "f32"),
    (2, 3, 200, 128, 1, "f32"),   # several row blocks per head, the last one partial
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}H{c[1]}P{c[2]}N{c[3]}G{c[4]}{c[5]}" for c in CASES])
def test_decode_step_matches_oracle(case):
    batch, H, P, N, G, dtype = case
    d = decode_inputs(batch, H, P, N, G, dtype, seed=300 + N + P)
    y, s = gpu_step(d, dtype)
    yr, sr = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    ey, es = normwise(y, yr), normwise(s, sr)
    print(f"[decode parity] {case} y_err={ey:.3e} state_err={es:.3e}")
    assert ey <= TOL[dtype] and es <= TOL[dtype]
    # the state is fp32 arithmetic on both sides: far inside the bar
    assert es <= 1e-5


def test_decode_in_place_equals_out_of_place_and_no_skip():
    d = decode_inputs(4, 6, 64, 128, 2, "bf16", seed=311)
    y1, s1 = gpu_step(d, "bf16", in_place=False)
    y2, s2 = gpu_step(d, "bf16", in_place=True)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)
    y0, s0 = gpu_step(d, "bf16", use_D=False)
    yr, _ = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], None)
    assert normwise(y0, yr) <= TOL["bf16"] and np.array_equal(s0, s1)


@pytest.mark.parametrize("N", [128, 256])
def test_prefill_then_decode_equals_recurrence(N):
    # forward over the first T0 tokens, then K recurrent steps from its final state, all on the GPU,
    # against the oracle's token-by-token recurrence over the T0 + K tokens
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step
    T0, K = 300, 6
    w = WORKLOADS["m2_2p7b"].with_(batch=2, seqlen=T0 + K, nheads=4, dstate=N, seed=320 + N)
    d = make_inputs(w)
    yr, fr = oracle.ssd_recurrence(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_state"])
    pre = {k: (v[:, :T0] if k in ("x", "dt", "B", "C") else v) for k, v in d.items()}
    y0, f0 = run_gpu(pre, "bf16", 256)
    assert normwise(y0, yr[:, :T0]) <= TOL["bf16"]
    state = torch.from_numpy(f0.astype(np.float32)).cuda()
    for k in range(K):
        t = T0 + k
        td = to_dev(dict(x=d["x"][:, t], dt=d["dt"][:, t], A=d["A"], B=d["B"][:, t], C=d["C"][:, t], D=d["D"]),
                    "bf16")
        y, state = ssd_decode_step(td["x"], td["dt"], td["A"], td["B"], td["C"], td["D"], state)
        torch.cuda.synchronize()
        assert normwise(y.float().cpu().numpy(), yr[:, t]) <= TOL["bf16"]
    assert normwise(state.cpu().numpy(), fr) <= TOL["bf16"]


def test_decode_full_workload():
    w = WORKLOADS["decode_2p7b"]
    d = decode_inputs(w.batch, w.nheads, w.headdim, w.dstate, w.ngroups, w.dtype, seed=w.seed)
    y, s = gpu_step(d, "bf16", in_place=True)
    yr, sr = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    ey, es = normwise(y, yr), normwise(s, sr)
    print(f"[decode parity] decode_2p7b y_err={ey:.3e} state_err={es:.3e}")
    assert ey <= TOL["bf16"] and es <= 1e-5


def test_decode_bf16_state_full_workload():
    from mamba_ssd_layer_gb300.inputs import bf16_round
    w = WORKLOADS["decode_2p7b_bf16state"]
    d = decode_inputs(w.batch, w.nheads, w.headdim, w.dstate, w.ngroups, w.dtype, seed=w.seed)
    d["state"] = bf16_round(d["state"])
    y, s = bf16_state_step(d, w.dtype, in_place=True)
    yr, sr = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    ey, es = normwise(y, yr), normwise(s, sr)
    print(f"[decode parity] decode_2p7b_bf16state y_err={ey:.3e} state_err={es:.3e}")
    assert ey <= TOL["bf16"] and es <= TOL["bf16"]


def test_decode_host_entry_matches_device_entry():
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step_host
    d = decode_inputs(3, 4, 64, 128, 1, "bf16", seed=330)
    y_dev, s_dev = gpu_step(d, "bf16")
    h = {k: torch.from_numpy(np.ascontiguousarray(d[k])) for k in d}
    for k in ("x", "B", "C"):
        h[k] = h[k].bfloat16()
    new = torch.empty_like(h["state"])
    y, s = ssd_decode_step_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["state"], new)
    assert np.array_equal(y.float().numpy(), y_dev.astype(np.float32))
    assert np.array_equal(s.numpy(), s_dev.astype(np.float32))
    assert np.array_equal(h["state"].numpy(), d["state"])          # the input state is left alone


def test_decode_empty_batch():
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step
    x = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((0, 2, 64, 128), dtype=torch.float32, device="cuda")
    y, s = ssd_decode_step(x, torch.empty((0, 2), device="cuda"), torch.ones(2, device="cuda").neg(), B, B.clone(),
                           None, st)
    torch.cuda.synchronize()
    assert y.shape == (0, 2, 64) and s.shape == st.shape


# ---------------------------------------------------------------- state stored in bf16
BF16S_CASES = [(3, 4, 64, 128, 1, "bf16"), (2, 6, 64, 256, 2, "bf16"), (2, 4, 64, 64, 1, "bf16"),
               (2, 4, 16, 8, 1, "f32"), (1, 2, 33, 24, 1, "f32"), (3, 3, 7, 136, 3, "f32"),
               (3, 2, 100, 128, 1, "bf16")]   # two row blocks per head, the second partial


def bf16_state_step(d, dtype, in_place=False):
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step
    t = to_dev({k: v for k, v in d.items() if k != "state"}, dtype)
    st = torch.from_numpy(np.ascontiguousarray(d["state"])).cuda().bfloat16()
    new = st if in_place else torch.empty_like(st)
    y, s = ssd_decode_step(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], st, new)
    torch.cuda.synchronize()
    assert s.dtype == torch.bfloat16
    return y.float().cpu().numpy().astype(np.float64), s.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", BF16S_CASES, ids=[f"b{c[0]}H{c[1]}P{c[2]}N{c[3]}G{c[4]}{c[5]}" for c in BF16S_CASES])
def test_decode_bf16_state_matches_oracle(case):
    from mamba_ssd_layer_gb300.inputs import bf16_round
    batch, H, P, N, G, dtype = case
    d = decode_inputs(batch, H, P, N, G, dtype, seed=400 + N + P)
    d["state"] = bf16_round(d["state"])                  # the carried state is stored in bf16 on both sides
    y, s = bf16_state_step(d, dtype)
    yr, sr = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"])
    ey, es = normwise(y, yr), normwise(s, sr)
    print(f"[decode bf16 state] {case} y_err={ey:.3e} state_err={es:.3e}")
    # y comes from the unrounded fp32 update; only the stored state is rounded to bf16
    assert ey <= TOL[dtype]
    assert es <= TOL["bf16"]
    assert np.array_equal(s, bf16_round(s.astype(np.float32)).astype(np.float64))


def test_decode_bf16_state_in_place_and_host_entry():
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step_host
    from mamba_ssd_layer_gb300.inputs import bf16_round
    d = decode_inputs(3, 4, 64, 128, 1, "bf16", seed=431)
    d["state"] = bf16_round(d["state"])
    y1, s1 = bf16_state_step(d, "bf16")
    y2, s2 = bf16_state_step(d, "bf16", in_place=True)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)
    h = {k: torch.from_numpy(np.ascontiguousarray(d[k])) for k in d}
    for k in ("x", "B", "C", "state"):
        h[k] = h[k].bfloat16()
    new = torch.empty_like(h["state"])
    y, s = ssd_decode_step_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["state"], new)
    assert np.array_equal(y.float().numpy().astype(np.float64), y1)
    assert np.array_equal(s.float().numpy().astype(np.float64), s1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_dt_scaled_input(dtype):
    d = decode_inputs(3, 4, 64, 128, 2, dtype, seed=440)
    y, s = gpu_step(d, dtype, scale_x_by_dt=True)
    yr, sr = oracle.ssd_decode_step(d["state"], d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], scale_x_by_dt=True)
    assert normwise(y, yr) <= TOL[dtype] and normwise(s, sr) <= 1e-5


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_host_pipeline_matches_device_entry(state_dtype):
    # enough carried states (at least 32 MB of state) that the host step runs as a pipeline over groups of
    # batch rows, with a ragged last group; rows are independent, so it must equal the device step exactly
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step_host
    from mamba_ssd_layer_gb300.inputs import bf16_round
    d = decode_inputs(70, 32, 64, 128, 1, "bf16", seed=450)
    if state_dtype == "bf16":
        d["state"] = bf16_round(d["state"])
        y_dev, s_dev = bf16_state_step(d, "bf16")
    else:
        y_dev, s_dev = gpu_step(d, "bf16")
    h = {k: torch.from_numpy(np.ascontiguousarray(d[k])) for k in d}
    for k in ("x", "B", "C") + (("state",) if state_dtype == "bf16" else ()):
        h[k] = h[k].bfloat16()
    h = {k: v.pin_memory() for k, v in h.items()}
    new = torch.empty_like(h["state"]).pin_memory()
    y, s = ssd_decode_step_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["state"], new)
    assert np.array_equal(y.float().numpy().astype(np.float64), np.asarray(y_dev, dtype=np.float64))
    assert np.array_equal(s.float().numpy().astype(np.float64), np.asarray(s_dev, dtype=np.float64))
