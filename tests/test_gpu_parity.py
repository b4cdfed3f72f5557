"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs. Tolerances (normwise max|out - ref| / max|ref|): 1e-4 for the fp32
path, 1e-2 for the bf16 path (fp32 accumulation), for y and the final states alike."""
import numpy as np
import pytest

from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant
from ssd_util import TOL, normwise, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def check(d, dtype, chunk, heads=None, use_D=True, scale_x_by_dt=False):
    y, f = run_gpu(d, dtype, chunk, use_D=use_D, scale_x_by_dt=scale_x_by_dt)
    yr, fr = run_oracle(d, heads=heads, use_D=use_D, scale_x_by_dt=scale_x_by_dt)
    if heads is not None:
        y, f = y[:, :, heads], f[:, heads]
    ey, ef = normwise(y, yr), normwise(f, fr)
    print(f"[parity] {dtype} chunk={chunk} y_err={ey:.3e} final_err={ef:.3e}")
    assert np.isfinite(y).all() and np.isfinite(f).all()
    assert ey <= TOL[dtype], f"y error {ey:.3e}"
    assert ef <= TOL[dtype], f"final state error {ef:.3e}"
    return ey, ef


# ---------------------------------------------------------------- fp32 path
def test_fp32_tiny_workload():
    d = make_inputs(WORKLOADS["fp32_tiny"])
    check(d, "f32", 64)


@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_fp32_chunk_sizes_ragged(chunk):
    w = WORKLOADS["fp32_tiny"].with_(batch=2, seqlen=700, nheads=4, init_state=True, seed=77)
    check(make_inputs(w), "f32", chunk)


def test_fp32_odd_sizes_groups():
    w = WORKLOADS["fp32_tiny"].with_(batch=3, seqlen=131, nheads=6, headdim=12, dstate=20, ngroups=3,
                                     init_state=True, seed=78)
    check(make_inputs(w), "f32", 64)


# ---------------------------------------------------------------- bf16 path, small (whole output vs oracle)
@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("N", [64, 128, 256])
def test_bf16_chunk_sizes_ragged(chunk, N):
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=1000, nheads=4, batch=2).with_(dstate=N, seed=90 + N)
    check(make_inputs(w), "bf16", chunk)


def test_bf16_chunk_does_not_change_the_result():
    """On the bf16 path the kernel's tile is 128 tokens whatever `chunk` says (the decomposition is exact
    for any block length, "LLM(十一)——Mamba" §3.5), so the three values give bit-identical outputs; the
    oracle check of each is in test_bf16_chunk_sizes_ragged."""
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=777, nheads=2, batch=1).with_(seed=91)
    d = make_inputs(w)
    outs = [run_gpu(d, "bf16", q) for q in (64, 128, 256)]
    for (y, f) in outs[1:]:
        assert np.array_equal(y, outs[0][0]) and np.array_equal(f, outs[0][1])


def test_bf16_skip_term_in_fp32():
    """With C = 0 the layer reduces to its skip term: y = D x exactly. D is fp32, so y must be the
    bf16 rounding (to nearest even) of the fp32 product D x, element by element."""
    import torch
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=700, nheads=4, batch=2).with_(seed=103)
    d = dict(make_inputs(w))
    d["C"] = np.zeros_like(d["C"])
    y, _ = run_gpu(d, "bf16", 256)
    prod = d["D"].astype(np.float32)[None, None, :, None] * d["x"].astype(np.float32)
    want = torch.from_numpy(prod).to(torch.bfloat16).float().numpy()
    assert np.array_equal(y.astype(np.float32), want)


def test_bf16_no_skip_no_init():
    w = small_variant(WORKLOADS["m2_130m"], seqlen=512, nheads=4, batch=2).with_(seed=92)
    check(make_inputs(w), "bf16", 256, use_D=False)


@pytest.mark.parametrize("T", [1, 17, 128, 129, 255, 256, 257])
def test_bf16_short_and_boundary_lengths(T):
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=T, nheads=2, batch=3).with_(seed=93 + T)
    check(make_inputs(w), "bf16", 256)


@pytest.mark.parametrize("T,H,batch,N", [(8192, 2, 1, 128), (3000, 4, 3, 128), (20000, 2, 1, 128),
                                         (8192, 2, 1, 256), (3000, 4, 3, 64)])
def test_bf16_long_chains_few_heads(T, H, batch, N):
    # few head pairs and long sequences: many windows per chain, a deep cross-window scan
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=T, nheads=H, batch=batch).with_(dstate=N, seed=99 + T + N)
    check(make_inputs(w), "bf16", 256)


@pytest.mark.parametrize("N", [128, 256])
def test_bf16_deterministic(N):
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=5000, nheads=4, batch=1).with_(dstate=N, seed=101)
    d = make_inputs(w)
    y1, f1 = run_gpu(d, "bf16", 256)
    y2, f2 = run_gpu(d, "bf16", 256)
    assert np.array_equal(y1, y2) and np.array_equal(f1, f2)


@pytest.mark.parametrize("N", [64, 128, 256])
def test_bf16_grouped_heads(N):
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=600, nheads=8, batch=1).with_(ngroups=2, dstate=N, seed=94)
    check(make_inputs(w), "bf16", 128)


@pytest.mark.parametrize("N", [128, 256])
def test_bf16_varlen_small(N):
    w = small_variant(WORKLOADS["varlen"], seqlen=3000, nheads=4).with_(seg_min=1, seg_max=700, seed=95,
                                                                      init_state=True, dstate=N)
    d = make_inputs(w)
    assert len(d["cu_seqlens"]) > 4
    check(d, "bf16", 256)


@pytest.mark.parametrize("N", [64, 128, 256])
def test_bf16_varlen_empty_segments(N):
    # zero-length segments first, between others and last: their final state is their initial state
    w = small_variant(WORKLOADS["varlen"], seqlen=2500, nheads=4).with_(seg_min=100, seg_max=900, seed=102,
                                                                      dstate=N)
    d = make_inputs(w)
    cu = [int(v) for v in d["cu_seqlens"]]
    cu = [0, 0] + cu[1:2] + cu[1:-1] + cu[-1:] + cu[-1:]
    d["cu_seqlens"] = np.asarray(cu, dtype=np.int32)
    nseq = len(cu) - 1
    rng = np.random.Generator(np.random.PCG64(103 + N))
    d["initial_state"] = rng.standard_normal((nseq, 4, 64, N), dtype=np.float32) * np.float32(0.1)
    ey, ef = check(d, "bf16", 256)
    _, f = run_gpu(d, "bf16", 256)
    for s in range(nseq):
        if cu[s + 1] == cu[s]:
            assert np.array_equal(f[s], d["initial_state"][s].astype(np.float64))


def test_fp32_varlen_small():
    w = small_variant(WORKLOADS["varlen"], seqlen=900, nheads=2).with_(headdim=16, dstate=16, dtype="f32",
                                                                     seg_min=1, seg_max=200, seed=96,
                                                                     init_state=True)
    check(make_inputs(w), "f32", 64)


@pytest.mark.parametrize("N", [128, 256])
def test_empty_sequence(N):
    import torch
    from mamba_ssd_layer_gb300 import ssd_forward
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=0, nheads=2, batch=2).with_(seed=97, dstate=N)
    d = make_inputs(w)
    from ssd_util import to_device
    t = to_device(d, "bf16")
    y, f = ssd_forward(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=256,
                       initial_state=t["initial_state"])
    torch.cuda.synchronize()
    assert y.shape[1] == 0
    assert torch.equal(f.cpu(), t["initial_state"].cpu())


def test_host_entry_point_matches_device_entry_point():
    import torch
    from mamba_ssd_layer_gb300 import ssd_forward_host
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=512, nheads=4, batch=2).with_(seed=98)
    d = make_inputs(w)
    y_dev, f_dev = run_gpu(d, "bf16", 256)
    h = {k: (torch.from_numpy(d[k]).bfloat16() if k in ("x", "B", "C") else torch.from_numpy(d[k]))
         for k in ("x", "dt", "A", "B", "C", "D", "initial_state")}
    y, f = ssd_forward_host(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], chunk=256,
                            initial_state=h["initial_state"])
    assert np.array_equal(y.float().numpy(), y_dev.astype(np.float32))
    assert np.array_equal(f.numpy(), f_dev.astype(np.float32))


# ---------------------------------------------------------------- full workloads, sampled heads
FULL = [("m2_130m", [0, 11, 23]), ("m2_2p7b", [0, 41, 79]), ("long_n64", [3, 77]),
        ("long_n128", [0, 40, 79]), ("long_n256", [1, 78]), ("varlen", [0, 31])]


@pytest.mark.parametrize("name,heads", FULL, ids=[f[0] for f in FULL])
def test_full_workload_sampled_heads(name, heads):
    w = WORKLOADS[name]
    d = make_inputs(w)
    check(d, "bf16", w.chunk, heads=heads)


# ---------------------------------------------------------------- dt-scaled input term (dt x B^T)
@pytest.mark.parametrize("N", [64, 128, 256])
def test_bf16_dt_scaled_input_ragged(N):
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=1000, nheads=4, batch=2).with_(dstate=N, seed=500 + N)
    check(make_inputs(w), "bf16", 256, scale_x_by_dt=True)


def test_bf16_dt_scaled_input_long_chain_and_packed():
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=8192, nheads=2, batch=1).with_(seed=510)
    check(make_inputs(w), "bf16", 256, scale_x_by_dt=True)
    wv = small_variant(WORKLOADS["varlen"], seqlen=3000, nheads=4).with_(seg_min=1, seg_max=700, seed=511,
                                                                       init_state=True)
    check(make_inputs(wv), "bf16", 256, scale_x_by_dt=True)


def test_bf16_dt_scaled_input_tiny_dt():
    # dt down to zero: the kernel floors log2(dt); the contribution of such a token is ~0 either way
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=700, nheads=2, batch=1).with_(seed=512)
    d = make_inputs(w)
    d["dt"] = d["dt"].copy()
    d["dt"][0, ::7, :] = 0.0
    d["dt"][0, 3::11, :] = 1e-12
    check(d, "bf16", 256, scale_x_by_dt=True)


def test_fp32_dt_scaled_input():
    w = WORKLOADS["fp32_tiny"].with_(batch=2, seqlen=300, nheads=4, init_state=True, seed=513)
    check(make_inputs(w), "f32", 64, scale_x_by_dt=True)


def test_dt_scaled_full_workload_sampled_heads():
    w = WORKLOADS["long_n128"]
    check(make_inputs(w), "bf16", w.chunk, heads=[0, 79], scale_x_by_dt=True)


# ---------------------------------------------------------------- the host entry point's pipeline
# A large dense bf16 batch is cut into pieces whose copies and forwards overlap: batch rows, or time
# slices of one sequence joined by the state hand-off. Both must match the oracle like the device path.
PIPELINED = [
    ("batch_rows", dict(batch=3, seqlen=4096, nheads=32), [0, 17, 31]),      # 3 pieces of one row
    ("time_slices", dict(batch=1, seqlen=16384, nheads=16), [0, 9, 15]),     # 4 slices of 4096 tokens
    ("time_ragged", dict(batch=1, seqlen=17000, nheads=16), [2, 13]),        # slices of 4352, the last short
]


@pytest.mark.parametrize("name,shape,heads", PIPELINED, ids=[p[0] for p in PIPELINED])
def test_host_entry_point_pipeline(name, shape, heads):
    import torch
    from mamba_ssd_layer_gb300 import ssd_forward_host
    w = small_variant(WORKLOADS["m2_2p7b"], **shape).with_(seed=400 + shape["seqlen"] % 97)
    d = make_inputs(w)
    h = {k: (torch.from_numpy(d[k]).bfloat16() if k in ("x", "B", "C") else torch.from_numpy(d[k]))
         for k in ("x", "dt", "A", "B", "C", "D", "initial_state")}
    pin = {k: v.pin_memory() for k, v in h.items()}
    y, f = ssd_forward_host(pin["x"], pin["dt"], pin["A"], pin["B"], pin["C"], pin["D"], chunk=256,
                            initial_state=pin["initial_state"])
    y_ref, f_ref = run_oracle(d, heads=heads)
    hs = np.asarray(heads)
    assert normwise(y.float().numpy()[:, :, hs], y_ref) <= TOL["bf16"]
    assert normwise(f.numpy()[:, hs], f_ref) <= TOL["bf16"]
