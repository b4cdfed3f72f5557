"""Out-of-bounds writes on the GPU, without a sanitizer: every buffer a call writes (outputs, states,
workspace) is a view into a larger allocation whose guard bands before and after hold a fixed bit
pattern. After the call the guard bands must be untouched, and the result must equal the same call on
unguarded buffers bit for bit. Shapes are ragged (partial tiles, partial row quadrants, 1-token and
empty segments) so that every edge path of the kernels runs."""
import numpy as np
import pytest

from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant
from ssd_util import to_device

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes on either side (a multiple of 256: the views keep their alignment)
PATTERN = 0x5A


def guarded(shape, dtype):
    """(view of `shape` and dtype, the whole uint8 allocation) with guard bands filled with PATTERN; the
    view itself is filled with the pattern too (so unwritten elements would show)."""
    import torch
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    view = raw[GUARD:GUARD + n].view(dtype).view(*shape)
    return view, raw


def assert_guards(raw, what):
    head = raw[:GUARD].cpu().numpy()
    tail = raw[-GUARD:].cpu().numpy()
    assert (head == PATTERN).all(), f"{what}: written before its start"
    assert (tail == PATTERN).all(), f"{what}: written past its end"


def forward_case(d, dtype, chunk):
    import torch
    from mamba_ssd_layer_gb300 import binding as bd
    from mamba_ssd_layer_gb300 import ssd_forward
    t = to_device(d, dtype)
    x = t["x"]
    cu = t["cu_seqlens"]
    nseq = x.shape[0] if cu is None else cu.shape[0] - 1
    H, P, N, G = x.shape[2], x.shape[3], t["B"].shape[3], t["B"].shape[2]
    code = bd.SSD_F32 if dtype == "f32" else bd.SSD_BF16
    ws_bytes = bd.ssd_workspace_size(x.shape[0], x.shape[1], H, P, N, G, code, chunk, 0 if cu is None else nseq)
    args = (t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"])
    kw = dict(chunk=chunk, initial_state=t["initial_state"], cu_seqlens=cu)
    y_ref, f_ref = ssd_forward(*args, **kw)
    y, y_raw = guarded(tuple(x.shape), x.dtype)
    f, f_raw = guarded((nseq, H, P, N), torch.float32)
    ws, ws_raw = guarded((ws_bytes,), torch.uint8)
    ssd_forward(*args, **kw, y=y, final_state=f, workspace=ws)
    torch.cuda.synchronize()
    assert bd.ssd_status(ws) == bd.SSD_OK
    assert_guards(y_raw, "y")
    assert_guards(f_raw, "final_state")
    assert_guards(ws_raw, "workspace")
    assert torch.equal(y, y_ref) and torch.equal(f, f_ref)


@pytest.mark.parametrize("N", [64, 128, 256])
def test_forward_dense_ragged(N):
    # two sequences of 300 tokens: a partial last tile and partial 32-row quadrants, with an initial state
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=300, nheads=4, batch=2).with_(dstate=N, seed=700 + N)
    forward_case(make_inputs(w), "bf16", 256)


def test_forward_long_chain_ranges():
    # one head pair over 5000 tokens: CTA ranges start inside the chain (look-back, correction tiles)
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=5000, nheads=2, batch=1).with_(seed=710)
    forward_case(make_inputs(w), "bf16", 256)


def test_forward_packed_with_short_and_empty_segments():
    w = small_variant(WORKLOADS["varlen"], seqlen=2000, nheads=4, seg_min=1, seg_max=300).with_(seed=711)
    d = make_inputs(w)
    # an empty segment and a 1-token one in the middle of the packed row
    cu = [int(v) for v in d["cu_seqlens"]]
    cu = cu[:3] + [cu[2], cu[2] + 1] + cu[3:]
    d["cu_seqlens"] = np.asarray(cu, dtype=np.int32)
    forward_case(d, "bf16", 256)


def test_forward_fp32():
    w = WORKLOADS["fp32_tiny"].with_(batch=2, seqlen=333, nheads=2, init_state=True, seed=712)
    forward_case(make_inputs(w), "f32", 64)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_step(state_dtype):
    import torch
    from mamba_ssd_layer_gb300 import ssd_decode_step
    w = WORKLOADS["decode_2p7b"].with_(batch=5, nheads=6, headdim=40, dstate=64, seed=713)
    d = make_inputs(w)
    sdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.float32)
    args = (bf(d["x"][:, 0]), f32(d["dt"][:, 0]), f32(d["A"]), bf(d["B"][:, 0]), bf(d["C"][:, 0]), f32(d["D"]))
    state = torch.from_numpy(d["initial_state"]).cuda().to(sdt)
    y_ref, s_ref = ssd_decode_step(*args, state=state, new_state=torch.empty_like(state))
    ns, ns_raw = guarded(tuple(state.shape), sdt)
    y, y_raw = guarded(tuple(args[0].shape), torch.bfloat16)
    ssd_decode_step(*args, state=state, new_state=ns, y=y)
    torch.cuda.synchronize()
    assert_guards(ns_raw, "new_state")
    assert_guards(y_raw, "y")
    assert torch.equal(y, y_ref) and torch.equal(ns, s_ref)


@pytest.mark.parametrize("gated", [True, False])
def test_gated_rmsnorm(gated):
    import torch
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    rng = np.random.default_rng(714)
    y = torch.from_numpy(rng.standard_normal((3, 77, 20, 64), dtype=np.float32)).cuda().bfloat16()
    z = torch.from_numpy(rng.standard_normal((3, 77, 20, 64), dtype=np.float32)).cuda().bfloat16() if gated else None
    wt = torch.from_numpy(rng.uniform(0.5, 1.5, 20 * 64).astype(np.float32)).cuda()
    ref = ssd_gated_rmsnorm(y, z, wt, groups=32)
    out, out_raw = guarded(tuple(y.shape), torch.bfloat16)
    ssd_gated_rmsnorm(y, z, wt, groups=32, out=out)
    torch.cuda.synchronize()
    assert_guards(out_raw, "out")
    assert torch.equal(out, ref)


def test_slice_correct():
    import torch
    from mamba_ssd_layer_gb300 import ssd_forward, ssd_slice_correct
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=301, nheads=4, batch=2).with_(seed=715)
    d = make_inputs(w)
    t = to_device(d, "bf16")
    y0, f0 = ssd_forward(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"])
    h_in = t["initial_state"]
    y_ref, f_ref = ssd_slice_correct(t["dt"], t["A"], t["C"], h_in, y0.clone(), f0.clone())
    y, y_raw = guarded(tuple(y0.shape), torch.bfloat16)
    f, f_raw = guarded(tuple(f0.shape), torch.float32)
    y.copy_(y0)
    f.copy_(f0)
    ssd_slice_correct(t["dt"], t["A"], t["C"], h_in, y, f)
    torch.cuda.synchronize()
    assert_guards(y_raw, "y")
    assert_guards(f_raw, "final_state")
    assert torch.equal(y, y_ref) and torch.equal(f, f_ref)
