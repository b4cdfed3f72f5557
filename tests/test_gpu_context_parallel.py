"""The device pieces of the sequence-parallel forward on one GPU: a sequence batch cut into slices,
each run from a zero state by ssd_forward, its decay by ssd_slice_decay and its correction for the
entering state by ssd_slice_correct, handed along in order (context_parallel.run_slices). The composed
outputs and final state must match the oracle run over the whole sequence."""
import numpy as np
import pytest

from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant
from ssd_util import TOL, normwise

pytestmark = pytest.mark.gpu


def _slices(t, cuts):
    return [tuple(t[k][:, a:b].contiguous() for k in ("x", "dt", "B", "C")) for a, b in zip(cuts[:-1], cuts[1:])]


def _dev(d):
    import torch
    t = {k: torch.from_numpy(d[k]).cuda().to(torch.bfloat16).contiguous() for k in ("x", "B", "C")}
    for k in ("dt", "A", "D"):
        t[k] = torch.from_numpy(d[k]).cuda().contiguous()
    t["init"] = None if d["initial_state"] is None else torch.from_numpy(d["initial_state"]).cuda()
    return t


@pytest.mark.parametrize("N,cuts", [
    (128, [0, 300, 301, 700, 1000]),     # a one-token slice, ragged tiles
    (64, [0, 512, 1000]),
    (256, [0, 129, 640, 1000]),
])
def test_slices_compose_to_the_whole_sequence(N, cuts):
    import torch
    import oracle
    from mamba_ssd_layer_gb300.context_parallel import cuda_ops, run_slices
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=1000, nheads=4, batch=2).with_(dstate=N, seed=300 + N)
    d = make_inputs(w)
    t = _dev(d)
    ys, fin = run_slices(_slices(t, cuts), t["A"], t["D"], t["init"], ops=cuda_ops())
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=1).float().cpu().numpy()
    y_ref, fin_ref = oracle.ssd_recurrence(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                           initial_state=d["initial_state"])
    assert normwise(y, y_ref) <= TOL["bf16"]
    assert normwise(fin.cpu().numpy(), fin_ref) <= TOL["bf16"]
    # the comparison is not vacuous: the last slice run from a zero state, uncorrected, is off
    xs, dts, Bs, Cs = _slices(t, cuts)[-1]
    y_last, _ = cuda_ops().forward(xs, dts, t["A"], Bs, Cs, t["D"], None)
    torch.cuda.synchronize()
    err_plain = normwise(y_last.float().cpu().numpy(), y_ref[:, cuts[-2]:])
    err_corrected = normwise(ys[-1].float().cpu().numpy(), y_ref[:, cuts[-2]:])
    assert err_plain > 3 * err_corrected


def test_slice_decay_is_exp_of_the_summed_log_decay():
    import torch
    from mamba_ssd_layer_gb300 import binding as bd
    w = small_variant(WORKLOADS["m2_130m"], seqlen=333, nheads=6, batch=3).with_(seed=311)
    d = make_inputs(w)
    dt = torch.from_numpy(d["dt"]).cuda()
    A = torch.from_numpy(d["A"]).cuda()
    dec = bd.ssd_slice_decay(dt, A)
    torch.cuda.synchronize()
    ref = np.exp(d["A"][None, :].astype(np.float64) * d["dt"].astype(np.float64).sum(axis=1))
    np.testing.assert_allclose(dec.cpu().numpy(), ref, rtol=2e-5, atol=1e-30)


def test_correction_of_an_empty_slice_passes_the_state_through():
    import torch
    from mamba_ssd_layer_gb300 import binding as bd
    H, P, N, G = 4, 64, 128, 1
    dt = torch.empty((2, 0, H), dtype=torch.float32, device="cuda")
    A = -torch.ones(H, dtype=torch.float32, device="cuda")
    C = torch.empty((2, 0, G, N), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((2, 0, H, P), dtype=torch.bfloat16, device="cuda")
    h_in = torch.randn((2, H, P, N), dtype=torch.float32, device="cuda")
    fin = torch.randn((2, H, P, N), dtype=torch.float32, device="cuda")
    want = fin + h_in
    bd.ssd_slice_correct(dt, A, C, h_in, y, fin)
    torch.cuda.synchronize()
    assert torch.equal(fin, want)
    dec = bd.ssd_slice_decay(dt, A)
    torch.cuda.synchronize()
    assert torch.equal(dec.cpu(), torch.ones((2, H)))
