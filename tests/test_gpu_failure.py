"""Device-side failure detection on the bf16 path, tested without faulting the GPU.

The failure is made on the host side of the kernel's protocol: the test hook SSD_DEBUG_FORCE_TIMEOUT makes
every cross-CTA wait (the look-back of the inter-chunk pass) wait for a published state that never
comes, with a limit of about a millisecond. The kernel must then record SSD_ERR_TIMEOUT and the location
code of the look-back in the workspace, let its copies and tensor-core work in flight finish, and
return; the next normal call on the same workspace must be correct. A malformed cu_seqlens is reported
the same way, through the workspace status (the device-side table builder finds it)."""
import ctypes

import numpy as np
import pytest

from mamba_ssd_layer_gb300 import binding as bd
from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant
from ssd_util import TOL, normwise, run_oracle, to_device

pytestmark = pytest.mark.gpu

LOC_LOOKBACK = 0x300


def _forward_ex(t, flags, ws, y, f, cu=None, nseq=0):
    import torch
    lib = bd.load_library()
    x = t["x"]
    shape = bd._shape(x.shape[0], x.shape[1], x.shape[2], x.shape[3], t["B"].shape[3], t["B"].shape[2])
    p = lambda v: None if v is None else v.data_ptr()
    return lib.ssd_forward_ex(ctypes.byref(shape), bd.SSD_BF16, flags, p(x), p(t["dt"]), p(t["A"]), p(t["B"]),
                              p(t["C"]), p(t["D"]), 256, p(t["initial_state"]), p(cu), nseq, p(y), p(f),
                              ws.data_ptr(), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("N", [64, 128, 256])
def test_forced_lookback_timeout_is_reported_and_the_next_call_is_correct(N):
    import torch
    # one head pair and a long sequence: a single chain cut into several windows, so that most windows
    # look back at another CTA's published state
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=4096, nheads=2, batch=1).with_(dstate=N, seed=301)
    d = make_inputs(w)
    t = to_device(d, "bf16")
    nbytes = bd.ssd_workspace_size(1, w.seqlen, 2, 64, N, 1, bd.SSD_BF16, 256, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["x"])
    f = torch.empty((1, 2, 64, N), dtype=torch.float32, device="cuda")
    rc = _forward_ex(t, bd.SSD_DEBUG_FORCE_TIMEOUT, ws, y, f)
    assert rc == bd.SSD_OK
    assert bd.ssd_status(ws) == bd.SSD_ERR_TIMEOUT
    header = ws[:16].cpu().numpy().view(np.int32)
    assert header[2] == LOC_LOOKBACK, header.tolist()
    # the context is still usable, and the same workspace serves a normal call
    rc = _forward_ex(t, 0, ws, y, f)
    assert rc == bd.SSD_OK
    assert bd.ssd_status(ws) == bd.SSD_OK
    yr, fr = run_oracle(d)
    assert normwise(y.float().cpu().numpy(), yr) <= TOL["bf16"]
    assert normwise(f.cpu().numpy(), fr) <= TOL["bf16"]


@pytest.mark.parametrize("cu", [[0, 100, 50, 300], [0, 100, 200, 250], [5, 100, 200, 300]],
                         ids=["decreasing", "short_of_the_end", "not_from_zero"])
def test_malformed_cu_seqlens_is_reported_by_status(cu):
    import torch
    w = small_variant(WORKLOADS["varlen"], seqlen=300, nheads=2).with_(seg_min=50, seg_max=120, seed=302)
    d = make_inputs(w)
    t = to_device(d, "bf16")
    cut = torch.tensor(cu, dtype=torch.int32, device="cuda")
    nseq = len(cu) - 1
    t["initial_state"] = None
    nbytes = bd.ssd_workspace_size(1, 300, 2, 64, 128, 1, bd.SSD_BF16, 256, nseq)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = torch.zeros_like(t["x"])
    f = torch.empty((nseq, 2, 64, 128), dtype=torch.float32, device="cuda")
    assert _forward_ex(t, 0, ws, y, f, cu=cut, nseq=nseq) == bd.SSD_OK
    assert bd.ssd_status(ws) == bd.SSD_ERR_INVALID_ARG
    assert torch.count_nonzero(y).item() == 0      # nothing was written
