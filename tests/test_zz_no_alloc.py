"""ssd_forward_noalloc: the same forward pass with scratch in a static device array, for
callers that cannot allocate device memory. Checked through the C ABI against ssd_forward
on the same inputs, on two calls in a row. The array is shared and keeps the previous call's
contents, so a call on other inputs runs between the two compared calls: the second compared call
then starts from another problem's scratch, which must not leak into its results.

This file is named to run last: if it fails, a run that stops at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

from mamba_ssd_layer_gb300 import binding as bd
from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant
from ssd_util import TOL, normwise, to_device

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = bd.load_library()
    fn = lib.ssd_forward_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(bd._Shape), ctypes.c_int, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp,
                   ctypes.c_int, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("dtype,w", [
    ("bf16", small_variant(WORKLOADS["m2_2p7b"], seqlen=700, nheads=4, batch=2).with_(seed=201)),
    ("f32", WORKLOADS["fp32_tiny"].with_(batch=2, seqlen=300, nheads=2, init_state=True, seed=202)),
    ("bf16", small_variant(WORKLOADS["varlen"], seqlen=3000, nheads=4, seg_min=17, seg_max=900).with_(seed=203)),
])
def test_noalloc_matches_workspace_entry_point(dtype, w):
    import torch
    from mamba_ssd_layer_gb300 import ssd_forward
    fn = _noalloc_fn()
    d = make_inputs(w)
    t = to_device(d, dtype)
    cu = t["cu_seqlens"]
    nseq = 0 if cu is None else cu.shape[0] - 1
    y_ref, f_ref = ssd_forward(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], chunk=w.chunk,
                               initial_state=t["initial_state"], cu_seqlens=cu)
    torch.cuda.synchronize()
    x = t["x"]
    shape = bd._shape(x.shape[0], x.shape[1], x.shape[2], x.shape[3], t["B"].shape[3], t["B"].shape[2])
    code = bd.SSD_F32 if dtype == "f32" else bd.SSD_BF16
    stream = torch.cuda.current_stream()
    def call(tt, y, f):
        return fn(ctypes.byref(shape), code, _ptr(tt["x"]), _ptr(tt["dt"]), _ptr(tt["A"]), _ptr(tt["B"]),
                  _ptr(tt["C"]), _ptr(tt["D"]), w.chunk, _ptr(tt["initial_state"]), _ptr(cu), nseq, _ptr(y),
                  _ptr(f), ctypes.c_void_p(stream.cuda_stream))

    other = to_device(make_inputs(w.with_(seed=w.seed + 1000)), dtype)
    for k in range(2):
        y = torch.full_like(x, float("nan"))
        f = torch.full_like(f_ref, float("nan"))
        rc = call(t, y, f)
        assert rc == bd.SSD_OK, bd.ssd_status_string(rc)
        torch.cuda.synchronize()
        assert normwise(y.float().cpu().numpy(), y_ref.float().cpu().numpy()) <= TOL[dtype]
        assert normwise(f.cpu().numpy(), f_ref.cpu().numpy()) <= TOL[dtype]
        if k == 0:
            # another problem of the same shape in between: it leaves its own scratch behind
            rc = call(other, torch.empty_like(x), torch.empty_like(f_ref))
            assert rc == bd.SSD_OK, bd.ssd_status_string(rc)
            torch.cuda.synchronize()


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc_fn()
    big = bd._shape(1, 1 << 20, 80, 64, 128, 1)   # far more scratch than the built-in array
    fake = 1 << 20
    rc = fn(ctypes.byref(big), bd.SSD_BF16, fake, fake, fake, fake, fake, None, 256, None, None, 0, fake, None,
            None)
    assert rc == bd.SSD_ERR_WORKSPACE
    assert "bytes of scratch" in bd.load_library().ssd_last_error_detail().decode()
