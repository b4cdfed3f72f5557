"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the binding, run the oracle (optionally on a subset of heads), and
measure the normwise error max|out - ref| / max|ref| used as the pass criterion."""
from __future__ import annotations

import numpy as np

import oracle

TOL = {"f32": 1e-4, "bf16": 1e-2}


def normwise(out, ref) -> float:
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(out - ref)) / (den if den > 0 else 1.0))


def to_device(d: dict, dtype: str, device="cuda"):
    import torch
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    t = {}
    for k in ("x", "B", "C"):
        t[k] = torch.from_numpy(d[k]).to(device=device, dtype=tdt).contiguous()
    for k in ("dt", "A", "D"):
        t[k] = torch.from_numpy(d[k]).to(device=device, dtype=torch.float32).contiguous()
    t["initial_state"] = (None if d.get("initial_state") is None else
                          torch.from_numpy(d["initial_state"]).to(device=device, dtype=torch.float32))
    t["cu_seqlens"] = (None if d.get("cu_seqlens") is None else
                       torch.from_numpy(np.asarray(d["cu_seqlens"], dtype=np.int32)).to(device))
    return t


def run_gpu(d: dict, dtype: str, chunk: int, use_D=True, return_final=True, scale_x_by_dt=False):
    import torch
    from mamba_ssd_layer_gb300 import binding as bd
    from mamba_ssd_layer_gb300 import ssd_forward
    t = to_device(d, dtype)
    x = t["x"]
    nseq = 0 if t["cu_seqlens"] is None else t["cu_seqlens"].shape[0] - 1
    ws_bytes = bd.ssd_workspace_size(x.shape[0], x.shape[1], x.shape[2], x.shape[3], t["B"].shape[3],
                                     t["B"].shape[2], bd.SSD_F32 if dtype == "f32" else bd.SSD_BF16, chunk, nseq)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    y, f = ssd_forward(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"] if use_D else None, chunk=chunk,
                       initial_state=t["initial_state"], cu_seqlens=t["cu_seqlens"],
                       return_final_state=return_final, workspace=ws, scale_x_by_dt=scale_x_by_dt)
    torch.cuda.synchronize()
    st = bd.ssd_status(ws)
    if st != bd.SSD_OK:
        hdr = ws[:16].cpu().numpy().view(np.int32)
        raise AssertionError(f"device status: {bd.ssd_status_string(st)}; header {hdr.tolist()}")
    return (y.float().cpu().numpy().astype(np.float64),
            None if f is None else f.cpu().numpy().astype(np.float64))


def run_oracle(d: dict, heads=None, use_D=True, scale_x_by_dt=False):
    x, dt, A, B, C, D, init = d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d.get("initial_state")
    if heads is not None:
        heads = np.asarray(heads)
        H = x.shape[2]
        G = B.shape[2]
        assert G == 1, "head sampling assumes one B/C group"
        x, dt, A, D = x[:, :, heads], dt[:, :, heads], A[heads], D[heads]
        if init is not None:
            init = init[:, heads]
        del H
    return oracle.ssd_recurrence(x, dt, A, B, C, D if use_D else None, init, d.get("cu_seqlens"),
                                 scale_x_by_dt=scale_x_by_dt)
