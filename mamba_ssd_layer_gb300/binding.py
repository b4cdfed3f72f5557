"""Thin Python binding of the SSD C ABI (``include/ssd.h``), via ctypes.

Argument marshalling only: every step of the forward pass runs in the CUDA
library. PyTorch supplies device memory and the current stream. If the library
has not been built, importing the entry points raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA, SSD_ERR_TIMEOUT, SSD_ERR_WORKSPACE = range(6)
SSD_F32, SSD_BF16 = 0, 1
SSD_SCALE_X_BY_DT = 1
# failure-detection test hook (include/ssd.h): cross-CTA waits of the bf16 path are made to run out
SSD_DEBUG_FORCE_TIMEOUT = 0x80000000

_lib = None


class SSDError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == SSD_ERR_CUDA:
            try:
                detail = load_library().ssd_last_error_detail().decode()
            except Exception:
                pass
        super().__init__(f"{where}: {ssd_status_string(code)} (code {code})" + (f" [{detail}]" if detail else ""))


class _Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64)]


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load ``_lib/libssd_gb300.so`` and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"SSD CUDA library not built ({path} missing); run mamba_ssd_layer_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, fp, sz, i32 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    shp = ctypes.POINTER(_Shape)
    lib.ssd_workspace_size.argtypes = [shp, i32, i32, i32]
    lib.ssd_workspace_size.restype = sz
    lib.ssd_host_buffer_size.argtypes = [shp, i32, i32, i32]
    lib.ssd_host_buffer_size.restype = sz
    fwd_args = [shp, i32, vp, fp, fp, vp, vp, fp, i32, fp, vp, i32, vp, fp, vp, sz, vp]
    lib.ssd_forward.argtypes = fwd_args
    lib.ssd_forward.restype = i32
    lib.ssd_forward_host.argtypes = fwd_args
    lib.ssd_forward_host.restype = i32
    fwd_ex_args = fwd_args[:2] + [ctypes.c_uint] + fwd_args[2:]
    lib.ssd_forward_ex.argtypes = fwd_ex_args
    lib.ssd_forward_ex.restype = i32
    lib.ssd_forward_host_ex.argtypes = fwd_ex_args
    lib.ssd_forward_host_ex.restype = i32
    dec_args = [shp, i32, vp, fp, fp, vp, vp, fp, fp, fp, vp, vp]
    lib.ssd_decode_step.argtypes = dec_args
    lib.ssd_decode_step.restype = i32
    lib.ssd_decode_step_ex.argtypes = [shp, i32, i32, ctypes.c_uint, vp, fp, fp, vp, vp, fp, vp, vp, vp, vp]
    lib.ssd_decode_step_ex.restype = i32
    lib.ssd_decode_host_buffer_size.argtypes = [shp, i32]
    lib.ssd_decode_host_buffer_size.restype = sz
    lib.ssd_decode_step_host.argtypes = dec_args[:-1] + [vp, sz, vp]
    lib.ssd_decode_step_host.restype = i32
    lib.ssd_decode_step_host_ex.argtypes = [shp, i32, i32, ctypes.c_uint, vp, fp, fp, vp, vp, fp, vp, vp, vp, vp, sz,
                                            vp]
    lib.ssd_decode_step_host_ex.restype = i32
    lib.ssd_slice_workspace_size.argtypes = [shp]
    lib.ssd_slice_workspace_size.restype = sz
    lib.ssd_slice_decay.argtypes = [shp, fp, fp, fp, vp, sz, vp]
    lib.ssd_slice_decay.restype = i32
    lib.ssd_slice_correct.argtypes = [shp, i32, fp, fp, vp, fp, vp, fp, vp, sz, vp]
    lib.ssd_slice_correct.restype = i32
    lib.ssd_gated_rmsnorm.argtypes = [shp, vp, vp, fp, ctypes.c_float, i32, vp, vp]
    lib.ssd_gated_rmsnorm.restype = i32
    lib.ssd_gated_rmsnorm_host_buffer_size.argtypes = [shp, i32]
    lib.ssd_gated_rmsnorm_host_buffer_size.restype = sz
    lib.ssd_gated_rmsnorm_host.argtypes = [shp, vp, vp, fp, ctypes.c_float, i32, vp, vp, sz, vp]
    lib.ssd_gated_rmsnorm_host.restype = i32
    lib.ssd_status.argtypes = [vp, vp]
    lib.ssd_status.restype = i32
    lib.ssd_profile_enable.argtypes = [i32]
    lib.ssd_profile_enable.restype = i32
    lib.ssd_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
    lib.ssd_profile_read.restype = i32
    lib.ssd_profile_kernel_launches.argtypes = []
    lib.ssd_profile_kernel_launches.restype = ctypes.c_longlong
    lib.ssd_profile_kernel_name.argtypes = []
    lib.ssd_profile_kernel_name.restype = ctypes.c_char_p
    lib.ssd_last_error_detail.argtypes = []
    lib.ssd_last_error_detail.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [i32]
    lib.ssd_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def ssd_status_string(code: int) -> str:
    return load_library().ssd_status_string(int(code)).decode()


def _shape(batch, seqlen, H, P, N, G) -> _Shape:
    return _Shape(int(batch), int(seqlen), int(H), int(P), int(N), int(G))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SSD_F32
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"x/B/C must be float32 or bfloat16, got {t.dtype}")


def ssd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, dtype_code, chunk, nseq=0) -> int:
    return int(load_library().ssd_workspace_size(ctypes.byref(_shape(batch, seqlen, nheads, headdim, dstate, ngroups)),
                                                 int(dtype_code), int(chunk), int(nseq)))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


def ssd_forward(x, dt, A, B, C, D=None, chunk: int = 256, initial_state=None, cu_seqlens=None,
                return_final_state: bool = True, y=None, final_state=None, workspace=None, stream=None,
                scale_x_by_dt: bool = False):
    """SSD forward through the C ABI on CUDA tensors (``ssd_forward_ex``).

    x (batch, T, H, P) and B, C (batch, T, G, N) in float32 or bfloat16 (the same);
    dt (batch, T, H), A (H,), D (H,) or None, initial_state (nseq, H, P, N) or None: float32.
    cu_seqlens: int32 (nseq + 1,) on the device, batch must be 1. Returns (y, final_state),
    final_state None when return_final_state is False. The work is enqueued on `stream`
    (default: torch's current stream); nothing is synchronised. ``scale_x_by_dt`` makes the input
    term dt x B^T (the skip term keeps D x).
    """
    import torch
    batch, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dev = x.device
    code = _dtype_code(x)
    _check(x, "x", (batch, T, H, P), x.dtype, dev)
    _check(dt, "dt", (batch, T, H), torch.float32, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(B, "B", (batch, T, G, N), x.dtype, dev)
    _check(C, "C", (batch, T, G, N), x.dtype, dev)
    _check(D, "D", (H,), torch.float32, dev)
    nseq = 0
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev:
            raise TypeError("cu_seqlens must be an int32 tensor on the same device")
        nseq = cu_seqlens.shape[0] - 1
    nseq_eff = nseq if cu_seqlens is not None else batch
    _check(initial_state, "initial_state", (nseq_eff, H, P, N), torch.float32, dev)
    if y is None:
        y = torch.empty_like(x)
    if return_final_state and final_state is None:
        final_state = torch.empty((nseq_eff, H, P, N), dtype=torch.float32, device=dev)
    shape = _shape(batch, T, H, P, N, G)
    lib = load_library()
    ws_bytes = int(lib.ssd_workspace_size(ctypes.byref(shape), code, int(chunk), int(nseq)))
    if ws_bytes == 0:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_workspace_size")
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    flags = SSD_SCALE_X_BY_DT if scale_x_by_dt else 0
    rc = lib.ssd_forward_ex(ctypes.byref(shape), code, flags, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                            int(chunk), _ptr(initial_state), _ptr(cu_seqlens), int(nseq), _ptr(y),
                            _ptr(final_state) if return_final_state else None,
                            workspace.data_ptr(), ws_bytes, ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_forward_ex")
    return y, (final_state if return_final_state else None)


def _slice_workspace(shape, dev, workspace):
    import torch
    lib = load_library()
    ws_bytes = int(lib.ssd_slice_workspace_size(ctypes.byref(shape)))
    if ws_bytes == 0:
        raise SSDError(SSD_ERR_INVALID_ARG, "ssd_slice_workspace_size")
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    return lib, workspace, ws_bytes


def ssd_slice_decay(dt, A, decay=None, workspace=None, stream=None):
    """exp(A[h] * sum_t dt[b, t, h]) per batch row and head (``ssd_slice_decay``): the decay a slice
    of a sequence applies to the state entering it. dt (batch, T, H), A (H,) float32 on the device.
    Returns decay (batch, H) float32."""
    import torch
    batch, T, H = dt.shape
    dev = dt.device
    _check(dt, "dt", (batch, T, H), torch.float32, dev)
    _check(A, "A", (H,), torch.float32, dev)
    if decay is None:
        decay = torch.empty((batch, H), dtype=torch.float32, device=dev)
    _check(decay, "decay", (batch, H), torch.float32, dev)
    shape = _shape(batch, T, H, 1, 1, 1)
    lib, workspace, ws_bytes = _slice_workspace(shape, dev, workspace)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.ssd_slice_decay(ctypes.byref(shape), _ptr(dt), _ptr(A), _ptr(decay), workspace.data_ptr(), ws_bytes,
                             ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_slice_decay")
    return decay


def ssd_slice_correct(dt, A, C, h_in, y, final_state=None, workspace=None, stream=None):
    """Turn a slice's zero-state outputs into the true ones given the state h_in entering it
    (``ssd_slice_correct``): y += exp(cs_l) C_l h_in^T in place (bf16), and final_state += decay h_in
    when given. dt (batch, T, H), A (H,), h_in and final_state (batch, H, P, N) float32; C (batch, T, G, N)
    and y (batch, T, H, P) bfloat16. Returns (y, final_state)."""
    import torch
    batch, T, H, P = y.shape
    G, N = C.shape[2], C.shape[3]
    dev = y.device
    _check(y, "y", (batch, T, H, P), torch.bfloat16, dev)
    _check(dt, "dt", (batch, T, H), torch.float32, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(C, "C", (batch, T, G, N), torch.bfloat16, dev)
    _check(h_in, "h_in", (batch, H, P, N), torch.float32, dev)
    _check(final_state, "final_state", (batch, H, P, N), torch.float32, dev)
    shape = _shape(batch, T, H, P, N, G)
    lib, workspace, ws_bytes = _slice_workspace(shape, dev, workspace)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.ssd_slice_correct(ctypes.byref(shape), SSD_BF16, _ptr(dt), _ptr(A), _ptr(C), _ptr(h_in), _ptr(y),
                               _ptr(final_state), workspace.data_ptr(), ws_bytes, ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_slice_correct")
    return y, final_state


def ssd_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status word of `workspace`."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return int(load_library().ssd_status(workspace.data_ptr(), ctypes.c_void_p(stream.cuda_stream)))


def ssd_forward_host(x, dt, A, B, C, D=None, chunk: int = 256, initial_state=None, cu_seqlens=None,
                     return_final_state: bool = True, y=None, final_state=None, device_buffer=None,
                     stream=None, scale_x_by_dt: bool = False):
    """The same forward pass on HOST (CPU, ideally pinned) tensors through ``ssd_forward_host``:
    host->device copies, the kernels and the device->host copies all happen inside the C call,
    which synchronises the stream before returning."""
    import torch
    batch, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    code = _dtype_code(x)
    cpu = torch.device("cpu")
    for t, name in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C"), (D, "D"), (initial_state, "initial_state"),
                    (cu_seqlens, "cu_seqlens")):
        if t is not None and (t.device != cpu or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    nseq = 0 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    nseq_eff = nseq if cu_seqlens is not None else batch
    if y is None:
        y = torch.empty_like(x)
    if return_final_state and final_state is None:
        final_state = torch.empty((nseq_eff, H, P, N), dtype=torch.float32)
    shape = _shape(batch, T, H, P, N, G)
    lib = load_library()
    need = int(lib.ssd_host_buffer_size(ctypes.byref(shape), code, int(chunk), int(nseq)))
    if need == 0:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_host_buffer_size")
    if device_buffer is None or device_buffer.numel() < need:
        device_buffer = torch.empty(need, dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream(device_buffer.device)
    flags = SSD_SCALE_X_BY_DT if scale_x_by_dt else 0
    rc = lib.ssd_forward_host_ex(ctypes.byref(shape), code, flags, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(D), int(chunk), _ptr(initial_state), _ptr(cu_seqlens), int(nseq), _ptr(y),
                                 _ptr(final_state) if return_final_state else None,
                                 device_buffer.data_ptr(), need, ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_forward_host_ex")
    return y, (final_state if return_final_state else None)


def _decode_shapes(x, B):
    batch, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    return batch, H, P, G, N


def ssd_decode_step(x, dt, A, B, C, D=None, state=None, new_state=None, y=None, stream=None,
                    scale_x_by_dt: bool = False):
    """One recurrent step on CUDA tensors through ``ssd_decode_step``.

    x (batch, H, P) and B, C (batch, G, N) in float32 or bfloat16 (the same); dt (batch, H),
    A (H,), D (H,) or None: float32; state (batch, H, P, N) float32, or bfloat16 for a state stored
    in bf16 (``ssd_decode_step_ex``). new_state defaults to ``state`` (updated in place); pass
    another tensor of the state's dtype to keep ``state``. Returns (y, new_state); the work is
    enqueued on `stream` (default: torch's current stream) and nothing is synchronised.
    """
    import torch
    batch, H, P, G, N = _decode_shapes(x, B)
    dev = x.device
    code = _dtype_code(x)
    _check(x, "x", (batch, H, P), x.dtype, dev)
    _check(dt, "dt", (batch, H), torch.float32, dev)
    _check(A, "A", (H,), torch.float32, dev)
    _check(B, "B", (batch, G, N), x.dtype, dev)
    _check(C, "C", (batch, G, N), x.dtype, dev)
    _check(D, "D", (H,), torch.float32, dev)
    if state is None:
        raise ValueError("state is required")
    state_code = _dtype_code(state)
    _check(state, "state", (batch, H, P, N), state.dtype, dev)
    if new_state is None:
        new_state = state
    _check(new_state, "new_state", (batch, H, P, N), state.dtype, dev)
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", (batch, H, P), x.dtype, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    flags = SSD_SCALE_X_BY_DT if scale_x_by_dt else 0
    rc = load_library().ssd_decode_step_ex(ctypes.byref(_shape(batch, 1, H, P, N, G)), code, state_code, flags, _ptr(x),
                                           _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state),
                                           _ptr(new_state), _ptr(y), ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_decode_step_ex")
    return y, new_state


def ssd_decode_step_host(x, dt, A, B, C, D=None, state=None, new_state=None, y=None, device_buffer=None,
                         stream=None, scale_x_by_dt: bool = False):
    """The same step on HOST (CPU, ideally pinned) tensors through ``ssd_decode_step_host``: the
    copies in, the kernel and the copies out all happen inside the C call, which synchronises."""
    import torch
    batch, H, P, G, N = _decode_shapes(x, B)
    code = _dtype_code(x)
    cpu = torch.device("cpu")
    if state is None:
        raise ValueError("state is required")
    for t, name in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C"), (D, "D"), (state, "state")):
        if t is not None and (t.device != cpu or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if new_state is None:
        new_state = state
    if y is None:
        y = torch.empty_like(x)
    shape = _shape(batch, 1, H, P, N, G)
    lib = load_library()
    need = int(lib.ssd_decode_host_buffer_size(ctypes.byref(shape), code))
    if need == 0:
        raise SSDError(SSD_ERR_UNSUPPORTED, "ssd_decode_host_buffer_size")
    if device_buffer is None or device_buffer.numel() < need:
        device_buffer = torch.empty(need, dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream(device_buffer.device)
    flags = SSD_SCALE_X_BY_DT if scale_x_by_dt else 0
    rc = lib.ssd_decode_step_host_ex(ctypes.byref(shape), code, _dtype_code(state), flags, _ptr(x), _ptr(dt), _ptr(A),
                                     _ptr(B), _ptr(C), _ptr(D), _ptr(state), _ptr(new_state), _ptr(y),
                                     device_buffer.data_ptr(), need, ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_decode_step_host_ex")
    return y, new_state


def profile_enable(on: bool = True) -> None:
    """Record CUDA events around the dominant kernel of every later ssd_forward, ssd_decode_step or
    ssd_gated_rmsnorm on this thread."""
    load_library().ssd_profile_enable(1 if on else 0)


def profile_read():
    """(summed milliseconds, launches) of the dominant kernel since the last read; resets."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int(0)
    rc = load_library().ssd_profile_read(ctypes.byref(ms), ctypes.byref(n))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_profile_read")
    return ms.value, n.value


def profile_kernel_launches() -> int:
    """Kernels the library launched on this thread since recording was last enabled."""
    return int(load_library().ssd_profile_kernel_launches())


def profile_kernel_name() -> str:
    """Name of the kernel the recorded events bracket."""
    return load_library().ssd_profile_kernel_name().decode()


def ssd_gated_rmsnorm(y, z=None, weight=None, eps: float = 1e-5, groups: int = 1, out=None, stream=None):
    """The block's output gate and extra normalization (``ssd_gated_rmsnorm``): per token and group of
    H*P/groups channels, v = y * silu(z) (no gate when z is None), out = v / sqrt(mean(v^2) + eps) * weight.
    y, z, out (batch, T, H, P) bfloat16 on the device (out may be y); weight (H*P,) float32 or None.
    Returns out."""
    import torch
    batch, T, H, P = y.shape
    dev = y.device
    _check(y, "y", (batch, T, H, P), torch.bfloat16, dev)
    _check(z, "z", (batch, T, H, P), torch.bfloat16, dev)
    _check(weight, "weight", (H * P,), torch.float32, dev)
    if out is None:
        out = torch.empty_like(y)
    _check(out, "out", (batch, T, H, P), torch.bfloat16, dev)
    shape = _shape(batch, T, H, P, 1, 1)
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.ssd_gated_rmsnorm(ctypes.byref(shape), _ptr(y), _ptr(z), _ptr(weight), float(eps), int(groups),
                               _ptr(out), ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_gated_rmsnorm")
    return out


def ssd_gated_rmsnorm_host(y, z=None, weight=None, eps: float = 1e-5, groups: int = 1, out=None, device_buffer=None,
                           stream=None):
    """The same on HOST (CPU, ideally pinned) tensors through ``ssd_gated_rmsnorm_host``: the copies in, the
    kernel and the copy out all happen inside the C call, which synchronises. Returns out."""
    import torch
    batch, T, H, P = y.shape
    cpu = torch.device("cpu")
    _check(y, "y", (batch, T, H, P), torch.bfloat16, cpu)
    _check(z, "z", (batch, T, H, P), torch.bfloat16, cpu)
    _check(weight, "weight", (H * P,), torch.float32, cpu)
    if out is None:
        out = torch.empty_like(y)
    _check(out, "out", (batch, T, H, P), torch.bfloat16, cpu)
    shape = _shape(batch, T, H, P, 1, 1)
    lib = load_library()
    need = int(lib.ssd_gated_rmsnorm_host_buffer_size(ctypes.byref(shape), 1 if z is not None else 0))
    if need == 0:
        raise SSDError(SSD_ERR_INVALID_ARG, "ssd_gated_rmsnorm_host_buffer_size")
    if device_buffer is None or device_buffer.numel() < need:
        device_buffer = torch.empty(need, dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream(device_buffer.device)
    rc = lib.ssd_gated_rmsnorm_host(ctypes.byref(shape), _ptr(y), _ptr(z), _ptr(weight), float(eps), int(groups),
                                    _ptr(out), device_buffer.data_ptr(), need, ctypes.c_void_p(stream.cuda_stream))
    if rc != SSD_OK:
        raise SSDError(rc, "ssd_gated_rmsnorm_host")
    return out
