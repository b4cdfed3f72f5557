"""Oracle for the SSD layer forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
never calls the CUDA library.

Two independent formulations live here:

* :func:`ssd_recurrence` -- the fp64 token-by-token recurrence
  ``h_t = a_t h_{t-1} + x_t B_t^T``, ``y_t = h_t C_t + D x_t`` in plain C
  (``ssd_oracle.c``), threaded over (sequence, head). This is the oracle the
  GPU path is compared against.
* :func:`ssd_quadratic` (``quadratic.py``) -- the dual "attention" form
  ``Y = (L o C B^T) X + D X`` with the 1-semiseparable mask materialised as a
  T x T matrix, in numpy. It is used to pin the recurrence on tiny inputs.
* :func:`ssd_decode_step` (``decode.py``) -- one token of the recurrence on a
  batch of carried states (the recurrent inference step), in numpy fp64.

The C file is compiled with the system ``gcc`` into ``oracle/_build`` the first
time it is needed (or by ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .decode import ssd_decode_step  # noqa: F401
from .gated_norm import gated_rmsnorm, silu  # noqa: F401
from .quadratic import ssd_quadratic  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssd_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libssd_oracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.ssd_oracle_f64.argtypes = [i64, i64, i64, i64, i64, i64,
                                           dp, dp, dp, dp, dp, dp, dp,
                                           ctypes.POINTER(ctypes.c_int32), i64,
                                           dp, dp, ctypes.c_int]
            lib.ssd_oracle_f64.restype = ctypes.c_int
            lib.ssd_oracle_f64_ex.argtypes = [i64, i64, i64, i64, i64, i64,
                                              dp, dp, dp, dp, dp, dp, dp,
                                              ctypes.POINTER(ctypes.c_int32), i64,
                                              dp, dp, ctypes.c_int, ctypes.c_int]
            lib.ssd_oracle_f64_ex.restype = ctypes.c_int
            lib.ssd_oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().ssd_oracle_default_threads())


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def ssd_recurrence(x, dt, A, B, C, D=None, initial_state=None, cu_seqlens=None,
                   nthreads: int = 0, return_final: bool = True, scale_x_by_dt: bool = False):
    """fp64 recurrence. Shapes follow the library's call:

    x (batch, T, H, P); dt (batch, T, H); A (H,); B, C (batch, T, G, N); D (H,) or None;
    initial_state (nseq, H, P, N) or None; cu_seqlens (nseq+1,) int32 or None (then batch == 1
    is required and the row is split into sequences at those offsets).

    Returns ``(y, final_state)`` as float64 arrays; ``y`` has x's shape and
    ``final_state`` is (nseq, H, P, N), nseq = batch for a dense call. With ``scale_x_by_dt`` the
    input term is ``dt_t x_t (outer) B_t`` (the skip term keeps ``D x_t``).
    """
    x, dt, A, B, C, D, init = (_f64(v) for v in (x, dt, A, B, C, D, initial_state))
    batch, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt.shape == (batch, T, H) and A.shape == (H,)
    assert B.shape == (batch, T, G, N) and C.shape == B.shape
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        nseq = cu.shape[0] - 1
        assert batch == 1
    else:
        cu, nseq = None, batch
    if init is not None:
        assert init.shape == (nseq, H, P, N)
    y = np.empty_like(x)
    final = np.empty((nseq, H, P, N), dtype=np.float64) if return_final else None
    rc = _load().ssd_oracle_f64_ex(batch, T, H, P, N, G,
                                   _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(init),
                                   _ptr(cu, ctypes.c_int32), nseq, _ptr(y), _ptr(final), 1 if scale_x_by_dt else 0,
                                   int(nthreads))
    if rc != 0:
        raise RuntimeError(f"ssd_oracle_f64 failed with code {rc}")
    return y, final
