"""C-ABI checks that need no GPU: the library builds, loads, exports every entry point the
header declares, sizes workspaces, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from mamba_ssd_layer_gb300 import build as B
from mamba_ssd_layer_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return bd.load_library()


def header_functions():
    inc = os.path.join(ROOT, "include")
    txt = "\n".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char)\s*\*?\s*(ssd_\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_entry_points():
    names = header_functions()
    assert {"ssd_forward", "ssd_workspace_size", "ssd_status", "ssd_status_string",
            "ssd_forward_host", "ssd_host_buffer_size"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def shape(batch=1, T=256, H=4, P=64, N=128, G=1):
    return bd._Shape(batch, T, H, P, N, G)


def test_workspace_size(lib):
    s = shape(batch=2, T=1000, H=4, P=64, N=128)
    ws = lib.ssd_workspace_size(ctypes.byref(s), bd.SSD_BF16, 256, 0)
    chunks = 2 * 4  # ceil(1000/256) per row
    assert ws >= chunks * 4 * 64 * 128 * 4
    # varlen bound: ceil(rows/Q) + nseq chunks
    s1 = shape(batch=1, T=1000)
    wv = lib.ssd_workspace_size(ctypes.byref(s1), bd.SSD_BF16, 256, 5)
    assert wv >= (4 + 5) * 4 * 64 * 128 * 4
    # unsupported chunk / shapes give 0
    assert lib.ssd_workspace_size(ctypes.byref(s), bd.SSD_BF16, 100, 0) == 0
    assert lib.ssd_workspace_size(ctypes.byref(shape(P=32)), bd.SSD_BF16, 256, 0) == 0
    assert lib.ssd_workspace_size(ctypes.byref(shape(H=3, G=2)), bd.SSD_F32, 64, 0) == 0
    assert lib.ssd_workspace_size(ctypes.byref(shape(P=16, N=16)), bd.SSD_F32, 64, 0) > 0


def test_status_strings(lib):
    for code in range(6):
        assert isinstance(bd.ssd_status_string(code), str) and bd.ssd_status_string(code)
    assert bd.ssd_status_string(99) == "unknown status"


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every case below fails host-side checks


def call(lib, s, dtype=bd.SSD_BF16, chunk=256, x=FAKE, ws=FAKE, ws_bytes=1 << 40, cu=None, nseq=0, A=FAKE):
    return lib.ssd_forward(ctypes.byref(s), dtype, x, FAKE, A, FAKE, FAKE, None, chunk, None, cu, nseq,
                           FAKE, None, ws, ws_bytes, None)


def test_argument_errors_before_any_device_work(lib):
    s = shape()
    assert call(lib, shape(H=3, G=2)) == bd.SSD_ERR_INVALID_ARG            # H % G
    assert call(lib, s, chunk=100) == bd.SSD_ERR_UNSUPPORTED                 # chunk
    assert call(lib, shape(P=32)) == bd.SSD_ERR_UNSUPPORTED                  # bf16 needs P == 64
    assert call(lib, shape(N=96)) == bd.SSD_ERR_UNSUPPORTED
    assert call(lib, s, x=FAKE + 2) == bd.SSD_ERR_INVALID_ARG                # misaligned
    assert call(lib, s, x=None) == bd.SSD_ERR_INVALID_ARG                    # NULL input
    assert call(lib, s, A=None) == bd.SSD_ERR_INVALID_ARG
    assert call(lib, s, ws=None) == bd.SSD_ERR_WORKSPACE
    assert call(lib, s, ws=FAKE + 16) == bd.SSD_ERR_WORKSPACE               # not 256-aligned
    assert call(lib, s, ws_bytes=16) == bd.SSD_ERR_WORKSPACE
    assert call(lib, shape(batch=2), cu=FAKE, nseq=2) == bd.SSD_ERR_INVALID_ARG  # varlen needs batch 1
    assert call(lib, s, cu=FAKE, nseq=0) == bd.SSD_ERR_INVALID_ARG
    assert call(lib, s, dtype=7) == bd.SSD_ERR_INVALID_ARG


def test_no_gpu_reports_cuda_or_unsupported(lib):
    # valid arguments on a machine without a usable sm_103 device: an error code, never a crash
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    s = shape()
    rc = call(lib, s)
    assert rc in (bd.SSD_ERR_CUDA, bd.SSD_ERR_UNSUPPORTED)


def dcall(lib, s, dtype=bd.SSD_BF16, x=FAKE, state=FAKE, new_state=FAKE, B=FAKE):
    return lib.ssd_decode_step(ctypes.byref(s), dtype, x, FAKE, FAKE, B, FAKE, None, state, new_state, FAKE, None)


def test_decode_argument_errors_before_any_device_work(lib):
    s = shape(batch=4, T=1)
    assert dcall(lib, shape(batch=4, T=2)) == bd.SSD_ERR_INVALID_ARG          # one token per row
    assert dcall(lib, shape(batch=4, T=1, H=3, G=2)) == bd.SSD_ERR_INVALID_ARG   # H % G
    assert dcall(lib, shape(batch=4, T=1, N=18)) == bd.SSD_ERR_UNSUPPORTED    # N % 4
    assert dcall(lib, shape(batch=4, T=1, N=260)) == bd.SSD_ERR_UNSUPPORTED
    assert dcall(lib, shape(batch=4, T=1, P=300)) == bd.SSD_ERR_UNSUPPORTED
    assert dcall(lib, s, x=None) == bd.SSD_ERR_INVALID_ARG
    assert dcall(lib, s, state=FAKE + 8) == bd.SSD_ERR_INVALID_ARG            # state not 16-byte aligned
    assert dcall(lib, s, B=FAKE + 8) == bd.SSD_ERR_INVALID_ARG
    assert dcall(lib, s, new_state=FAKE + 16) == bd.SSD_ERR_INVALID_ARG       # partial overlap with state
    assert dcall(lib, s, dtype=7) == bd.SSD_ERR_INVALID_ARG
    assert dcall(lib, shape(batch=0, T=1)) == bd.SSD_OK                       # nothing to do
    assert lib.ssd_decode_host_buffer_size(ctypes.byref(shape(batch=4, T=1, N=18)), bd.SSD_BF16) == 0
    need = lib.ssd_decode_host_buffer_size(ctypes.byref(s), bd.SSD_BF16)
    assert need >= 4 * 4 * 64 * 128 * 4                                        # holds the state
    rc = lib.ssd_decode_step_host(ctypes.byref(s), bd.SSD_BF16, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                                  FAKE, FAKE, 16, None)
    assert rc == bd.SSD_ERR_WORKSPACE


def test_decode_state_dtype_errors(lib):
    s = shape(batch=4, T=1)
    call = lambda sh, sd, fl=0: lib.ssd_decode_step_ex(ctypes.byref(sh), bd.SSD_BF16, sd, fl, FAKE, FAKE, FAKE, FAKE,
                                                        FAKE, None, FAKE, FAKE, FAKE, None)
    assert call(s, 7) == bd.SSD_ERR_INVALID_ARG                                # unknown state type
    assert call(shape(batch=4, T=1, N=20), bd.SSD_BF16) == bd.SSD_ERR_UNSUPPORTED   # bf16 state: N % 8
    assert call(shape(batch=0, T=1), bd.SSD_BF16) == bd.SSD_OK
    assert call(s, bd.SSD_F32, 6) == bd.SSD_ERR_INVALID_ARG                    # unknown flag bits
    rc = lib.ssd_decode_step_host_ex(ctypes.byref(s), bd.SSD_BF16, 7, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                     FAKE, FAKE, FAKE, 1 << 40, None)
    assert rc == bd.SSD_ERR_INVALID_ARG


def test_forward_flag_errors(lib):
    s = shape()
    ex = lambda fl: lib.ssd_forward_ex(ctypes.byref(s), bd.SSD_BF16, fl, FAKE, FAKE, FAKE, FAKE, FAKE, None, 256,
                                       None, None, 0, FAKE, None, FAKE, 1 << 40, None)
    assert ex(2) == bd.SSD_ERR_INVALID_ARG
    assert ex(0x40000000) == bd.SSD_ERR_INVALID_ARG
    # the failure-detection test hook is a known flag: the call gets past the flag check
    assert ex(bd.SSD_DEBUG_FORCE_TIMEOUT) != bd.SSD_ERR_INVALID_ARG
    rc = lib.ssd_forward_host_ex(ctypes.byref(s), bd.SSD_BF16, 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, 256, None,
                                 None, 0, FAKE, None, FAKE, 1 << 40, None)
    assert rc == bd.SSD_ERR_INVALID_ARG


def test_slice_handoff_argument_errors_before_any_device_work(lib):
    s = shape(batch=2, T=300, H=4, P=64, N=128)
    ws = lib.ssd_slice_workspace_size(ctypes.byref(s))
    assert ws >= 256 + 2 * 3 * 4 * 4 + 2 * 4 * 4        # header, tile sums, decays
    assert lib.ssd_slice_workspace_size(ctypes.byref(shape(H=3, G=2))) == 0
    dec = lambda sh, A=FAKE, out=FAKE, w=FAKE, wb=1 << 30: lib.ssd_slice_decay(ctypes.byref(sh), FAKE, A, out, w, wb,
                                                                             None)
    assert dec(s, A=None) == bd.SSD_ERR_INVALID_ARG
    assert dec(s, out=FAKE + 4) == bd.SSD_ERR_INVALID_ARG
    assert dec(s, w=FAKE + 16) == bd.SSD_ERR_WORKSPACE
    assert dec(s, wb=16) == bd.SSD_ERR_WORKSPACE
    cor = lambda sh, dtype=bd.SSD_BF16, h=FAKE, y=FAKE: lib.ssd_slice_correct(ctypes.byref(sh), dtype, FAKE, FAKE,
                                                                              FAKE, h, y, None, FAKE, 1 << 30, None)
    assert cor(s, dtype=bd.SSD_F32) == bd.SSD_ERR_UNSUPPORTED
    assert cor(shape(batch=2, T=300, H=4, P=32, N=128)) == bd.SSD_ERR_UNSUPPORTED
    assert cor(s, dtype=7) == bd.SSD_ERR_INVALID_ARG
    assert cor(s, h=None) == bd.SSD_ERR_INVALID_ARG
    assert cor(s, y=FAKE + 2) == bd.SSD_ERR_INVALID_ARG


def test_gated_rmsnorm_argument_errors_before_any_device_work(lib):
    s = shape(batch=2, T=100, H=4, P=64, N=128)
    norm = lambda sh, y=FAKE, z=FAKE, w=FAKE, eps=1e-5, groups=1, out=FAKE: lib.ssd_gated_rmsnorm(
        ctypes.byref(sh), y, z, w, eps, groups, out, None)
    assert norm(s, groups=0) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, groups=3) == bd.SSD_ERR_INVALID_ARG              # 256 channels are not 3 groups
    assert norm(s, groups=64) == bd.SSD_ERR_UNSUPPORTED             # a group of 4 channels: not 16-byte pieces
    assert norm(shape(batch=1, T=4, H=98, P=64, N=128)) == bd.SSD_ERR_UNSUPPORTED    # 6272 channels a token
    assert norm(s, eps=-1.0) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, eps=float("nan")) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, y=None) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, out=None) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, z=FAKE + 8) == bd.SSD_ERR_INVALID_ARG
    assert norm(s, w=FAKE + 4) == bd.SSD_ERR_INVALID_ARG
    assert norm(shape(batch=0, T=100, H=4, P=64, N=128), y=None, out=None) == bd.SSD_OK   # nothing to do


def test_gated_rmsnorm_host_buffer_and_argument_errors(lib):
    s = shape(batch=2, T=100, H=4, P=64, N=128)
    size = lambda sh, gated: lib.ssd_gated_rmsnorm_host_buffer_size(ctypes.byref(sh), gated)
    # y (and z when gated) of 200 tokens x 256 bf16 channels, 256-byte aligned, then the fp32 weight
    assert size(s, 0) == 200 * 256 * 2 + 256 * 4
    assert size(s, 1) == 2 * 200 * 256 * 2 + 256 * 4
    assert size(shape(batch=1, T=3, H=1, P=64), 1) == 2 * 512 + 256
    assert size(shape(batch=-1), 1) == 0
    need = size(s, 1)
    host = lambda sh, y=FAKE, z=FAKE, w=FAKE, eps=1e-5, groups=1, out=FAKE, buf=FAKE, nb=need: \
        lib.ssd_gated_rmsnorm_host(ctypes.byref(sh), y, z, w, eps, groups, out, buf, nb, None)
    assert host(s, buf=None) == bd.SSD_ERR_WORKSPACE
    assert host(s, buf=FAKE + 16) == bd.SSD_ERR_WORKSPACE                # not 256-aligned
    assert host(s, nb=need - 1) == bd.SSD_ERR_WORKSPACE
    assert host(s, groups=3) == bd.SSD_ERR_INVALID_ARG
    assert host(s, groups=64) == bd.SSD_ERR_UNSUPPORTED
    assert host(s, eps=-1.0) == bd.SSD_ERR_INVALID_ARG
    assert host(s, y=None) == bd.SSD_ERR_INVALID_ARG
    assert host(s, out=None) == bd.SSD_ERR_INVALID_ARG
    assert host(shape(batch=0, T=100, H=4, P=64, N=128), y=None, out=None) == bd.SSD_OK   # nothing to do
