"""The block's output gate and extra normalization on the GPU (ssd_gated_rmsnorm) against the oracle
(oracle.gated_norm), through the C ABI: full-size token rows sampled, several group counts, in place, without
gate or weight, and the saturated ends of the gate."""
import numpy as np
import pytest

import oracle
from ssd_util import TOL, normwise

pytestmark = pytest.mark.gpu


def _data(batch, T, H, P, seed, zscale=1.0):
    import torch
    rng = np.random.default_rng(seed)
    y = torch.from_numpy(rng.standard_normal((batch, T, H, P), dtype=np.float32)).bfloat16()
    z = torch.from_numpy((zscale * rng.standard_normal((batch, T, H, P))).astype(np.float32)).bfloat16()
    w = torch.from_numpy(rng.uniform(0.5, 1.5, H * P).astype(np.float32))
    return y, z, w


def _check_rows(out, y, z, w, eps, groups, rows):
    yb, zb = y.float().numpy(), None if z is None else z.float().numpy()
    b, T, H, P = yb.shape
    flat = lambda a: a.reshape(b * T, H, P)[rows]
    ref = oracle.gated_rmsnorm(flat(yb), None if zb is None else flat(zb),
                               None if w is None else w.numpy(), eps=eps, groups=groups)
    got = out.float().cpu().numpy().reshape(b * T, H, P)[rows]
    assert normwise(got, ref) <= TOL["bf16"]
    return got, ref


@pytest.mark.parametrize("groups", [1, 8, 80])
def test_full_size_rows_match_the_oracle(groups):
    # a long-sequence layer's output: 16384 tokens of 80 heads x 64 channels
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(1, 16384, 80, 64, seed=500 + groups)
    out = ssd_gated_rmsnorm(y.cuda(), z.cuda(), w.cuda(), eps=1e-5, groups=groups)
    rows = np.random.default_rng(7).choice(16384, 256, replace=False)
    got, ref = _check_rows(out, y, z, w, 1e-5, groups, rows)
    # each output is the bf16 rounding of the exact value, within a few bf16 steps
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)) < 2e-2


def test_in_place_and_batch_rows():
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(3, 333, 8, 64, seed=510)
    yd, zd, wd = y.cuda(), z.cuda(), w.cuda()
    out = ssd_gated_rmsnorm(yd, zd, wd, eps=1e-6, groups=2)
    y2 = yd.clone()
    ssd_gated_rmsnorm(y2, zd, wd, eps=1e-6, groups=2, out=y2)
    assert np.array_equal(out.float().cpu().numpy(), y2.float().cpu().numpy())
    _check_rows(out, y, z, w, 1e-6, 2, np.arange(3 * 333))


def test_without_gate_or_weight():
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(2, 200, 4, 64, seed=520)
    out = ssd_gated_rmsnorm(y.cuda(), None, None, eps=1e-5, groups=1)
    _check_rows(out, y, None, None, 1e-5, 1, np.arange(400))


def test_saturated_gate():
    # z far below zero closes the gate (out = 0 exactly); far above zero it passes y * z
    import torch
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(1, 64, 4, 64, seed=530, zscale=60.0)
    out = ssd_gated_rmsnorm(y.cuda(), z.cuda(), w.cuda(), eps=1e-5)
    _check_rows(out, y, z, w, 1e-5, 1, np.arange(64))
    closed = ssd_gated_rmsnorm(y.cuda(), torch.full_like(z, -200.0).cuda(), w.cuda(), eps=1e-5)
    assert torch.count_nonzero(closed.float()).item() == 0


@pytest.mark.parametrize("groups", [1, 768])
def test_widest_token(groups):
    # 6144 channels a token (the most it takes), in one group or in 8-channel groups
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(1, 157, 96, 64, seed=540 + groups)
    out = ssd_gated_rmsnorm(y.cuda(), z.cuda(), w.cuda(), eps=1e-5, groups=groups)
    _check_rows(out, y, z, w, 1e-5, groups, np.arange(157))


@pytest.mark.parametrize("T,H,gated", [(16384, 80, True), (4099, 48, False), (37, 4, True)])
def test_host_form_equals_device_form(T, H, gated):
    # ssd_gated_rmsnorm_host: 16384 x 80 x 64 (168 MB of y) runs as a pipeline of row groups, the others in
    # one piece; either way the result is bit for bit the device form's, and out may be y itself
    import torch
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm, ssd_gated_rmsnorm_host
    y, z, w = _data(1, T, H, 64, seed=550 + H)
    zz = z if gated else None
    ref = ssd_gated_rmsnorm(y.cuda(), None if zz is None else zz.cuda(), w.cuda(), eps=1e-5, groups=H // 4 or 1)
    yh = y.pin_memory()
    got = ssd_gated_rmsnorm_host(yh, None if zz is None else zz.pin_memory(), w.pin_memory(), eps=1e-5,
                                 groups=H // 4 or 1, out=yh)
    assert got.data_ptr() == yh.data_ptr()
    assert torch.equal(got, ref.cpu())


# channel counts for every number of 8-channel pieces a thread holds (1 to 6 of 128 threads), most of them
# ragged, and group sizes that split a warp's 32 pieces unevenly (5 pieces), span two warps (64 pieces) or
# are the finest allowed (8 channels)
@pytest.mark.parametrize("H,P,groups", [(1, 64, 8), (20, 64, 32), (72, 32, 12), (64, 64, 64), (72, 64, 9),
                                        (88, 64, 88)])
def test_every_piece_count_and_ragged_groups(H, P, groups):
    from mamba_ssd_layer_gb300 import ssd_gated_rmsnorm
    y, z, w = _data(1, 1500, H, P, seed=560 + H + groups)
    out = ssd_gated_rmsnorm(y.cuda(), z.cuda(), w.cuda(), eps=1e-6, groups=groups)
    _check_rows(out, y, z, w, 1e-6, groups, np.arange(1500))
