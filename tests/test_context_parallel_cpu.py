"""Host logic of the sequence-parallel forward (mamba_ssd_layer_gb300.context_parallel) on the CPU:
the slices run one after another and as two gloo ranks, with per-slice steps written here in fp64
from their definitions, and the composed result must equal the oracle run over the whole sequence."""
import os
import socket
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(seed=7, batch=2, T=90, H=4, P=8, N=6, G=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, T, H, P))
    dt = np.log1p(np.exp(rng.standard_normal((batch, T, H)) - 1.0))
    A = -np.exp(rng.uniform(0.0, np.log(8.0), size=H))
    B = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    C = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    D = rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((batch, H, P, N))
    return x, dt, A, B, C, D, h0


def _cpu_ops():
    """fp64 per-slice steps: the forward is the oracle; the correction is its definition,
    y_l += exp(cs_l) C_l . h_in^T and final += exp(cs_last) h_in, cs_l the inclusive cumsum of dt*A."""
    import torch
    import oracle

    def forward(x, dt, A, B, C, D, init):
        y, fin = oracle.ssd_recurrence(x.numpy(), dt.numpy(), A.numpy(), B.numpy(), C.numpy(),
                                       None if D is None else D.numpy(),
                                       initial_state=None if init is None else init.numpy())
        return torch.from_numpy(y), torch.from_numpy(fin)

    def correct(dt, A, C, h_in, y, fin):
        dtn, An, Cn, h = dt.numpy(), A.numpy(), C.numpy(), h_in.numpy()
        H, G = An.shape[0], Cn.shape[2]
        cs = np.cumsum(dtn * An, axis=1)                                  # (batch, T, H)
        Ch = Cn[:, :, np.arange(H) // (H // G), :]                        # (batch, T, H, N)
        corr = np.einsum("bthn,bhpn->bthp", Ch, h) * np.exp(cs)[..., None]
        y += torch.from_numpy(corr)
        fin += torch.from_numpy(np.exp(cs[:, -1, :])[:, :, None, None] * h)

    return SimpleNamespace(forward=forward, correct=correct)


def _slices(arrs, cuts):
    x, dt, B, C = arrs
    import torch
    out = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        out.append(tuple(torch.from_numpy(np.ascontiguousarray(v[:, a:b])) for v in (x, dt, B, C)))
    return out


def test_slices_one_after_another_match_the_whole_sequence():
    import torch
    import oracle
    from mamba_ssd_layer_gb300.context_parallel import run_slices
    x, dt, A, B, C, D, h0 = _problem()
    cuts = [0, 17, 18, 60, 90]            # includes a one-token slice
    ys, fin = run_slices(_slices((x, dt, B, C), cuts), torch.from_numpy(A), torch.from_numpy(D),
                         torch.from_numpy(h0), ops=_cpu_ops())
    y_ref, fin_ref = oracle.ssd_recurrence(x, dt, A, B, C, D, initial_state=h0)
    np.testing.assert_allclose(torch.cat(ys, dim=1).numpy(), y_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(fin.numpy(), fin_ref, rtol=1e-11, atol=1e-11)


def test_planted_error_in_a_correction_is_seen():
    # the comparison above is not vacuous: a correction that drops the decay fails it
    import torch
    import oracle
    from mamba_ssd_layer_gb300.context_parallel import run_slices
    x, dt, A, B, C, D, h0 = _problem(seed=8)
    ops = _cpu_ops()
    good = ops.correct

    def bad(dt_, A_, C_, h_in, y, fin):
        good(dt_ * 0.0, A_, C_, h_in, y, fin)
    ops.correct = bad
    ys, fin = run_slices(_slices((x, dt, B, C), [0, 40, 90]), torch.from_numpy(A), torch.from_numpy(D),
                         torch.from_numpy(h0), ops=ops)
    y_ref, _ = oracle.ssd_recurrence(x, dt, A, B, C, D, initial_state=h0)
    assert np.max(np.abs(torch.cat(ys, dim=1).numpy() - y_ref)) > 1e-3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, cuts):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from mamba_ssd_layer_gb300.context_parallel import context_parallel_forward
    from test_context_parallel_cpu import _cpu_ops, _problem, _slices
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        x, dt, A, B, C, D, h0 = _problem()
        xs, dts, Bs, Cs = _slices((x, dt, B, C), cuts)[rank]
        y, fin = context_parallel_forward(xs, dts, torch.from_numpy(A), Bs, Cs, torch.from_numpy(D),
                                          initial_state=torch.from_numpy(h0) if rank == 0 else None,
                                          ops=_cpu_ops())
        np.save(os.path.join(out_dir, f"y{rank}.npy"), y.numpy())
        np.save(os.path.join(out_dir, f"f{rank}.npy"), fin.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [[0, 45, 90], [0, 1, 90]])
def test_two_gloo_ranks_hand_off_the_state(tmp_path, cuts):
    import torch.multiprocessing as mp
    import oracle
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), cuts), nprocs=world,
                       start_method="spawn")
    x, dt, A, B, C, D, h0 = _problem()
    y_ref, fin_ref = oracle.ssd_recurrence(x, dt, A, B, C, D, initial_state=h0)
    y = np.concatenate([np.load(tmp_path / f"y{r}.npy") for r in range(world)], axis=1)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.load(tmp_path / f"f{world - 1}.npy"), fin_ref, rtol=1e-11, atol=1e-11)
    # rank 0's final state is the state after its own slice
    _, fin0 = oracle.ssd_recurrence(x[:, :cuts[1]], dt[:, :cuts[1]], A, B[:, :cuts[1]], C[:, :cuts[1]], D,
                                    initial_state=h0)
    np.testing.assert_allclose(np.load(tmp_path / "f0.npy"), fin0, rtol=1e-11, atol=1e-11)
