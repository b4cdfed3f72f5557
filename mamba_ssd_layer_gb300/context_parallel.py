"""Sequence (context) parallel SSD forward: a sequence cut into consecutive slices, one per rank.

"LLM(十一)——Mamba" §3.7.2 (Sequence Parallelism): each worker runs its slice and passes its final
state to the next worker. Every rank runs its slice from a zero state (``ssd_forward``), which is
independent of the other ranks; then the state is handed along the ranks in order. Rank k receives
h_in from rank k - 1 and turns its local results into the true ones (``ssd_slice_correct``, by
linearity of the recurrence, "LLM(十一)——Mamba" §3.5.2):

    y_l   += exp(cs_l) C_l h_in^T          cs_l = sum of dt*A from the slice's first token through l
    final += exp(cs_last) h_in             (this is the h_in of rank k + 1)

Only one (batch, H, P, N) fp32 state crosses each rank boundary, copied into the receiver's own
memory by a point-to-point send/receive (NCCL between GPUs, gloo on the host): no remote loads and
no multicast. Rank 0 starts from the caller's initial state directly.

The per-slice device work comes from ``ops`` (default: the CUDA library through the binding); the
hand-off order does not depend on it, so the host logic can run on the CPU with other ops.
"""
from __future__ import annotations

from types import SimpleNamespace


def cuda_ops(chunk: int = 256):
    """The per-slice steps on the CUDA library: forward from a given (or zero) entering state, the
    slice's decay, and the correction for a nonzero entering state."""
    from . import binding as bd

    def forward(x, dt, A, B, C, D, initial_state):
        return bd.ssd_forward(x, dt, A, B, C, D, chunk=chunk, initial_state=initial_state)

    return SimpleNamespace(forward=forward, decay=bd.ssd_slice_decay, correct=bd.ssd_slice_correct)


def slice_step(x, dt, A, B, C, D, h_in, ops, first: bool):
    """One slice: its forward, then (except for the first slice, which starts from h_in directly) the
    correction for h_in. Returns (y, final) of the slice, final being the next slice's h_in."""
    if first:
        return ops.forward(x, dt, A, B, C, D, h_in)
    y, fin = ops.forward(x, dt, A, B, C, D, None)
    ops.correct(dt, A, C, h_in, y, fin)
    return y, fin


def run_slices(slices, A, D=None, initial_state=None, ops=None):
    """All slices of a sequence batch one after another on one device: ``slices`` is a list of
    (x, dt, B, C) with the same batch rows and consecutive token ranges. Returns the list of the slices'
    y and the final state of the last one (the same hand-off as across ranks, without the transport)."""
    ops = ops or cuda_ops()
    ys, h = [], initial_state
    for k, (x, dt, B, C) in enumerate(slices):
        if k > 0 and h is None:
            raise ValueError("a slice after the first needs the previous slice's final state")
        y, h = slice_step(x, dt, A, B, C, D, h, ops, first=(k == 0))
        ys.append(y)
    return ys, h


def context_parallel_forward(x, dt, A, B, C, D=None, initial_state=None, group=None, ops=None):
    """This rank's slice of a sequence parallel forward over the ranks of ``group`` (rank order =
    token order). x (batch, T_rank, H, P), dt, B, C likewise; A, D per head; initial_state (batch, H, P, N)
    is used by rank 0 only. Returns (y, final): this rank's outputs and the state after its slice (the
    sequence's final state on the last rank)."""
    import torch
    import torch.distributed as dist
    ops = ops or cuda_ops()
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if rank == 0:
        y, fin = ops.forward(x, dt, A, B, C, D, initial_state)
    else:
        # the slice's own work needs nothing from the other ranks; only the correction waits
        y, fin = ops.forward(x, dt, A, B, C, D, None)
        h_in = torch.empty_like(fin)
        dist.recv(h_in, src=_global_rank(group, rank - 1), group=group)
        ops.correct(dt, A, C, h_in, y, fin)
    if rank + 1 < world:
        dist.send(fin.contiguous(), dst=_global_rank(group, rank + 1), group=group)
    return y, fin


def _global_rank(group, group_rank: int) -> int:
    import torch.distributed as dist
    if group is None:
        return group_rank
    return dist.get_global_rank(group, group_rank)
