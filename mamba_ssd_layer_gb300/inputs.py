"""Seeded synthetic inputs for the SSD layer (shared by tests, bench and smoke).

This module only draws random numbers and rounds them to the storage type; it
holds none of the layer's arithmetic, so both the oracle side and the CUDA side
may use it without sharing any of the method.

Distributions (all workloads): x ~ N(0, 1); dt = softplus(N(0, 1) - 2) (> 0);
A = -exp(U(ln 1, ln 16)) per head (so A in [-16, -1]); B, C ~ N(0, std 1/sqrt(N));
D ~ N(0, 1) per head; a nonzero initial state, where used, ~ N(0, std 0.1).
Draw order: x, dt, A, B, C, D, segment lengths, initial state. Generator:
numpy PCG64 with the workload's seed. For bf16 workloads x, B, C are rounded
to bf16 (round-to-nearest-even) once, and both sides consume those values.

The output gate and normalization workloads (norm_groups > 0) draw y ~ N(0, 1) (the layer's output),
z ~ N(0, 1) (the gate branch), both rounded to bf16, and the scale weight ~ U(0.5, 1.5) per channel, fp32;
draw order y, z, weight.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk: int
    dtype: str               # "f32" or "bf16": storage type of x, B, C and y
    seed: int
    init_state: bool = False  # draw a nonzero initial state
    varlen_total: int = 0     # >0: one packed row of this many tokens, split into segments
    seg_min: int = 64
    seg_max: int = 4096
    state_dtype: str = "f32"  # recurrent-step workloads: storage type of the carried state
    scale_x_by_dt: bool = False  # the input term is dt x B^T (the layer's option, not an input draw)
    norm_groups: int = 0      # >0: an output gate and normalization workload with this many groups per token
    note: str = field(default="", compare=False)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The forward workloads: tiny fp32, Mamba-2-130M-shaped, Mamba-2-2.7B-shaped, long sequence with
# a state-size sweep, and a variable-length packed batch; and one recurrent-step workload.
WORKLOADS = {
    "fp32_tiny": Workload("fp32_tiny", 1, 256, 2, 16, 16, 1, 64, "f32", 1000),
    "m2_130m": Workload("m2_130m", 8, 2048, 24, 64, 128, 1, 256, "bf16", 1001),
    "m2_2p7b": Workload("m2_2p7b", 4, 4096, 80, 64, 128, 1, 256, "bf16", 1002, init_state=True),
    "long_n64": Workload("long_n64", 1, 16384, 80, 64, 64, 1, 256, "bf16", 1003 + 64),
    "long_n128": Workload("long_n128", 1, 16384, 80, 64, 128, 1, 256, "bf16", 1003 + 128),
    "long_n256": Workload("long_n256", 1, 16384, 80, 64, 256, 1, 256, "bf16", 1003 + 256),
    # the long-sequence layer with the dt-scaled input term (same draws as long_n128)
    "long_n128_dtscaled": Workload("long_n128_dtscaled", 1, 16384, 80, 64, 128, 1, 256, "bf16", 1003 + 128,
                                   scale_x_by_dt=True),
    "varlen": Workload("varlen", 1, 32768, 32, 64, 128, 1, 256, "bf16", 1004, varlen_total=32768),
    # one recurrent step for 64 carried states of a Mamba-2-2.7B-shaped layer (seqlen 1; the
    # initial state is the carried state)
    "decode_2p7b": Workload("decode_2p7b", 64, 1, 80, 64, 128, 1, 256, "bf16", 1005, init_state=True),
    # the same step with the carried state stored in bf16 (the state is rounded to bf16 once on the host)
    "decode_2p7b_bf16state": Workload("decode_2p7b_bf16state", 64, 1, 80, 64, 128, 1, 256, "bf16", 1005,
                                      init_state=True, state_dtype="bf16"),
    # the block's output gate and normalization over the long-sequence layer's output (16384 tokens of
    # 80 heads x 64 channels), one RMSNorm group per token (dstate, ngroups and chunk are unused)
    "gated_norm_long": Workload("gated_norm_long", 1, 16384, 80, 64, 128, 1, 256, "bf16", 1006, norm_groups=1),
}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # finite values stay below 2**32 after adding the rounding bias; NaN is restored below
    r = ((u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16) << 16
    nan = np.isnan(a)
    out = r.astype(np.uint32).view(np.float32)
    if nan.any():
        out = out.copy()
        out[nan] = np.float32("nan")
    return out.reshape(a.shape)


def segment_lengths(rng: np.random.Generator, total: int, lo: int, hi: int) -> np.ndarray:
    """Lengths drawn uniformly from [lo, hi] until they reach `total`; the last is clipped."""
    lens = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return np.asarray(lens, dtype=np.int64)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw one workload's inputs.

    Returns a dict of numpy arrays: x (batch, T, H, P), dt (batch, T, H), A (H,),
    B, C (batch, T, G, N), D (H,) -- all fp32 (x, B, C hold bf16-representable values
    when w.dtype == "bf16") -- plus initial_state (nseq, H, P, N) fp32 or None and
    cu_seqlens (nseq + 1,) int32 or None.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    T = w.varlen_total if w.varlen_total else w.seqlen
    batch = 1 if w.varlen_total else w.batch
    H, P, N, G = w.nheads, w.headdim, w.dstate, w.ngroups
    x = rng.standard_normal((batch, T, H, P), dtype=np.float32)
    z = rng.standard_normal((batch, T, H), dtype=np.float32) - np.float32(2.0)
    dt = np.logaddexp(np.float32(0.0), z).astype(np.float32)          # softplus
    A = -np.exp(rng.uniform(np.log(1.0), np.log(16.0), size=H)).astype(np.float32)
    sd = np.float32(1.0 / np.sqrt(N))
    B = rng.standard_normal((batch, T, G, N), dtype=np.float32) * sd
    C = rng.standard_normal((batch, T, G, N), dtype=np.float32) * sd
    D = rng.standard_normal(H, dtype=np.float32)
    cu = None
    if w.varlen_total:
        lens = segment_lengths(rng, T, w.seg_min, w.seg_max)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    nseq = (len(cu) - 1) if cu is not None else batch
    init = None
    if w.init_state:
        init = (rng.standard_normal((nseq, H, P, N), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    if w.dtype == "bf16":
        x, B, C = bf16_round(x), bf16_round(B), bf16_round(C)
    if init is not None and w.state_dtype == "bf16":
        init = bf16_round(init)
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D, initial_state=init, cu_seqlens=cu)


def make_norm_inputs(w: Workload, rows: Optional[int] = None) -> dict:
    """Draw a gate and normalization workload's inputs: y, z (batch, T, H, P) fp32 holding bf16 values and
    weight (H*P,) fp32. With `rows`: a draw of that many tokens (batch 1), the CPU side's sample."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    b, T = (w.batch, w.seqlen) if rows is None else (1, rows)
    shp = (b, T, w.nheads, w.headdim)
    y = bf16_round(rng.standard_normal(shp, dtype=np.float32))
    z = bf16_round(rng.standard_normal(shp, dtype=np.float32))
    weight = rng.uniform(0.5, 1.5, w.nheads * w.headdim).astype(np.float32)
    return dict(y=y, z=z, weight=weight)


def small_variant(w: Workload, seqlen: int, nheads: int, batch: Optional[int] = None, **kw) -> Workload:
    """A cut-down copy of a workload (same distributions and head shape) that the oracle runs in seconds."""
    d = dict(seqlen=seqlen, nheads=nheads, name=w.name + f"_T{seqlen}_H{nheads}")
    if batch is not None:
        d["batch"] = batch
    if w.varlen_total:
        d["varlen_total"] = seqlen
    d.update(kw)
    return w.with_(**d)
