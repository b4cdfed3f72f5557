"""Oracle for the layer's output gate and extra normalization (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it.

"LLM(十一)——Mamba" §3.6.1 (Block Design, Extra Normalization): the Mamba-2 block multiplies the SSD
layer's output by a gate branch and then adds a normalization layer (LayerNorm, GroupNorm or RMSNorm)
before the output projection; the normalization comes after the multiplicative gate. Read here as
(the pages print neither formula): the gate is SiLU of a second input z of y's shape, the default
nonlinearity of "LLM(十一)——Mamba" §3.6.2, and the normalization is RMSNorm over each group of
``H*P / groups`` consecutive channels of a token (one group: the whole token), with a learned scale:

    v       = y * silu(z),                 silu(z) = z / (1 + exp(-z))
    out     = v / sqrt(mean(v**2 over the group) + eps) * weight

Written from that definition in fp64 numpy, one token row at a time.
"""
from __future__ import annotations

import numpy as np


def silu(z):
    """z * logistic(z), fp64, computed without overflow for either sign."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def gated_rmsnorm(y, z=None, weight=None, eps=1e-5, groups=1):
    """y, z: (..., H, P); weight: (H*P,) or None (ones). z None: no gate. Returns float64 of y's shape."""
    y = np.asarray(y, dtype=np.float64)
    lead, (H, P) = y.shape[:-2], y.shape[-2:]
    C = H * P
    assert C % groups == 0, "groups must divide H*P"
    v = y if z is None else y * silu(z)
    rows = v.reshape(-1, groups, C // groups)
    out = np.empty_like(rows)
    for r in range(rows.shape[0]):
        for g in range(groups):
            seg = rows[r, g]
            out[r, g] = seg / np.sqrt(np.mean(seg * seg) + eps)
    out = out.reshape(lead + (C,))
    if weight is not None:
        out = out * np.asarray(weight, dtype=np.float64)
    return out.reshape(y.shape)
