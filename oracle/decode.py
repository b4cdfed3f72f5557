"""Oracle for the one-token recurrent step of the SSD layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it.

The step is the recurrent (autoregressive inference) mode of the selective SSM with a
scalar-times-identity A: "Transformers是SSMs：通过结构化状态空间对偶性的广义模型和高效算法(一)"
§2.1 (the recurrent mode used for inference, one input step at a time), the recurrence of
"LLM(十一)——Mamba" §3.1.1-3.1.2 and "Mamba-2 状态空间对偶性理论" §1.2, whose per-token cost
("Inference FLOPs", N^2 for a state of N x P with P = N) is tabulated in "LLM(十一)——Mamba" §3.5.3.

For every batch row b and head h (group g = h // (H/G)):

    a            = exp(dt[b, h] * A[h])
    S[b, h]      = a * S[b, h] + outer(x[b, h, :], B[b, g, :])      (P x N)
    y[b, h, :]   = S[b, h] @ C[b, g, :] + D[h] * x[b, h, :]

Written directly from that definition in fp64 numpy, one (batch, head) at a time.
"""
from __future__ import annotations

import numpy as np


def ssd_decode_step(state, x, dt, A, B, C, D=None, scale_x_by_dt=False):
    """One recurrent step.

    state (batch, H, P, N); x (batch, H, P); dt (batch, H); A (H,); B, C (batch, G, N);
    D (H,) or None. Returns ``(y, new_state)`` as float64 arrays of shapes (batch, H, P)
    and (batch, H, P, N); the inputs are not modified. With ``scale_x_by_dt`` the input term
    is ``dt x (outer) B`` and the skip term keeps ``D x``.
    """
    S = np.array(state, dtype=np.float64, copy=True)
    x = np.asarray(x, dtype=np.float64)
    dt = np.asarray(dt, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    batch, H, P, N = S.shape
    G = B.shape[1]
    assert x.shape == (batch, H, P) and dt.shape == (batch, H) and A.shape == (H,)
    assert B.shape == (batch, G, N) and C.shape == B.shape and H % G == 0
    y = np.empty((batch, H, P), dtype=np.float64)
    for b in range(batch):
        for h in range(H):
            g = h // (H // G)
            a = np.exp(dt[b, h] * A[h])
            xin = x[b, h] * dt[b, h] if scale_x_by_dt else x[b, h]
            S[b, h] = a * S[b, h] + np.outer(xin, B[b, g])
            y[b, h] = S[b, h] @ C[b, g]
            if D is not None:
                y[b, h] += float(D[h]) * x[b, h]
    return y, S
