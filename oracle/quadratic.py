"""Dual (quadratic, attention-like) form of the SSD layer, materialised (test infrastructure only).

For one sequence and head, the map x -> y is y = M x + D x with the T x T matrix

    M_ij = C_i . B_j * L_ij   for i >= j,   0 above the diagonal,
    L_ij = a_i * a_{i-1} * ... * a_{j+1}   (L_ii = 1),   a_t = exp(dt_t * A_h),

i.e. M = L o (C B^T) with L the 1-semiseparable mask. An initial state h0 adds
C_i . (a_i ... a_0) h0 to row i, the same product extended down to token 0.

Sources: "Transformers是SSMs：通过结构化状态空间对偶性的广义模型和高效算法(一)",
§3.1 (M_ji = C_j^T A_j ... A_{i+1} B_i, lower triangular) and §3.2.2 (the
1-SS matrix); "LLM(十一)——Mamba", §3.1.3 (quadratic mode, M = L o C B^T);
"Mamba-2 状态空间对偶性理论", §1.3 and §3.1 (matrix expansion, 1-SS mask).

The mask is built from running products of a_t in fp64, an independent route
from the recurrence in ``ssd_oracle.c``. Cost is O(T^2) per head: tiny T only.
"""
from __future__ import annotations

import numpy as np


def one_ss_mask(a: np.ndarray) -> np.ndarray:
    """L with L_ij = prod_{k=j+1..i} a_k for i >= j, else 0 (a: (T,))."""
    T = a.shape[0]
    L = np.zeros((T, T), dtype=np.float64)
    for j in range(T):
        prod = 1.0
        L[j, j] = 1.0
        for i in range(j + 1, T):
            prod *= a[i]
            L[i, j] = prod
    return L


def ssd_quadratic(x, dt, A, B, C, D=None, initial_state=None):
    """Dense batch only. Shapes as in ``oracle.ssd_recurrence``.

    Returns (y, final_state); the final state is h_T = sum_j (a_T..a_{j+1}) x_j B_j^T
    plus (a_T..a_0) h0, read off the same mask.
    """
    x, dt, A, B, C = (np.asarray(v, dtype=np.float64) for v in (x, dt, A, B, C))
    batch, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    y = np.zeros_like(x)
    final = np.zeros((batch, H, P, N), dtype=np.float64)
    for b in range(batch):
        for h in range(H):
            g = h // hpg
            a = np.exp(dt[b, :, h] * A[h])
            L = one_ss_mask(a)
            CB = C[b, :, g, :] @ B[b, :, g, :].T
            M = L * CB
            y[b, :, h, :] = M @ x[b, :, h, :]
            if D is not None:
                y[b, :, h, :] += float(D[h]) * x[b, :, h, :]
            # weights of each input in the final state: a_{T-1} ... a_{j+1}
            w_last = L[T - 1, :]
            final[b, h] = (x[b, :, h, :] * w_last[:, None]).T @ B[b, :, g, :]
            if initial_state is not None:
                h0 = np.asarray(initial_state[b, h], dtype=np.float64)
                decay0 = np.cumprod(a)          # a_0 ... a_i
                y[b, :, h, :] += decay0[:, None] * (C[b, :, g, :] @ h0.T)
                final[b, h] += decay0[-1] * h0
    return y, final
