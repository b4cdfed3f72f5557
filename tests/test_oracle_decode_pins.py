"""Pins for the oracle's one-token recurrent step (oracle.ssd_decode_step), each against
something other than the function itself:

- closed forms: from a zero state the new state is the outer product x B^T and
  y = (B . C) x + D x; with x = 0 the state only decays, S' = a S and y = a S C;
- chaining T steps from an initial state equals the pinned token-by-token recurrence
  (oracle.ssd_recurrence) over those T tokens, outputs and final state;
- grouped heads: head h reads the B/C of group h // (H/G);
- the D term: y(D) - y(0) = D x; linearity of the step in (state, x).
"""
import numpy as np
import pytest

import oracle


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def rand_step(rng, batch=3, H=4, P=5, N=6, G=2):
    S = 0.1 * rng.standard_normal((batch, H, P, N))
    x = rng.standard_normal((batch, H, P))
    dt = np.logaddexp(0, rng.standard_normal((batch, H)) - 1.0)
    A = -np.exp(rng.uniform(0, np.log(16), H))
    B = rng.standard_normal((batch, G, N)) / np.sqrt(N)
    C = rng.standard_normal((batch, G, N)) / np.sqrt(N)
    D = rng.standard_normal(H)
    return S, x, dt, A, B, C, D


def test_zero_state_closed_form():
    rng = np.random.default_rng(21)
    S, x, dt, A, B, C, D = rand_step(rng, G=1)
    y, S1 = oracle.ssd_decode_step(np.zeros_like(S), x, dt, A, B, C, D)
    for b in range(S.shape[0]):
        bc = float(np.sum(B[b, 0] * C[b, 0]))
        for h in range(S.shape[1]):
            for p in range(S.shape[2]):
                for n in range(S.shape[3]):
                    assert S1[b, h, p, n] == x[b, h, p] * B[b, 0, n]
            assert rel(y[b, h], (bc + D[h]) * x[b, h]) < 1e-14


def test_zero_input_only_decays():
    rng = np.random.default_rng(22)
    S, x, dt, A, B, C, D = rand_step(rng)
    y, S1 = oracle.ssd_decode_step(S, np.zeros_like(x), dt, A, B, C, D)
    H = S.shape[1]
    G = B.shape[1]
    for b in range(S.shape[0]):
        for h in range(H):
            a = np.exp(dt[b, h] * A[h])
            g = h // (H // G)
            assert rel(S1[b, h], a * S[b, h]) < 1e-15
            assert rel(y[b, h], a * (S[b, h] @ C[b, g])) < 1e-14


@pytest.mark.parametrize("T,G", [(1, 1), (9, 1), (25, 2)])
def test_chained_steps_equal_recurrence(T, G):
    rng = np.random.default_rng(23 + T)
    batch, H, P, N = 2, 4, 3, 5
    x = rng.standard_normal((batch, T, H, P))
    dt = np.logaddexp(0, rng.standard_normal((batch, T, H)) - 1.0)
    A = -np.exp(rng.uniform(0, np.log(16), H))
    B = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    C = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    D = rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((batch, H, P, N))
    y_ref, f_ref = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    S = h0
    for t in range(T):
        y_t, S = oracle.ssd_decode_step(S, x[:, t], dt[:, t], A, B[:, t], C[:, t], D)
        assert rel(y_t, y_ref[:, t]) < 1e-12
    assert rel(S, f_ref) < 1e-12


def test_grouped_heads_use_their_group():
    rng = np.random.default_rng(24)
    S, x, dt, A, B, C, D = rand_step(rng, H=6, G=3)
    y, S1 = oracle.ssd_decode_step(S, x, dt, A, B, C, D)
    for g in range(3):
        hs = slice(2 * g, 2 * g + 2)
        y_g, S_g = oracle.ssd_decode_step(S[:, hs], x[:, hs], dt[:, hs], A[hs], B[:, g:g + 1], C[:, g:g + 1], D[hs])
        assert np.array_equal(y[:, hs], y_g) and np.array_equal(S1[:, hs], S_g)


def test_skip_term_and_linearity():
    rng = np.random.default_rng(25)
    S, x, dt, A, B, C, D = rand_step(rng)
    y1, S1 = oracle.ssd_decode_step(S, x, dt, A, B, C, D)
    y0, S0 = oracle.ssd_decode_step(S, x, dt, A, B, C, None)
    assert rel(y1 - y0, D[None, :, None] * x) < 1e-13
    assert np.array_equal(S1, S0)
    S2, x2 = 0.1 * rng.standard_normal(S.shape), rng.standard_normal(x.shape)
    ya, Sa = oracle.ssd_decode_step(S + 2.0 * S2, x + 2.0 * x2, dt, A, B, C, None)
    yb, Sb = oracle.ssd_decode_step(S2, x2, dt, A, B, C, None)
    assert rel(ya, y0 + 2.0 * yb) < 1e-13 and rel(Sa, S0 + 2.0 * Sb) < 1e-13


def test_inputs_are_not_modified():
    rng = np.random.default_rng(26)
    S, x, dt, A, B, C, D = rand_step(rng)
    keep = S.copy()
    oracle.ssd_decode_step(S, x, dt, A, B, C, D)
    assert np.array_equal(S, keep)


def test_dt_scaled_step_closed_form_and_chain():
    rng = np.random.default_rng(27)
    S, x, dt, A, B, C, D = rand_step(rng, G=1)
    y, S1 = oracle.ssd_decode_step(S, x, dt, A, B, C, D, scale_x_by_dt=True)
    for b in range(S.shape[0]):
        for h in range(S.shape[1]):
            a = np.exp(dt[b, h] * A[h])
            Sr = a * S[b, h] + dt[b, h] * np.outer(x[b, h], B[b, 0])
            assert rel(S1[b, h], Sr) < 1e-15
            assert rel(y[b, h], Sr @ C[b, 0] + D[h] * x[b, h]) < 1e-14
    # chained steps equal the pinned recurrence with the same option
    T, batch, H, P, N = 7, 2, 3, 4, 5
    xs = rng.standard_normal((batch, T, H, P))
    dts = np.logaddexp(0, rng.standard_normal((batch, T, H)) - 1.0)
    Bs = rng.standard_normal((batch, T, 1, N)) / np.sqrt(N)
    Cs = rng.standard_normal((batch, T, 1, N)) / np.sqrt(N)
    A3, D3 = -np.exp(rng.uniform(0, np.log(16), H)), rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((batch, H, P, N))
    yr, fr = oracle.ssd_recurrence(xs, dts, A3, Bs, Cs, D3, h0, scale_x_by_dt=True)
    St = h0
    for t in range(T):
        yt, St = oracle.ssd_decode_step(St, xs[:, t], dts[:, t], A3, Bs[:, t], Cs[:, t], D3, scale_x_by_dt=True)
        assert rel(yt, yr[:, t]) < 1e-12
    assert rel(St, fr) < 1e-12
