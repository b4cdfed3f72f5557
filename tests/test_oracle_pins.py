"""Pins for the fp64 oracle: each test checks it against something other than itself.

- the dual quadratic form M = L o C B^T (independent numpy code, running products);
- closed forms: causal linear attention when every a_t = 1, the geometric series
  of a constant-decay scalar recurrence, a one-token hand expansion;
- the pages' 1-SS scalar example (tests/golden/one_ss_scalar.json);
- structural identities: sequence split with state hand-off, variable-length
  packing equals independent runs, linearity, the D term, grouped heads.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle.quadratic import one_ss_mask, ssd_quadratic
from mamba_ssd_layer_gb300.inputs import WORKLOADS, make_inputs, small_variant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng(7)


def rand_problem(rng, batch=2, T=37, H=4, P=3, N=5, G=2, init=True, dt_scale=1.0):
    x = rng.standard_normal((batch, T, H, P))
    dt = np.logaddexp(0, rng.standard_normal((batch, T, H)) - 1.0) * dt_scale
    A = -np.exp(rng.uniform(0, np.log(16), H))
    B = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    C = rng.standard_normal((batch, T, G, N)) / np.sqrt(N)
    D = rng.standard_normal(H)
    h0 = 0.1 * rng.standard_normal((batch, H, P, N)) if init else None
    return x, dt, A, B, C, D, h0


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("T,G", [(1, 1), (17, 1), (64, 2), (40, 4)])
def test_recurrence_equals_quadratic_form(T, G):
    # "LLM(十一)——Mamba" §3.1.4: the linear (recurrent) and quadratic (masked attention) forms are the same map
    x, dt, A, B, C, D, h0 = rand_problem(np.random.default_rng(T * 10 + G), T=T, G=G, H=4)
    y_r, f_r = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    y_q, f_q = ssd_quadratic(x, dt, A, B, C, D, h0)
    assert rel(y_r, y_q) < 1e-12
    assert rel(f_r, f_q) < 1e-12


def test_one_ss_mask_matches_page_example():
    # "Mamba-2 状态空间对偶性理论" §3.1: rows 1, a1, a2 a1 / a2 ... of the 1-SS matrix
    a = np.array([9.0, 2.0, 3.0, 5.0])
    L = one_ss_mask(a)
    expect = np.array([[1, 0, 0, 0], [2, 1, 0, 0], [6, 3, 1, 0], [30, 15, 5, 1]], dtype=float)
    assert np.array_equal(L, expect)


def test_golden_scalar_one_ss():
    g = json.load(open(os.path.join(GOLDEN, "one_ss_scalar.json")))
    a = np.array(g["a"])
    T = len(a)
    x = np.array(g["x"]).reshape(1, T, 1, 1)
    dt = np.log(1.0 / a).reshape(1, T, 1)
    A = np.array([-1.0])
    ones = np.ones((1, T, 1, 1))
    y, f = oracle.ssd_recurrence(x, dt, A, ones, ones, None, None)
    assert np.allclose(y.ravel(), g["y_expected"], rtol=0, atol=1e-14)
    assert abs(f.ravel()[0] - g["final_state_expected"]) < 1e-14


def test_linear_attention_special_case():
    # a_t = 1 (A = 0): Y = C . cumsum_s(x_s B_s^T), causal linear attention
    # ("LLM(十一)——Mamba" §3.1.3; "Transformers是SSMs…(一)" eq. (14))
    rng = np.random.default_rng(3)
    x, dt, A, B, C, D, _ = rand_problem(rng, batch=1, T=50, H=3, P=4, N=6, G=1, init=False)
    A = np.zeros_like(A)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, None, None)
    for h in range(3):
        KV = np.cumsum(x[0, :, h, :, None] * B[0, :, 0, None, :], axis=0)  # (T, P, N)
        ref = np.einsum("tpn,tn->tp", KV, C[0, :, 0, :])
        assert rel(y[0, :, h, :], ref) < 1e-12
        assert rel(f[0, h], KV[-1]) < 1e-12


def test_constant_decay_geometric_closed_form():
    # scalar SSM with constant a: y_t = sum_{s<=t} a^{t-s} x_s; with x = 1, y_t = (1 - a^{t+1}) / (1 - a)
    # ("Transformers是SSMs…(一)" §3.2.2 scalar recurrence; constant a is the RetNet decay mask)
    T = 200
    a = 0.97
    x = np.ones((1, T, 1, 1))
    dt = np.full((1, T, 1), -np.log(a) / 2.0)
    A = np.array([-2.0])
    ones = np.ones((1, T, 1, 1))
    y, f = oracle.ssd_recurrence(x, dt, A, ones, ones, None, None)
    t = np.arange(T)
    assert rel(y.ravel(), (1 - a ** (t + 1)) / (1 - a)) < 1e-13
    # impulse response: x = delta at s0 gives y_t = a^{t-s0} for t >= s0, 0 before
    s0 = 31
    x = np.zeros((1, T, 1, 1)); x[0, s0] = 1.0
    y, _ = oracle.ssd_recurrence(x, dt, A, ones, ones, None, None)
    expect = np.where(t >= s0, a ** np.clip(t - s0, 0, None), 0.0)
    assert rel(y.ravel(), expect) < 1e-13


def test_one_token_hand_expansion():
    # T = 1: h_0 = a_0 h_init + x_0 B_0^T, y_0 = h_0 C_0 + D x_0
    rng = np.random.default_rng(11)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=1, T=1, H=2, P=3, N=4, G=1)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    for h in range(2):
        a = np.exp(dt[0, 0, h] * A[h])
        S = a * h0[0, h] + np.outer(x[0, 0, h], B[0, 0, 0])
        assert rel(f[0, h], S) < 1e-15
        assert rel(y[0, 0, h], S @ C[0, 0, 0] + D[h] * x[0, 0, h]) < 1e-14


def test_sequence_split_state_handoff():
    # context-parallel identity ("LLM(十一)——Mamba" §3.7.2): run(x[:T1], h0) -> h1; run(x[T1:], h1) == run(x, h0)
    rng = np.random.default_rng(5)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=2, T=90, H=3, P=4, N=6, G=1)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    for T1 in (1, 33, 89):
        y1, h1 = oracle.ssd_recurrence(x[:, :T1], dt[:, :T1], A, B[:, :T1], C[:, :T1], D, h0)
        y2, h2 = oracle.ssd_recurrence(x[:, T1:], dt[:, T1:], A, B[:, T1:], C[:, T1:], D, h1)
        assert rel(np.concatenate([y1, y2], axis=1), y) < 1e-13
        assert rel(h2, f) < 1e-13


def test_varlen_equals_independent_runs():
    # variable length by state reset ("LLM(十一)——Mamba" §3.7.3): packed run == separate runs per segment
    rng = np.random.default_rng(9)
    lens = [5, 1, 40, 17, 3]
    T = sum(lens)
    x, dt, A, B, C, D, _ = rand_problem(rng, batch=1, T=T, H=3, P=2, N=4, G=1, init=False)
    h0 = 0.1 * rng.standard_normal((len(lens), 3, 2, 4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0, cu_seqlens=cu)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        ys, fs = ssd_quadratic(x[:, sl], dt[:, sl], A, B[:, sl], C[:, sl], D, h0[s:s + 1])
        assert rel(y[:, sl], ys) < 1e-12
        assert rel(f[s], fs[0]) < 1e-12


def test_linearity_and_skip_term():
    rng = np.random.default_rng(13)
    x1, dt, A, B, C, D, h1 = rand_problem(rng, batch=1, T=30, H=2, P=3, N=4, G=1)
    x2 = rng.standard_normal(x1.shape)
    h2 = rng.standard_normal(h1.shape)
    al, be = 0.7, -1.3
    ya, fa = oracle.ssd_recurrence(x1, dt, A, B, C, D, h1)
    yb, fb = oracle.ssd_recurrence(x2, dt, A, B, C, D, h2)
    yc, fc = oracle.ssd_recurrence(al * x1 + be * x2, dt, A, B, C, D, al * h1 + be * h2)
    assert rel(yc, al * ya + be * yb) < 1e-12
    assert rel(fc, al * fa + be * fb) < 1e-12
    # D term: y(D) - y(0) = D * x exactly up to rounding
    y0, _ = oracle.ssd_recurrence(x1, dt, A, B, C, None, h1)
    assert rel(ya - y0, D[None, None, :, None] * x1) < 1e-12


def test_grouped_heads_equal_expanded_heads():
    # grouped B, C: heads [g*H/G, (g+1)*H/G) share group g ("LLM(十一)——Mamba" §3.6 head patterns)
    rng = np.random.default_rng(17)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=1, T=25, H=6, P=2, N=3, G=3)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    Be = np.repeat(B, 2, axis=2)
    Ce = np.repeat(C, 2, axis=2)
    ye, fe = oracle.ssd_recurrence(x, dt, A, Be, Ce, D, h0)
    assert np.array_equal(y, ye) and np.array_equal(f, fe)


def test_empty_sequence_returns_initial_state():
    rng = np.random.default_rng(19)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=1, T=0, H=2, P=2, N=3, G=1)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0)
    assert y.shape == (1, 0, 2, 2)
    assert np.array_equal(f, h0)


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(23)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=2, T=70, H=5, P=4, N=8, G=1)
    y1, f1 = oracle.ssd_recurrence(x, dt, A, B, C, D, h0, nthreads=1)
    y8, f8 = oracle.ssd_recurrence(x, dt, A, B, C, D, h0, nthreads=8)
    assert np.array_equal(y1, y8) and np.array_equal(f1, f8)


def test_workload_inputs_follow_recipe():
    w = small_variant(WORKLOADS["m2_2p7b"], seqlen=128, nheads=4, batch=2)
    d = make_inputs(w)
    assert d["x"].shape == (2, 128, 4, 64) and d["B"].shape == (2, 128, 1, 128)
    assert (d["dt"] > 0).all() and (d["A"] <= -1.0 + 1e-6).all() and (d["A"] >= -16.0 - 1e-4).all()
    # bf16-representable: low 16 bits clear
    assert not (d["x"].view(np.uint32) & 0xFFFF).any()
    assert d["initial_state"].shape == (2, 4, 64, 128)
    v = make_inputs(small_variant(WORKLOADS["varlen"], seqlen=9000, nheads=2))
    cu = v["cu_seqlens"]
    assert cu[0] == 0 and cu[-1] == 9000 and (np.diff(cu) > 0).all()
    assert (np.diff(cu)[:-1] >= 64).all() and (np.diff(cu) <= 4096).all()


# ---------------------------------------------------------------- dt-scaled input term
@pytest.mark.parametrize("T,G", [(1, 1), (23, 1), (48, 2)])
def test_dt_scaled_input_against_quadratic_form(T, G):
    # dt x as the input term equals the dense quadratic form on dt o x, with the skip on the unscaled x
    x, dt, A, B, C, D, h0 = rand_problem(np.random.default_rng(70 + T + G), T=T, G=G, H=4)
    y_s, f_s = oracle.ssd_recurrence(x, dt, A, B, C, D, h0, scale_x_by_dt=True)
    xs = x * dt[..., None]
    y_q, f_q = ssd_quadratic(xs, dt, A, B, C, None, h0)
    assert rel(y_s, y_q + D[None, None, :, None] * x) < 1e-12
    assert rel(f_s, f_q) < 1e-12


def test_dt_scaled_input_one_token_closed_form():
    rng = np.random.default_rng(73)
    x, dt, A, B, C, D, h0 = rand_problem(rng, batch=1, T=1, H=2, P=3, N=4, G=1)
    y, f = oracle.ssd_recurrence(x, dt, A, B, C, D, h0, scale_x_by_dt=True)
    for h in range(2):
        a = np.exp(dt[0, 0, h] * A[h])
        S = a * h0[0, h] + dt[0, 0, h] * np.outer(x[0, 0, h], B[0, 0, 0])
        assert rel(f[0, h], S) < 1e-15
        assert rel(y[0, 0, h], S @ C[0, 0, 0] + D[h] * x[0, 0, h]) < 1e-14


def test_dt_scaled_input_packed_and_unit_dt():
    # with dt = 1 the option changes nothing; packed sequences still reset at every boundary
    rng = np.random.default_rng(74)
    x, dt, A, B, C, D, _ = rand_problem(rng, batch=1, T=60, H=2, G=1, init=False)
    one = np.ones_like(dt)
    y1, f1 = oracle.ssd_recurrence(x, one, A, B, C, D, None, scale_x_by_dt=True)
    y0, f0 = oracle.ssd_recurrence(x, one, A, B, C, D, None)
    assert np.array_equal(y1, y0) and np.array_equal(f1, f0)
    cu = np.array([0, 17, 17, 60], dtype=np.int32)
    yp, fp = oracle.ssd_recurrence(x, dt, A, B, C, D, None, cu_seqlens=cu, scale_x_by_dt=True)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        ys, fs = oracle.ssd_recurrence(x[:, a:b], dt[:, a:b], A, B[:, a:b], C[:, a:b], D, None,
                                       scale_x_by_dt=True)
        assert rel(yp[:, a:b], ys) < 1e-13 if b > a else True
        assert rel(fp[s], fs[0]) < 1e-13 if b > a else np.array_equal(fp[s], np.zeros_like(fp[s]))
