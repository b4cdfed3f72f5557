"""Pins of the gate-and-normalization oracle (oracle.gated_norm), against identities that do not restate
its code: the logistic function's symmetry, the defining property of an RMS normalization, scale and
permutation invariance, and a hand-worked token."""
import numpy as np

import oracle


def test_silu_symmetry_and_special_values():
    # logistic(z) + logistic(-z) = 1, so silu(z) - silu(-z) = z for every z
    z = np.concatenate([np.linspace(-30, 30, 601), [-700.0, 700.0, 1e-300, -1e-300]])
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=1e-15, atol=1e-15)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # far on either side: the identity, or zero
    assert np.isclose(oracle.silu(np.array([50.0]))[0], 50.0, rtol=1e-15)
    assert abs(oracle.silu(np.array([-50.0]))[0]) < 1e-19
    # silu(ln 3) = ln 3 * 3 / 4 (logistic(ln 3) = 3/4)
    assert np.isclose(oracle.silu(np.array([np.log(3.0)]))[0], 0.75 * np.log(3.0), rtol=1e-15)


def test_each_group_has_unit_rms_without_weight():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((3, 5, 4, 8))
    z = rng.standard_normal((3, 5, 4, 8))
    for groups in (1, 2, 4, 32):
        out = oracle.gated_rmsnorm(y, z, eps=0.0, groups=groups).reshape(15, groups, -1)
        assert np.allclose(np.sqrt(np.mean(out ** 2, axis=-1)), 1.0, rtol=1e-13)


def test_scale_invariance_sign_and_weight():
    rng = np.random.default_rng(2)
    y = rng.standard_normal((2, 7, 3, 16))
    z = rng.standard_normal((2, 7, 3, 16))
    w = rng.standard_normal(48)
    base = oracle.gated_rmsnorm(y, z, w, eps=0.0, groups=3)
    assert np.allclose(oracle.gated_rmsnorm(5.5 * y, z, w, eps=0.0, groups=3), base, rtol=1e-13)
    assert np.allclose(oracle.gated_rmsnorm(-y, z, w, eps=0.0, groups=3), -base, rtol=1e-13)
    # the weight scales channels after the normalization
    ones = oracle.gated_rmsnorm(y, z, None, eps=0.0, groups=3)
    assert np.allclose(base, ones * w.reshape(3, 16), rtol=1e-13)


def test_gate_is_elementwise_and_zero_gate_gives_zero():
    rng = np.random.default_rng(3)
    y = rng.standard_normal((4, 2, 8))
    out = oracle.gated_rmsnorm(y, np.zeros_like(y), eps=1e-5)
    assert np.all(out == 0.0)
    # a gate of silu(z) = 3/4 everywhere (z = ln 3) normalizes to the same as no gate (eps = 0)
    z = np.full_like(y, np.log(3.0))
    assert np.allclose(oracle.gated_rmsnorm(y, z, eps=0.0), oracle.gated_rmsnorm(y, None, eps=0.0), rtol=1e-13)


def test_groups_are_independent_and_ordered():
    # permuting whole groups of channels permutes the output the same way
    rng = np.random.default_rng(4)
    y = rng.standard_normal((3, 4, 6))
    z = rng.standard_normal((3, 4, 6))
    out = oracle.gated_rmsnorm(y, z, eps=1e-6, groups=4).reshape(3, 4, 6)
    perm = [2, 0, 3, 1]
    out_p = oracle.gated_rmsnorm(y[:, perm], z[:, perm], eps=1e-6, groups=4).reshape(3, 4, 6)
    assert np.allclose(out_p, out[:, perm], rtol=1e-14)


def test_hand_worked_token():
    # one token, H = 1, P = 4, no gate, one group: v = (1, 2, 2, 4), mean(v^2) = 25/4, rms = 5/2
    y = np.array([[[1.0, 2.0, 2.0, 4.0]]])
    out = oracle.gated_rmsnorm(y, None, eps=0.0)
    assert np.array_equal(out, np.array([[[0.4, 0.8, 0.8, 1.6]]]))


def test_eps_is_inside_the_root():
    # v = 0.1 on every channel: mean(v^2) = 0.01; with eps = 0.03 the root is sqrt(0.04) = 0.2
    y = np.full((1, 1, 4), 0.1)
    out = oracle.gated_rmsnorm(y, None, eps=0.03)
    assert np.allclose(out, 0.5, rtol=1e-14)
