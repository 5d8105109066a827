"""Pins of the Adam (DistAdam) oracle to things other than itself."""

import numpy as np
import pytest

import oracle


def test_settings_match_pages(golden):
    h = golden("muon_hyperparams.txt")
    assert oracle.ADAM_LR == h["adam_lr"]
    assert oracle.ADAM_BETAS == (h["adam_beta1"], h["adam_beta2"])
    assert oracle.ADAM_EPS == h["adam_eps"]


def test_first_step_closed_form():
    # zero state, t = 1: m = (1-b1) g, v = (1-b2) g^2, bias corrections cancel:
    # p1 = p0 - lr g / (|g| + eps / sqrt(1-b2))
    r = np.random.default_rng(0)
    g = r.standard_normal(100)
    p = r.standard_normal(100)
    z = np.zeros(100)
    p1, m1, v1 = oracle.adam_step(p, g, z, z, step=1, lr=0.01, betas=(0.9, 0.99), eps=1e-3)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v1, 0.01 * g * g, rtol=1e-14)
    np.testing.assert_allclose(p1, p - 0.01 * g / (np.abs(g) + 1e-3 / np.sqrt(0.01)), rtol=1e-13)


def test_scalar_recurrence_three_steps_brute_force():
    b1, b2, lr, eps, wd = 0.8, 0.95, 0.05, 1e-8, 0.1
    gs = [0.3, -1.2, 0.7]
    p, m, v = 1.5, 0.0, 0.0
    P, M, V = np.array([p]), np.zeros(1), np.zeros(1)
    for t, g in enumerate(gs, start=1):
        p *= 1 - lr * wd
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        step_size = lr * (1 - b2 ** t) ** 0.5 / (1 - b1 ** t)
        p -= step_size * m / (v ** 0.5 + eps)
        P, M, V = oracle.adam_step(P, np.array([g]), M, V, step=t, lr=lr, betas=(b1, b2), eps=eps,
                                   weight_decay=wd)
        assert abs(P[0] - p) < 1e-15 and abs(M[0] - m) < 1e-15 and abs(V[0] - v) < 1e-15


def test_zero_gradient_with_zero_state_is_pure_decay():
    p = np.linspace(-1, 1, 9)
    z = np.zeros(9)
    p1, m1, v1 = oracle.adam_step(p, z, z, z, step=4, lr=0.02, weight_decay=0.5, lr_scale=2.0,
                                  wd_scale=0.5)
    np.testing.assert_allclose(p1, p * (1 - 0.02 * 2.0 * 0.5 * 0.5), rtol=1e-15)
    assert np.all(m1 == 0) and np.all(v1 == 0)


def test_lr_scale_scales_the_step():
    r = np.random.default_rng(1)
    g, p, m, v = (r.standard_normal(20) for _ in range(4))
    v = np.abs(v)
    a, _, _ = oracle.adam_step(p, g, m, v, step=3, lr=0.01)
    b, _, _ = oracle.adam_step(p, g, m, v, step=3, lr=0.01, lr_scale=3.0)
    np.testing.assert_allclose(b - p, 3.0 * (a - p), rtol=1e-12, atol=1e-14)


def test_step_must_count_from_one():
    with pytest.raises(ValueError):
        oracle.adam_step(np.zeros(1), np.zeros(1), np.zeros(1), np.zeros(1), step=0)


def _mutant(kind):
    def step(p, g, m, v, t, lr=0.05, b1=0.8, b2=0.95, eps=1e-8):
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        bias1, bias2 = 1 - b1 ** t, 1 - b2 ** t
        if kind == "no_bias_correction":
            return p - lr * m / (np.sqrt(v) + eps)
        if kind == "bias2_not_rooted":
            return p - lr * bias2 / bias1 * m / (np.sqrt(v) + eps)
        if kind == "eps_inside_sqrt":
            return p - lr * np.sqrt(bias2) / bias1 * m / np.sqrt(v + eps)
        if kind == "betas_swapped":
            m2 = b2 * 0 + (1 - b2) * g
            return p - lr * np.sqrt(bias2) / bias1 * m2 / (np.sqrt(v) + eps)
        raise AssertionError(kind)
    return step


@pytest.mark.parametrize("kind", ["no_bias_correction", "bias2_not_rooted", "eps_inside_sqrt",
                                  "betas_swapped"])
def test_planted_mistakes_are_caught(kind):
    # the scalar brute force of test_scalar_recurrence_three_steps_brute_force, step 1-2,
    # with eps large enough to make its placement visible
    b1, b2, lr, eps = 0.8, 0.95, 0.05, 1e-2
    ref_p, mut_p = np.array([1.0]), np.array([1.0])
    m = v = np.zeros(1)
    mm = vv = np.zeros(1)
    diff = 0.0
    for t, g in enumerate([0.3, -1.2], start=1):
        ref_p, m, v = oracle.adam_step(ref_p, np.array([g]), m, v, step=t, lr=lr, betas=(b1, b2),
                                       eps=eps)
        mut = _mutant(kind)
        mut_p = mut(mut_p, np.array([g]), mm, vv, t, lr, b1, b2, eps)
        mm = b1 * mm + (1 - b1) * g
        vv = b2 * vv + (1 - b2) * g * g
        diff = max(diff, abs(float(mut_p[0] - ref_p[0])))
    assert diff > 1e-6, kind
