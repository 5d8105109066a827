"""Pins of the CPU float64 oracle to things other than itself.

Each oracle function is checked against at least one of: the SVD closed form
of the iteration, exact decimal constants of the scalar quintic map
(tests/golden/poly_constants.txt), values the pages print
(tests/golden/ns5_coefficients.txt, muon_hyperparams.txt), invariants, and
brute force on tiny inputs.  ``test_planted_mistakes_are_caught`` plants the
plausible mistakes in copies of the oracle and checks a pin rejects each.
"""

import numpy as np
import pytest

import oracle
from oracle import muon_oracle as om


def _rng(seed):
    return np.random.default_rng(seed)


def svd_closed_form(G, steps, coeffs, eps):
    """Exact result of the NS iteration, built from numpy's SVD.

    If X = U diag(s) V^T then X X^T = U diag(s^2) U^T, so one round maps
    s -> a s + b s^3 + c s^5 and keeps U, V.  The singular values are mapped
    through that scalar polynomial `steps` times.
    """
    G = np.asarray(G, dtype=np.float64)
    a, b, c = coeffs
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    s = S / (np.linalg.norm(G, "fro") + eps)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return (U * s) @ Vt


def rel_fro(x, ref):
    return np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300)


SHAPES = [(1, 12), (12, 1), (3, 5), (5, 3), (8, 8), (12, 40), (40, 12), (33, 65), (64, 64), (65, 33)]


# ---------------------------------------------------------------- page values
def test_coefficients_match_pages(golden):
    g = golden("ns5_coefficients.txt")
    assert oracle.NS5_COEFFS == (g["a"], g["b"], g["c"])
    assert oracle.NS5_STEPS == int(g["steps"])


def test_hyperparams_fixture_is_consistent(golden):
    h = golden("muon_hyperparams.txt")
    assert (h["default_lr"], h["default_weight_decay"], h["default_momentum"]) == (0.02, 0.01, 0.95)
    assert h["warmup_momentum_start"] < h["warmup_momentum_end"] == h["train_momentum"]


# ---------------------------------------------------------- closed-form pins
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_ns_matches_svd_closed_form(shape, steps):
    G = _rng(hash(shape) % 1000 + steps).standard_normal(shape)
    O = oracle.newton_schulz5(G, steps)
    ref = svd_closed_form(G, steps, oracle.NS5_COEFFS, oracle.NS5_EPS)
    assert O.shape == G.shape
    assert rel_fro(O, ref) < 1e-11


@pytest.mark.parametrize("shape", [(128, 256), (256, 128), (96, 300)])
def test_ns_closed_form_heavy_tailed_rows(shape):
    # rows scaled x100 give a spread of singular values, like the d=2048 workload
    G = _rng(7).standard_normal(shape)
    G[: max(1, shape[0] // 100)] *= 100.0
    ref = svd_closed_form(G, 5, oracle.NS5_COEFFS, oracle.NS5_EPS)
    assert rel_fro(oracle.newton_schulz5(G), ref) < 1e-10


def test_poly_constants_fixture_matches_recomputation(golden):
    # the stored decimals agree with a float64 scalar evaluation
    g = golden("poly_constants.txt")
    a, b, c = oracle.NS5_COEFFS

    def p5(s):
        for _ in range(5):
            s = a * s + b * s ** 3 + c * s ** 5
        return s
    assert abs(p5(1.0) - g["p5_at_1"]) < 1e-13
    for m in (4, 128, 512, 768, 4096):
        assert abs(p5(1 / np.sqrt(m)) - g[f"p5_at_inv_sqrt_{m}"]) < 1e-13


# ----------------------------------------------------------- special cases
@pytest.mark.parametrize("shape", [(1, 12), (1, 768), (12, 1), (7, 9)])
def test_rank_one_gives_p5_of_one(shape, golden):
    r = _rng(3)
    x = r.standard_normal((shape[0], 1))
    y = r.standard_normal((1, shape[1]))
    G = 3.0 * (x @ y)
    O = oracle.newton_schulz5(G)
    k = golden("poly_constants.txt")["p5_at_1"]
    # eps shifts the single singular value by eps/||G|| ~ 1e-8
    np.testing.assert_allclose(O, k * G / np.linalg.norm(G), rtol=0, atol=1e-7)


@pytest.mark.parametrize("m,n", [(4, 9), (128, 256), (512, 640), (768, 768)])
def test_orthonormal_rows(m, n, golden):
    Q, _ = np.linalg.qr(_rng(m).standard_normal((n, m)))
    Q = Q.T  # m x n, orthonormal rows
    O = oracle.newton_schulz5(2.5 * Q)
    k = golden("poly_constants.txt")[f"p5_at_inv_sqrt_{m}"]
    # eps moves s = 1/sqrt(m) by a relative 1e-7/||G||_F; the map amplifies that a little
    np.testing.assert_allclose(O, k * Q, rtol=0, atol=1e-6 / np.sqrt(n))
    # the transposed input takes the tall branch and gives the transposed answer
    np.testing.assert_allclose(oracle.newton_schulz5(2.5 * Q.T), k * Q.T, rtol=0, atol=1e-6 / np.sqrt(n))


def test_zero_matrix_stays_zero():
    O = oracle.newton_schulz5(np.zeros((5, 7)))
    assert np.all(O == 0.0) and np.all(np.isfinite(O))


def test_one_by_one_brute_force(golden):
    k = golden("poly_constants.txt")["p5_at_1"]
    for x in (-3.0, 0.5, 1e3):
        s = abs(x) / (abs(x) + oracle.NS5_EPS)
        a, b, c = oracle.NS5_COEFFS
        for _ in range(5):
            s = a * s + b * s ** 3 + c * s ** 5
        assert abs(oracle.newton_schulz5(np.array([[x]]))[0, 0] - np.sign(x) * s) < 1e-14
        assert abs(abs(oracle.newton_schulz5(np.array([[x]]))[0, 0]) - k) < 1e-6


def test_two_by_two_diagonal_brute_force():
    # diag(3, 4): ||G||_F = 5, singular vectors are the axes
    G = np.diag([3.0, -4.0])
    a, b, c = oracle.NS5_COEFFS
    out = []
    for d in (3.0, 4.0):
        s = d / (5.0 + oracle.NS5_EPS)
        for _ in range(5):
            s = a * s + b * s ** 3 + c * s ** 5
        out.append(s)
    np.testing.assert_allclose(oracle.newton_schulz5(G), np.diag([out[0], -out[1]]), atol=1e-14)


# -------------------------------------------------------------- invariants
@pytest.mark.parametrize("shape", [(48, 96), (96, 48), (64, 64)])
def test_singular_vectors_preserved_and_band(shape, golden):
    G = _rng(11).standard_normal(shape)
    O = oracle.newton_schulz5(G)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    D = U.T @ O @ Vt.T
    off = D - np.diag(np.diag(D))
    assert np.abs(off).max() < 1e-10
    g = golden("poly_constants.txt")
    s_in = S / np.linalg.norm(G)
    s_out = np.diag(D)
    sel = s_in >= 2e-3
    assert np.all(s_out[sel] >= g["band_min_from_0.002"] - 1e-6)
    assert np.all(s_out[sel] <= g["band_max_from_0.002"] + 1e-6)


def test_small_singular_values_stay_small():
    # a direction with s < 1e-3 is amplified by about a^5 ~ 487 and stays < 0.5
    U, _ = np.linalg.qr(_rng(5).standard_normal((6, 6)))
    V, _ = np.linalg.qr(_rng(6).standard_normal((6, 6)))
    S = np.array([1.0, 1.0, 1.0, 1.0, 1.0, 2e-3])
    G = (U * S) @ V.T
    D = U.T @ oracle.newton_schulz5(G) @ V
    assert D[5, 5] < 0.5 and D[0, 0] > 0.68


def test_scale_invariance_and_transpose_equivariance():
    G = _rng(9).standard_normal((20, 50))
    O = oracle.newton_schulz5(G)
    # equal up to the eps term: relative eps/||G||_F ~ 3e-9 here
    assert rel_fro(oracle.newton_schulz5(1e3 * G), O) < 1e-7
    assert rel_fro(oracle.newton_schulz5(G.T), O.T) < 1e-12


# --------------------------------------------------------- momentum / apply
def test_momentum_closed_forms():
    g = _rng(1).standard_normal((4, 6))
    buf = oracle.momentum_buffer_update(np.zeros_like(g), g, 0.95)
    np.testing.assert_allclose(buf, 0.05 * g, rtol=1e-15)
    u = oracle.nesterov_blend(g, buf, 0.95)
    # (1 - beta) g + beta (1 - beta) g = 0.0975 g
    np.testing.assert_allclose(u, 0.0975 * g, rtol=1e-14)


def test_momentum_two_steps_brute_force():
    beta = 0.85
    g1, g2, b0 = 0.3, -1.7, 0.25
    b1 = beta * b0 + (1 - beta) * g1
    b2 = beta * b1 + (1 - beta) * g2
    u2 = (1 - beta) * g2 + beta * b2
    buf = oracle.momentum_buffer_update(np.array([[b0]]), np.array([[g1]]), beta)
    buf = oracle.momentum_buffer_update(buf, np.array([[g2]]), beta)
    assert abs(buf[0, 0] - b2) < 1e-15
    assert abs(oracle.nesterov_blend(np.array([[g2]]), buf, beta)[0, 0] - u2) < 1e-15


def test_rescale_factor_values():
    assert oracle.rescale_factor(3072, 768) == 2.0
    assert oracle.rescale_factor(768, 3072) == 1.0
    assert oracle.rescale_factor(512, 1024) == 1.0   # the page's 512x1024 example
    assert abs(oracle.rescale_factor(1024, 512) - 2 ** 0.5) < 1e-15


def test_step_zero_grad_is_pure_decay():
    p = _rng(2).standard_normal((6, 10)) * 0.02
    newp, newbuf, O = oracle.muon_step(p, np.zeros_like(p), np.zeros_like(p), momentum=0.95,
                                       lr=0.02, weight_decay=0.01)
    assert np.all(O == 0) and np.all(newbuf == 0)
    np.testing.assert_allclose(newp, 0.9998 * p, rtol=1e-15)


def test_step_config1_identity():
    # zero buffer: u = 0.0975 g and NS is scale invariant, so O = NS(g)
    r = _rng(0)
    g = r.standard_normal((16, 32))
    p = 0.02 * r.standard_normal((16, 32))
    newp, _, O = oracle.muon_step(p, g, np.zeros_like(g), momentum=0.95, lr=0.02, weight_decay=0.01)
    assert rel_fro(O, svd_closed_form(g, 5, oracle.NS5_COEFFS, 0.0)) < 1e-7
    np.testing.assert_allclose(newp, 0.9998 * p - 0.02 * O, rtol=1e-14, atol=1e-17)


def test_tall_step_uses_rows_over_cols_rescale():
    r = _rng(4)
    g = r.standard_normal((40, 10))
    p = r.standard_normal((40, 10))
    newp, _, O = oracle.muon_step(p, g, np.zeros_like(g), momentum=0.9, lr=0.1, weight_decay=0.0)
    np.testing.assert_allclose(newp, p - 0.1 * 2.0 * O, rtol=1e-14)
    newp2, _, _ = oracle.muon_step(p, g, np.zeros_like(g), momentum=0.9, lr=0.1, weight_decay=0.0,
                                   lr_scale=1.0)
    np.testing.assert_allclose(newp2, p - 0.1 * O, rtol=1e-14)


def test_nesterov_off_uses_buffer():
    r = _rng(8)
    g = r.standard_normal((5, 9))
    b = r.standard_normal((5, 9))
    _, newbuf, O = oracle.muon_step(np.zeros_like(g), g, b, momentum=0.9, nesterov=False,
                                    lr=0.1, weight_decay=0.0)
    assert rel_fro(O, svd_closed_form(0.9 * b + 0.1 * g, 5, oracle.NS5_COEFFS, oracle.NS5_EPS)) < 1e-11


def test_batched_equals_per_matrix():
    r = _rng(12)
    G = r.standard_normal((3, 7, 11))
    P = r.standard_normal((3, 7, 11))
    B = r.standard_normal((3, 7, 11))
    bp, bb, bo = oracle.muon_step_batched(P, G, B, momentum=0.9, lr=0.1, weight_decay=0.1)
    for i in range(3):
        p, b, o = oracle.muon_step(P[i], G[i], B[i], momentum=0.9, lr=0.1, weight_decay=0.1)
        assert np.array_equal(bp[i], p) and np.array_equal(bb[i], b) and np.array_equal(bo[i], o)
    assert oracle.newton_schulz5_batched(np.zeros((0, 4, 5))).shape == (0, 4, 5)


# ------------------------------------------------------------ planted mistakes
def _mutant(kind):
    a0, b0, c0 = oracle.NS5_COEFFS

    def ns(G, steps=5, coeffs=oracle.NS5_COEFFS, eps=oracle.NS5_EPS):
        a, b, c = coeffs
        if kind == "wrong_sign_b":
            b = -b
        X = np.array(G, dtype=np.float64)
        tr = X.shape[0] > X.shape[1]
        if tr:
            X = X.T
        if kind == "spectral_norm":
            X = X / (np.linalg.norm(X, 2) + eps)
        else:
            X = X / (np.linalg.norm(X) + eps)
        for _ in range(steps):
            A = X @ X.T
            if kind == "dropped_c_term":
                B = b * A
            elif kind == "swapped_a_b":
                B = a * A + c * (A @ A)
            else:
                B = b * A + c * (A @ A)
            if kind == "right_multiply":
                X = a * X + X @ B  # shape error unless square; wrong unless commuting
            else:
                X = a * X + B @ X
        if tr and kind != "no_transpose_back":
            X = X.T
        return X
    return ns


@pytest.mark.parametrize("kind", ["wrong_sign_b", "dropped_c_term", "swapped_a_b", "spectral_norm",
                                  "right_multiply", "no_transpose_back"])
def test_planted_mistakes_are_caught(kind):
    ns = _mutant(kind)
    caught = False
    for shape in [(12, 40), (40, 12), (16, 16)]:
        G = _rng(21).standard_normal(shape)
        ref = svd_closed_form(G, 5, oracle.NS5_COEFFS, oracle.NS5_EPS)
        try:
            with np.errstate(all="ignore"):
                out = ns(G)
            with np.errstate(all="ignore"):
                caught |= out.shape != ref.shape or not rel_fro(out, ref) <= 1e-6
        except ValueError:
            caught = True
    assert caught, kind


def _momentum_mutant(kind):
    def step(g, buf, beta):
        if kind == "swapped_lerp_weight":
            nb = buf + beta * (g - buf)
        else:
            nb = buf + (1 - beta) * (g - buf)
        if kind == "blend_with_old_buffer":
            u = g + beta * (buf - g)
        elif kind == "blend_reversed":
            u = nb + beta * (g - nb)
        else:
            u = g + beta * (nb - g)
        return nb, u
    return step


@pytest.mark.parametrize("kind", ["swapped_lerp_weight", "blend_with_old_buffer", "blend_reversed"])
def test_planted_momentum_mistakes_are_caught(kind):
    # brute-force scalar recurrence of test_momentum_two_steps_brute_force
    beta, g1, g2, b0 = 0.85, 0.3, -1.7, 0.25
    b1 = beta * b0 + (1 - beta) * g1
    b2 = beta * b1 + (1 - beta) * g2
    u2 = (1 - beta) * g2 + beta * b2
    step = _momentum_mutant(kind)
    nb, _ = step(g1, b0, beta)
    nb, u = step(g2, nb, beta)
    assert abs(nb - b2) > 1e-6 or abs(u - u2) > 1e-6
