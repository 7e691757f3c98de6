"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics,
never by re-running the oracle's own formulas: hand-worked examples, closed
forms through an independent SVD, invariants, special cases and brute force.
Each test names the slip it would catch."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _frac_matrix(rows):
    return np.array([[float(Fraction(v)) for v in row] for row in rows])


# ---------------------------------------------------------------- RowNorm step
def test_worked_rownorm_step_3x4():
    """Hand-worked 3x4 RowNorm step (golden file). Catches: wrong axis, a zero
    row mapped to 1/eps, weight decay scaled by gamma, gamma missing."""
    gd = _load("rownorm_worked_3x4.json")
    inp, exp = gd["inputs"], gd["expected"]
    G = np.array(inp["G"], float)
    W_new, M_new, D, rho = O.prmuon_step(
        np.array(inp["W"], float), np.array(inp["M_prev"], float), G, inp["t"], inp["K"],
        inp["gamma"], inp["lr"], inp["wd"], inp["beta"], inp["eps"])
    assert rho == exp["branch"]
    np.testing.assert_allclose(M_new, G, rtol=0, atol=0)
    np.testing.assert_allclose(D, _frac_matrix(exp["D"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(W_new, _frac_matrix(exp["W_new"]), rtol=0, atol=1e-15)
    assert abs(np.linalg.norm(D) - math.sqrt(2)) < 1e-15


def test_worked_rownorm_step_transposed_4x3():
    """Same example stored tall (4x3): columns are normalised and the shape
    scale is sqrt(4/3). Catches: rows normalised on tall matrices, a shape
    scale taken from the wrong orientation."""
    gd = _load("rownorm_worked_3x4.json")
    inp = gd["inputs"]
    G = np.array(inp["G"], float).T
    W_new, _, D, rho = O.prmuon_step(np.ones((4, 3)), np.zeros((4, 3)), G, 1, 3,
                                     inp["gamma"], inp["lr"], inp["wd"], inp["beta"], inp["eps"])
    np.testing.assert_allclose(D, _frac_matrix(gd["expected"]["D"]).T, atol=1e-15)
    assert O.lr_shape_scale(4, 3) == pytest.approx(math.sqrt(4 / 3), abs=1e-15)
    assert W_new[0, 0] == pytest.approx(0.99 - 0.015 * math.sqrt(4 / 3) * 0.6, abs=1e-15)


@pytest.mark.parametrize("shape", [(5, 9), (9, 5), (7, 7), (1, 6), (6, 1)])
def test_rownorm_unit_short_side_vectors(shape):
    """Every short-side vector has norm 1, so ||R(M)||_F = sqrt(r) (the
    walkthrough's remark that both maps have Frobenius norm sqrt(r))."""
    rng = np.random.default_rng(1)
    M = rng.standard_normal(shape)
    D = O.row_normalize(M, 1e-8)
    m, n = shape
    axis = 1 if m <= n else 0
    np.testing.assert_allclose(np.linalg.norm(D, axis=axis), 1.0, atol=1e-14)
    assert np.linalg.norm(D) == pytest.approx(math.sqrt(min(m, n)), rel=1e-14)


def test_rownorm_below_eps_and_zero_vectors():
    """max(norm, eps): a vector shorter than eps is divided by eps, not
    normalised; a zero vector stays zero."""
    eps = 1e-3
    M = np.array([[3e-4, 4e-4, 0.0], [0.0, 0.0, 0.0], [2.0, 0.0, 0.0]])
    D = O.row_normalize(M, eps)
    np.testing.assert_allclose(D[0], [0.3, 0.4, 0.0], atol=1e-15)
    np.testing.assert_array_equal(D[1], 0.0)
    np.testing.assert_allclose(D[2], [1.0, 0.0, 0.0], atol=0)
    # the same vectors as the columns of a tall matrix
    Dt = O.row_normalize(np.vstack([M.T, np.zeros((1, 3))]), eps)
    np.testing.assert_allclose(Dt[:3].T, D, atol=1e-15)
    np.testing.assert_array_equal(Dt[3], 0.0)


def test_rownorm_scale_invariance_picks_the_right_axis():
    """Scaling a short-side vector leaves R unchanged, scaling along the long
    side does not. Catches a transposed axis on either orientation."""
    rng = np.random.default_rng(2)
    for shape in [(4, 11), (11, 4)]:
        M = rng.standard_normal(shape)
        m, n = shape
        if m <= n:
            short_scaled = M * rng.uniform(0.1, 10, (m, 1))
            long_scaled = M * rng.uniform(0.1, 10, (1, n))
        else:
            short_scaled = M * rng.uniform(0.1, 10, (1, n))
            long_scaled = M * rng.uniform(0.1, 10, (m, 1))
        D = O.row_normalize(M, 1e-12)
        np.testing.assert_allclose(O.row_normalize(short_scaled, 1e-12), D, atol=1e-14)
        assert np.abs(O.row_normalize(long_scaled, 1e-12) - D).max() > 1e-3


# ---------------------------------------------------------------- NS5
def _ns_scalar(s, coeffs, steps):
    a, b, c = coeffs
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def test_ns5_diagonal_worked_example():
    """Hand-worked NS5 on diag(3, 4) padded to 2x4 (golden file)."""
    gd = _load("ns5_diagonal_2x4.json")
    X = np.array(gd["X"], float)
    D = O.newton_schulz(X, gd["coeffs"], eps_ns=0.0)
    np.testing.assert_allclose(D, np.array(gd["expected_D"]), rtol=0, atol=gd["tolerance_abs"])
    for s0, key in ((0.6, "iterates_of_0.6"), (0.8, "iterates_of_0.8")):
        for k, v in enumerate(gd[key], start=1):
            assert _ns_scalar(s0, gd["coeffs"], k) == pytest.approx(v, abs=1e-11)
    # with the default eps the result moves by far less than the bf16 budget
    np.testing.assert_allclose(O.newton_schulz(X, gd["coeffs"]), np.array(gd["expected_D"]), atol=1e-6)


@pytest.mark.parametrize("coeffs", [None, (1.5, -0.5, 0.0), (1.875, -0.6, -0.275)])
@pytest.mark.parametrize("shape", [(3, 8), (8, 3), (6, 6), (1, 5), (5, 1), (12, 40)])
def test_ns5_matches_svd_closed_form(shape, coeffs):
    """NS commutes with the SVD: NS5(X) = U diag(p^5(sigma / ||X||_F)) V^T with
    p(s) = a s + b s^3 + c s^5 (numpy's LAPACK SVD, not the oracle's matmuls),
    for the default quintic and for triples with c = 0 and c < 0. Catches a
    dropped or sign-flipped polynomial term, X^T X in place of X X^T, and a
    missing transpose for tall inputs."""
    rng = np.random.default_rng(3)
    X = rng.standard_normal(shape)
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    sig = S / (np.linalg.norm(X) + O.NS_EPS)
    cf = O.DEFAULT_NS_COEFFS if coeffs is None else coeffs
    expected = U @ np.diag([_ns_scalar(s, cf, 5) for s in sig]) @ Vt
    got = O.newton_schulz(X) if coeffs is None else O.newton_schulz(X, coeffs)
    np.testing.assert_allclose(got, expected, rtol=0, atol=1e-12)


def test_cubic_newton_schulz_reaches_polar_factor():
    """With the cubic coefficients (1.5, -0.5, 0) Newton-Schulz converges to the
    polar factor U V^T (the method approximates the polar decomposition)."""
    rng = np.random.default_rng(4)
    X = rng.standard_normal((4, 6))
    U, _, Vt = np.linalg.svd(X, full_matrices=False)
    P = O.newton_schulz(X, (1.5, -0.5, 0.0), steps=60)
    np.testing.assert_allclose(P, U @ Vt, atol=1e-12)


def test_ns5_singular_values_in_narrow_band():
    """After NS5 with the default quintic the singular values of a random
    matrix sit in a narrow band around 1 (computed independently: every
    normalised singular value in [1.5e-3, 1] maps into [0.68, 1.21])."""
    rng = np.random.default_rng(5)
    grid = np.linspace(1.5e-3, 1.0, 20001)
    mapped = _ns_scalar(grid, O.DEFAULT_NS_COEFFS, 5)
    assert mapped.min() > 0.67 and mapped.max() < 1.21
    for shape in [(16, 48), (48, 16), (32, 32)]:
        X = rng.standard_normal(shape)
        S = np.linalg.svd(X, compute_uv=False)
        if (S / np.linalg.norm(X)).min() < 1.5e-3:
            continue
        Sd = np.linalg.svd(O.newton_schulz(X), compute_uv=False)
        assert Sd.min() > 0.67 and Sd.max() < 1.21


def test_ns5_zero_matrix_gives_zero():
    np.testing.assert_array_equal(O.newton_schulz(np.zeros((3, 5))), 0.0)


# ---------------------------------------------------------------- schedule
def test_refresh_schedule_table():
    """rho_t = [t mod K == 0]: the update rule's refresh indicator."""
    table = {1: "111111111111", 2: "101010101010", 3: "100100100100", 4: "100010001000"}
    for K, row in table.items():
        assert "".join(str(O.refresh_indicator(t, K)) for t in range(12)) == row
    with pytest.raises(ValueError):
        O.refresh_indicator(0, 0)


def test_tiny_run_refreshes_twice_in_six_steps():
    rng = np.random.default_rng(6)
    shapes = [(4, 6), (6, 4)]
    Gs = {(t, i): rng.standard_normal(s) for t in range(6) for i, s in enumerate(shapes)}
    _, _, br = O.run_steps([np.zeros(s) for s in shapes], [np.zeros(s) for s in shapes],
                           lambda t, i: Gs[(t, i)], 0, 6, 3, 0.15, 0.02, 0.01, 0.95, 1e-8)
    assert br == [1, 0, 0, 1, 0, 0]


# ---------------------------------------------------------------- momentum / update
def test_momentum_closed_form():
    """M_t = sum_k beta^(t-k) G_k over a run (no Nesterov term, no damping)."""
    rng = np.random.default_rng(7)
    beta = 0.9
    Gs = [rng.standard_normal((3, 5)) for _ in range(5)]
    M = np.zeros((3, 5))
    for G in Gs:
        M = O.momentum_update(M, G, beta)
    closed = sum(beta ** (4 - k) * Gs[k] for k in range(5))
    np.testing.assert_allclose(M, closed, atol=1e-14)


def test_decoupled_weight_decay_closed_form():
    """G = 0, M = 0: both branches give D = 0, so W_t = W_0 (1 - lr wd)^t."""
    rng = np.random.default_rng(8)
    W0 = rng.standard_normal((5, 7))
    Ws, _, _ = O.run_steps([W0], [np.zeros((5, 7))], lambda t, i: np.zeros((5, 7)), 0, 7,
                           3, 0.15, 0.05, 0.2, 0.95, 1e-8)
    np.testing.assert_allclose(Ws[0], W0 * (1 - 0.05 * 0.2) ** 7, rtol=1e-14)


def test_step_size_by_branch():
    """lr on refresh steps, lr * gamma on RowNorm steps (gamma calibrates the
    RowNorm branch), shape scale applied on both."""
    rng = np.random.default_rng(9)
    W, G = rng.standard_normal((6, 3)), rng.standard_normal((6, 3))
    s = O.lr_shape_scale(6, 3)
    for t, eta in ((3, 0.1), (4, 0.1 * 0.3)):
        W1, M1, D, rho = O.prmuon_step(W, np.zeros((6, 3)), G, t, 3, 0.3, 0.1, 0.0, 0.9, 1e-8)
        np.testing.assert_allclose(W - W1, eta * s * D, atol=1e-14)
    assert s == pytest.approx(math.sqrt(2.0))
    assert O.lr_shape_scale(3, 6) == 1.0


# ---------------------------------------------------------------- MuonBP
def test_block_slices_partition_long_side():
    for (m, n, P) in [(4, 20, 8), (20, 4, 8), (8, 8, 8), (3, 17, 4)]:
        covered = np.zeros((m, n), int)
        sl = O.block_slices(m, n, P)
        assert len(sl) == P
        for rs, cs in sl:
            covered[rs, cs] += 1
            if m <= n:
                assert (rs.start, rs.stop) == (0, m)
            else:
                assert (cs.start, cs.stop) == (0, n)
        np.testing.assert_array_equal(covered, 1)
    assert O.block_slices(3, 17, 4)[-1][1] == slice(12, 17)


def test_muonbp_single_block_equals_full_step():
    rng = np.random.default_rng(10)
    W, M, G = (rng.standard_normal((5, 9)) for _ in range(3))
    a = O.muonbp_step(W, M, G, 1, 3, 0.15, 0.02, 0.01, 0.95, 1e-8, P=1)
    b = O.muonbp_step(W, M, G, 0, 3, 0.15, 0.02, 0.01, 0.95, 1e-8, P=1)
    np.testing.assert_allclose(a[2], b[2], atol=1e-14)


def test_muonbp_block_step_is_per_block_svd_closed_form():
    """Block steps orthogonalise each block on its own: per-block SVD closed
    form (each block normalised by its own Frobenius norm)."""
    rng = np.random.default_rng(11)
    for shape in [(6, 24), (24, 6)]:
        M = rng.standard_normal(shape)
        _, _, D, full = O.muonbp_step(np.zeros(shape), np.zeros(shape), M, 2, 3, 0.15,
                                      0.02, 0.0, 0.9, 1e-8, P=4)
        assert full == 0
        for rs, cs in O.block_slices(*shape, 4):
            Bk = M[rs, cs]
            U, S, Vt = np.linalg.svd(Bk, full_matrices=False)
            sig = S / (np.linalg.norm(Bk) + O.NS_EPS)
            exp = U @ np.diag([_ns_scalar(s, O.DEFAULT_NS_COEFFS, 5) for s in sig]) @ Vt
            np.testing.assert_allclose(D[rs, cs], exp, atol=1e-12)


def test_muonbp_full_step_is_whole_matrix_ns5():
    rng = np.random.default_rng(12)
    M = rng.standard_normal((8, 16))
    W1, _, D, full = O.muonbp_step(np.zeros((8, 16)), np.zeros((8, 16)), M, 3, 3, 1.25,
                                   0.016, 0.0, 0.9, 1e-8, P=8)
    assert full == 1
    U, S, Vt = np.linalg.svd(M, full_matrices=False)
    sig = S / (np.linalg.norm(M) + O.NS_EPS)
    exp = U @ np.diag([_ns_scalar(s, O.DEFAULT_NS_COEFFS, 5) for s in sig]) @ Vt
    np.testing.assert_allclose(D, exp, atol=1e-12)
    np.testing.assert_allclose(W1, -0.016 * D, atol=1e-15)
