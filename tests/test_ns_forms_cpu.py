"""The library's two NS5 evaluation forms restated in fp64 numpy and checked
against the oracle's plain iteration ("Scaling Muon for Diffusion
Transformers", section "Periodic Row-wise Muon": X <- a X + (b A + c A A) X,
A = X X^T, five times). In exact arithmetic both forms are the iteration
itself; in fp64 they must agree with the oracle to rounding (~1e-13), so a
wrong recurrence, a lost scale, a leg boundary in the wrong place or a
transposed product fails here, on the CPU, before any kernel runs.

Direct form, as the kernels evaluate it: C = sqrt|c| A + sgn(c) b/(2 sqrt|c|) I,
P = sgn(c) C C + (a - b^2/(4c)) I, X <- P X (c = 0: P = b A + a I).

Gram route, as the kernels evaluate it: rounds in legs of at most three; per
leg, from X_s with A_0 = X_s X_s^T and a power-of-two S near r:
  round 1: C_1 from S A_0 (GRAM's second output), P_1 = Q_1, T_1 = P_1 S A_0
  round j: C_j = sqrt|c| T_{j-1} Q_{j-1}^T / S + sgn(c) b/(2 sqrt|c|) I,
           P_j as above, Q_j = P_j Q_{j-1}, T_j = P_j T_{j-1}
  end:     X_e = Q_L X_s
with the symmetric products formed on their upper 256 x 256 blocks and
mirrored, as the symmetric-output kernel does."""
import numpy as np
import pytest

import oracle as O

BLOCK = 256


def _sym_product(A, B):
    """A B^T from its upper block triangle, the lower blocks mirrored (the
    symmetric-output kernel's scheme; exact when A B^T is symmetric)."""
    n = A.shape[0]
    out = np.empty((n, B.shape[0]))
    for i0 in range(0, n, BLOCK):
        for j0 in range(i0, n, BLOCK):
            blk = A[i0:i0 + BLOCK] @ B[j0:j0 + BLOCK].T
            out[i0:i0 + BLOCK, j0:j0 + BLOCK] = blk
            if j0 > i0:
                out[j0:j0 + BLOCK, i0:i0 + BLOCK] = blk.T
    return out


def _coeff_forms(coeffs):
    a, b, c = coeffs
    if c == 0:
        return None
    root, sg = np.sqrt(abs(c)), np.sign(c)
    return root, sg * b / (2 * root), sg, a - b * b / (4 * c)


def _wide(M):
    X = np.asarray(M, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    return (X.T if tall else X), tall


def direct_form(M, coeffs=O.DEFAULT_NS_COEFFS, steps=5):
    a, b, c = coeffs
    X, tall = _wide(M)
    X = X / (np.linalg.norm(X) + O.NS_EPS)
    I = np.eye(X.shape[0])
    cf = _coeff_forms(coeffs)
    for _ in range(steps):
        A = _sym_product(X, X)
        if cf is None:
            P = b * A + a * I
        else:
            g, k0, sg, d0 = cf
            C = g * A + k0 * I
            P = sg * _sym_product(C, C) + d0 * I
        X = P @ X
    return X.T if tall else X


def gram_route(M, coeffs=O.DEFAULT_NS_COEFFS, steps=5, leg=3):
    g, k0, sg, d0 = _coeff_forms(coeffs)
    X, tall = _wide(M)
    r = X.shape[0]
    S = 1.0
    while S * 2 <= r and S < 8192:
        S *= 2
    I = np.eye(r)
    s = 1.0 / (np.linalg.norm(X) + O.NS_EPS)
    Xs, scale = X, s  # the first leg starts from the unnormalised X and its scale
    done = 0
    while done < steps:
        L = min(leg, steps - done)
        acc = _sym_product(Xs, Xs) * scale * scale
        A0s = S * acc                     # GRAM's second output
        C = g * acc + k0 * I              # GRAM's first output
        P = sg * _sym_product(C, C) + d0 * I
        if L == 1:
            Xs, scale = (P @ Xs) * scale, 1.0
            done += 1
            continue
        Q, T = P, _sym_product(P, A0s)    # P_1 written as Q_1; T_1 = P_1 S A_0 (A_0 symmetric)
        for j in range(2, L + 1):
            C = (g / S) * _sym_product(T, Q) + k0 * I
            P = sg * _sym_product(C, C) + d0 * I
            Qn = _sym_product(P, Q)       # P Q = P Q^T: both polynomials in A_0
            if j < L:
                T = _sym_product(P, T)
            Q = Qn
        Xs, scale = (Q @ Xs) * scale, 1.0
        done += L
    return Xs.T if tall else Xs


SHAPES = [(40, 1000), (300, 520), (520, 300), (96, 640), (600, 256), (384, 384), (2, 3), (1, 50)]


@pytest.mark.parametrize("shape", SHAPES)
def test_direct_form_is_the_iteration(shape):
    """Catches: a wrong completed square (sign, shift or gain), the s^2 scale
    on the wrong round, a transposed product."""
    M = np.random.default_rng(sum(shape)).standard_normal(shape)
    ref = O.newton_schulz(M)
    assert np.linalg.norm(direct_form(M) - ref) <= 1e-12 * max(1.0, np.linalg.norm(ref))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [1, 2, 3, 4, 5, 7])
def test_gram_route_is_the_iteration(shape, steps):
    """Any number of rounds, legs of three and a shorter last one. Catches: Q
    and T updated with the wrong P, T started from A_0 instead of P_1 A_0, the
    1/S of C dropped, the leg's end applied to the wrong X, the scale s used
    after the first leg."""
    M = np.random.default_rng(7 * sum(shape) + steps).standard_normal(shape)
    ref = O.newton_schulz(M, steps=steps)
    err = np.linalg.norm(gram_route(M, steps=steps) - ref) / max(1e-300, np.linalg.norm(ref))
    assert err <= 1e-11, (shape, steps, err)


@pytest.mark.parametrize("coeffs", [(3.4445, -4.7750, 2.0315), (1.875, -0.6, -0.275), (2.0, -1.5, 0.5)])
def test_gram_route_other_coefficients(coeffs):
    """c > 0 and c < 0: the completed square's sign enters C and P alike."""
    M = np.random.default_rng(3).standard_normal((200, 700))
    ref = O.newton_schulz(M, coeffs=coeffs)
    err = np.linalg.norm(gram_route(M, coeffs=coeffs) - ref) / np.linalg.norm(ref)
    assert err <= 1e-11


def test_gram_route_legs_matter_only_in_rounding():
    """One five-round leg, legs of three and two, and the direct form are the
    same function in exact arithmetic."""
    M = np.random.default_rng(11).standard_normal((300, 1100))
    a = gram_route(M, leg=5)
    b = gram_route(M, leg=3)
    c = direct_form(M)
    assert np.linalg.norm(a - b) <= 1e-11 * np.linalg.norm(b)
    assert np.linalg.norm(b - c) <= 1e-11 * np.linalg.norm(c)


def test_gram_route_zero_matrix():
    """NS5 of 0 is 0: every Q is a multiple of I, every T zero."""
    assert np.count_nonzero(gram_route(np.zeros((64, 256)))) == 0
