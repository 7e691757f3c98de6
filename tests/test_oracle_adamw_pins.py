"""Pins for the fp64 AdamW oracle (non-matrix parameters), against closed
forms that a slip in it would break: bias correction, decoupled weight decay,
eps outside the square root."""
import numpy as np
import pytest

import oracle as O

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1)


def test_first_step_from_zero_state_is_sign_like():
    """From m = v = 0 the bias-corrected moments are g and g^2, so the step is
    lr * g / (|g| + eps). Catches a missing bias correction (the step would be
    lr * 0.1 g / (sqrt(0.001) |g| + eps))."""
    rng = np.random.default_rng(0)
    p0, g = rng.standard_normal(64), rng.standard_normal(64) * 1e-3
    p1, m1, v1 = O.adamw_step(p0, np.zeros(64), np.zeros(64), g, 1, **HP)
    expect = p0 * (1 - HP["lr"] * HP["wd"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    np.testing.assert_allclose(p1, expect, rtol=0, atol=1e-15)
    np.testing.assert_allclose(m1, 0.1 * g, atol=1e-18)
    np.testing.assert_allclose(v1, 0.001 * g * g, atol=1e-24)


def test_constant_gradient_closed_form():
    """A constant gradient keeps m_hat = g and v_hat = g^2 at every t, so
    p_T = p_0 d^T - lr g/(|g|+eps) sum_{k<T} d^k with d = 1 - lr wd."""
    rng = np.random.default_rng(1)
    p, g = rng.standard_normal(32), rng.standard_normal(32)
    m, v = np.zeros(32), np.zeros(32)
    p0 = p.copy()
    T = 7
    for t in range(1, T + 1):
        p, m, v = O.adamw_step(p, m, v, g, t, **HP)
    d = 1 - HP["lr"] * HP["wd"]
    expect = p0 * d ** T - HP["lr"] * g / (np.abs(g) + HP["eps"]) * sum(d ** k for k in range(T))
    np.testing.assert_allclose(p, expect, rtol=1e-12, atol=1e-15)


def test_zero_gradient_is_pure_decoupled_decay():
    """g = 0: the moments stay zero and the parameter only decays (a coupled
    L2 term folded into g would leave p unchanged here)."""
    p0 = np.linspace(-1, 1, 11)
    p, m, v = p0.copy(), np.zeros(11), np.zeros(11)
    for t in range(1, 6):
        p, m, v = O.adamw_step(p, m, v, np.zeros(11), t, **HP)
    np.testing.assert_allclose(p, p0 * (1 - HP["lr"] * HP["wd"]) ** 5, rtol=1e-14)
    assert not m.any() and not v.any()


def test_eps_sits_outside_the_square_root():
    """A gradient far below eps: the step is lr g / eps (not lr g / sqrt(eps))."""
    g = np.full(3, 1e-12)
    p1, _, _ = O.adamw_step(np.zeros(3), np.zeros(3), np.zeros(3), g, 1, lr=1.0, beta1=0.9, beta2=0.999,
                            eps=1e-8, wd=0.0)
    np.testing.assert_allclose(p1, -g / (1e-12 + 1e-8), rtol=1e-12)


def test_step_count_starts_at_one():
    with pytest.raises(ValueError):
        O.adamw_step(np.zeros(1), np.zeros(1), np.zeros(1), np.zeros(1), 0, **HP)
