"""Pins of the AdamW oracle against properties the algorithm fixes (no GPU)."""
import numpy as np

from oracle.adamw_ref import adamw_step_ref


def _rng(seed):
    return np.random.default_rng(seed)


def test_first_step_from_zero_state_is_normalised_sign():
    # m_1 = (1-b1) g, v_1 = (1-b2) g^2 and the bias corrections undo the
    # factors exactly: the step is lr * g / (|g| + eps)
    r = _rng(1)
    p, g = r.normal(size=1000), r.normal(size=1000) * 10.0 ** r.uniform(-4, 2, 1000)
    z = np.zeros(1000)
    lr, wd, eps = 3e-3, 0.1, 1e-8
    p1, m1, v1 = adamw_step_ref(p, g, z, z, 1, lr=lr, beta1=0.9, beta2=0.95, eps=eps, wd=wd)
    np.testing.assert_allclose(p1, p * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-14)
    np.testing.assert_allclose(v1, 0.05 * g * g, rtol=1e-12)


def test_constant_gradient_moves_lr_per_step():
    # with a constant gradient the corrected averages equal g and g^2 at
    # every step, so (no decay) each step moves p by lr * g / (|g| + eps)
    r = _rng(2)
    p0, g = r.normal(size=64), r.normal(size=64)
    p, m, v = p0.copy(), np.zeros(64), np.zeros(64)
    lr, eps = 1e-2, 1e-8
    for t in range(1, 8):
        p, m, v = adamw_step_ref(p, g, m, v, t, lr=lr, beta1=0.8, beta2=0.99, eps=eps, wd=0.0)
    np.testing.assert_allclose(p, p0 - 7 * lr * g / (np.abs(g) + eps), rtol=1e-10, atol=1e-12)


def test_zero_gradient_is_pure_decay():
    p0 = _rng(3).normal(size=32)
    p, m, v = p0.copy(), np.zeros(32), np.zeros(32)
    for t in range(1, 6):
        p, m, v = adamw_step_ref(p, np.zeros(32), m, v, t, lr=0.05, wd=0.2)
    np.testing.assert_allclose(p, p0 * (1 - 0.05 * 0.2) ** 5, rtol=1e-13)
    assert not m.any() and not v.any()


def test_memoryless_betas():
    # beta1 = beta2 = 0: every step sees only its own gradient
    r = _rng(4)
    p, m, v = r.normal(size=16), r.normal(size=16), np.abs(r.normal(size=16))
    g = r.normal(size=16)
    p1, m1, v1 = adamw_step_ref(p, g, m, v, 9, lr=0.1, beta1=0.0, beta2=0.0, eps=1e-6, wd=0.0)
    np.testing.assert_allclose(p1, p - 0.1 * g / (np.abs(g) + 1e-6), rtol=1e-13)
    np.testing.assert_allclose(m1, g, rtol=0)
    np.testing.assert_allclose(v1, g * g, rtol=0)


def test_moving_averages_are_weighted_sums():
    # m_t = (1-b1) sum_i b1^(t-i) g_i and v_t likewise for g_i^2, from zero
    r = _rng(5)
    gs = r.normal(size=(6, 10))
    b1, b2 = 0.7, 0.9
    p, m, v = np.zeros(10), np.zeros(10), np.zeros(10)
    for t in range(1, 7):
        p, m, v = adamw_step_ref(p, gs[t - 1], m, v, t, beta1=b1, beta2=b2)
    w1 = np.array([(1 - b1) * b1 ** (6 - i) for i in range(1, 7)])
    w2 = np.array([(1 - b2) * b2 ** (6 - i) for i in range(1, 7)])
    np.testing.assert_allclose(m, w1 @ gs, rtol=1e-12)
    np.testing.assert_allclose(v, w2 @ (gs * gs), rtol=1e-12)


def test_rejects_step_zero():
    import pytest
    with pytest.raises(ValueError):
        adamw_step_ref(np.zeros(2), np.zeros(2), np.zeros(2), np.zeros(2), 0)
