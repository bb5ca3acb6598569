"""The Gram-space formulation of Newton-Schulz that the grouped GEMM path
runs (DMuon-2 Appendix C.3, with the mid-way restart read as a restart every
P steps), written out in float64 with NumPy and checked against the float64
oracle's X-space iteration.  In exact arithmetic the two are the same map,
so any slip in the order of the products, the shift alpha, the restart or
the first-step normalisation shows up as a large difference.

Per phase of P steps (the first phase starts from X0 / (||X0|| + eps)):
  R = X X^T; for each step k of the phase, B'_k = b R + c R^2 + alpha I,
  Q = P_k = a I + b R + c R^2 at the phase's first step, else
  Q <- (a - alpha) Q + Q B'_k; unless it is the phase's last step,
  T = (a - alpha) R + R B'_k and R <- (a - alpha) T + T B'_k;
  at the phase's end X <- Q X.
"""
import numpy as np
import pytest

from oracle import muon_ref as R

ALPHA_FRAC = 0.58
EPS = 1e-7   # the first-step normalisation X0 / (||X0|| + eps), as in the oracle


def gram_space_ns(x, coeffs, period):
    m, n = x.shape
    tr = m > n
    X = (x.T if tr else x) / (np.linalg.norm(x) + EPS)
    steps = len(coeffs)
    period = period if period > 0 else steps
    I = np.eye(X.shape[0])
    k0 = 0
    while k0 < steps:
        k1 = min(steps, k0 + period)
        Rm = X @ X.T
        Q = None
        for it in range(k0, k1):
            a, b, c = coeffs[it]
            al = ALPHA_FRAC * a
            Bp = b * Rm + c * Rm @ Rm + al * I
            Q = (a - al) * I + Bp if Q is None else (a - al) * Q + Q @ Bp
            if it + 1 < k1:
                T = (a - al) * Rm + Rm @ Bp
                Rm = (a - al) * T + T @ Bp
        X = Q @ X
        k0 = k1
    return X.T if tr else X


@pytest.mark.parametrize("period", [0, 1, 2, 3, 5])
@pytest.mark.parametrize("shape", [(6, 20), (20, 6), (9, 9)])
def test_gram_space_equals_oracle(shape, period):
    rng = np.random.default_rng(sum(shape) + period)
    x = rng.standard_normal(shape)
    coeffs = [(3.4445, -4.7750, 2.0315)] * 5
    got = gram_space_ns(x, coeffs, period)
    ref = R.newton_schulz_ref(x, steps=5, coeffs=coeffs)
    assert np.linalg.norm(got - ref) <= 1e-10 * np.linalg.norm(ref)


def test_gram_space_coefficient_table():
    """Per-step coefficients: the shift follows each step's a."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((8, 30))
    table = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3), (1.5, -0.5, 0.0)]
    for period in (1, 2, 3, 0):
        got = gram_space_ns(x, table, period)
        ref = R.newton_schulz_ref(x, steps=4, coeffs=table)
        assert np.linalg.norm(got - ref) <= 1e-10 * np.linalg.norm(ref)


def test_transposed_products_would_differ_only_off_symmetry():
    """The products are symmetric in exact arithmetic (B'_k, T, R, Q are
    polynomials of one R), so A B^T = A B there; the GEMM path still forms
    A B because rounded matrices are not exactly symmetric."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 25)) / 5
    Rm = x @ x.T
    a, b, c = 3.4445, -4.7750, 2.0315
    Bp = b * Rm + c * Rm @ Rm + ALPHA_FRAC * a * np.eye(7)
    T = Rm @ Bp
    assert np.allclose(T, T.T, atol=1e-12) and np.allclose(Rm @ Bp, Rm @ Bp.T, atol=1e-12)
