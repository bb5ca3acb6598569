"""Pins of the float64 oracle against what the mathematics fixes.

None of these tests re-types the oracle's own iteration: each expected value
comes from an independent route (a closed form on SVD-built inputs, exact
rational arithmetic, the other association of the polynomial, a library polar
factor, a geometric series), chosen so that a dropped term, a wrong sign, a
transposed operand or a wrong normalisation fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import muon_ref as R

QUINTIC = R.DEFAULT_COEFFS
CUBIC = (1.5, -0.5, 0.0)   # classical Newton-Schulz polar iteration


def _orth(rng, n, k):
    q, _ = np.linalg.qr(rng.standard_normal((n, k)))
    return q[:, :k]


def _relerr(x, y):
    den = max(np.linalg.norm(y), 1e-300)
    return np.linalg.norm(np.asarray(x) - np.asarray(y)) / den


# --------------------------------------------------------------------------
# Closed form: for G = U diag(s) V^T, NS(G) = U diag(f^K(s / (||s|| + eps))) V^T
# (HyperParallel-FSDP section 2.3: the iteration acts on singular values).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(6, 9), (9, 6), (7, 7), (1, 5), (5, 1), (24, 80)])
@pytest.mark.parametrize("spectrum", ["spread", "repeated", "rank_deficient", "tiny_top"])
def test_closed_form_svd(shape, spectrum):
    rng = np.random.default_rng(hash((shape, spectrum)) % 2**32)
    m, n = shape
    k = min(m, n)
    if spectrum == "spread":
        s = np.logspace(-6, 0, k)
    elif spectrum == "repeated":
        s = np.array([0.7] * (k // 2) + [0.2] * (k - k // 2))
    elif spectrum == "rank_deficient":
        s = np.linspace(1.0, 0.1, k)
        s[k // 2:] = 0.0
        if k == 1:
            s[:] = 1.0
    else:
        s = np.linspace(1e-3, 1e-5, k)
    U = _orth(rng, m, k)
    V = _orth(rng, n, k)
    G = (U * s) @ V.T
    eps = R.DEFAULT_EPS
    fs = R.scalar_polynomial_ref(s / (np.linalg.norm(s) + eps), 5, abc=QUINTIC)
    want = (U * fs) @ V.T
    got = R.newton_schulz_ref(G, 5, abc=QUINTIC, eps=eps)
    assert got.shape == G.shape
    assert _relerr(got, want) <= 1e-12


def test_closed_form_per_step_table():
    """A per-step coefficient table applies step k's triple at step k."""
    rng = np.random.default_rng(5)
    U, V = _orth(rng, 5, 5), _orth(rng, 8, 5)
    s = np.array([1.0, 0.5, 0.25, 0.1, 0.01])
    G = (U * s) @ V.T
    table = [(3.0, -3.2, 1.2), (2.5, -2.0, 0.6), (1.9, -1.2, 0.3)]
    x = s / (np.linalg.norm(s) + 1e-7)
    for a, b, c in table:
        x = a * x + b * x ** 3 + c * x ** 5
    want = (U * x) @ V.T
    got = R.newton_schulz_ref(G, 3, coeffs=table)
    assert _relerr(got, want) <= 1e-12
    # order matters: reversing the table changes the answer
    rev = R.newton_schulz_ref(G, 3, coeffs=table[::-1])
    assert _relerr(rev, want) > 1e-3


# --------------------------------------------------------------------------
# Exact rational arithmetic on a tiny case (eps = 0 and ||G||_F = 7 rational),
# using the OTHER association of the polynomial from the DMuon architecture
# page: X' = a X + b X (X^T X) + c X (X^T X)^2, right multiplication by the
# n x n Gram, without transposing first.
# --------------------------------------------------------------------------
def _frac_matmul(P, Q):
    return [[sum(P[i][k] * Q[k][j] for k in range(len(Q))) for j in range(len(Q[0]))]
            for i in range(len(P))]


def _frac_T(P):
    return [list(r) for r in zip(*P)]


def _exact_ns(G, norm, steps, abc):
    a, b, c = (Fraction(str(v)) for v in abc)
    X = [[Fraction(v) / norm for v in row] for row in G]
    for _ in range(steps):
        S = _frac_matmul(_frac_T(X), X)              # X^T X (n x n)
        S2 = _frac_matmul(S, S)
        XS = _frac_matmul(X, S)
        XS2 = _frac_matmul(X, S2)
        X = [[a * X[i][j] + b * XS[i][j] + c * XS2[i][j] for j in range(len(X[0]))]
             for i in range(len(X))]
    return np.array([[float(v) for v in row] for row in X])


@pytest.mark.parametrize("steps", [1, 2, 5])
@pytest.mark.parametrize("G,norm", [
    ([[2, 3, 0], [0, 0, 6]], 7),                      # 2x3
    ([[2, 0], [3, 0], [0, 6]], 7),                    # 3x2: transpose-first path
    ([[1, 2, 2], [4, 2, -4], [4, -4, 2]], 9),         # 3x3, full rank, square
    ([[4, 4, 7], [0, 0, 0], [0, 0, 0]], 9),           # rank 1
])
def test_exact_rational_bruteforce(G, norm, steps):
    Gf = np.array(G, dtype=np.float64)
    assert int((Gf ** 2).sum()) == norm * norm
    want = _exact_ns(G, Fraction(norm), steps, QUINTIC)
    got = R.newton_schulz_ref(Gf, steps, abc=QUINTIC, eps=0.0)
    assert np.max(np.abs(got - want)) <= 1e-13 * max(1.0, np.max(np.abs(want)))


# --------------------------------------------------------------------------
# Transpose equivariance NS(G^T) = NS(G)^T (HyperParallel-FSDP section 6.6's
# transpose-first rule must not change the result).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(4, 11), (11, 4), (8, 8), (1, 7)])
def test_transpose_equivariance(shape):
    rng = np.random.default_rng(11)
    G = rng.standard_normal(shape)
    a = R.newton_schulz_ref(G.T)
    b = R.newton_schulz_ref(G).T
    assert _relerr(a, b) <= 1e-13


def test_transposed_path_used_for_tall():
    """For a tall matrix the Gram must be taken over the small side; the
    closed form holds either way, so also check against the right-Gram form."""
    rng = np.random.default_rng(3)
    G = rng.standard_normal((9, 4))
    X = G / (np.linalg.norm(G) + R.DEFAULT_EPS)
    a, b, c = QUINTIC
    for _ in range(5):
        S = X.T @ X
        X = a * X + b * X @ S + c * X @ S @ S
    assert _relerr(R.newton_schulz_ref(G), X) <= 1e-12


# --------------------------------------------------------------------------
# Batching: [B, M, N] slices are independent (HyperParallel-FSDP section 6.3)
# and normalised per slice; flattening to [B, M*N] would differ.
# --------------------------------------------------------------------------
def test_batched_equals_loop_and_slices_independent():
    rng = np.random.default_rng(21)
    X = rng.standard_normal((5, 6, 10))
    X[2] *= 1e3
    X[4] *= 1e-4
    out = R.ns_batched_ref(X)
    for i in range(5):
        assert np.array_equal(out[i], R.newton_schulz_ref(X[i]))
    Y = X.copy()
    Y[1] = rng.standard_normal((6, 10))
    out2 = R.ns_batched_ref(Y)
    for i in (0, 2, 3, 4):
        assert np.array_equal(out[i], out2[i])
    # scale invariance per slice (exact with eps = 0)
    assert _relerr(R.newton_schulz_ref(X[2], eps=0.0),
                   R.newton_schulz_ref(X[2] * 1e-3, eps=0.0)) <= 1e-13
    flat = R.newton_schulz_ref(X.reshape(5 * 6, 10)).reshape(5, 6, 10)
    assert _relerr(flat, out) > 1e-2


# --------------------------------------------------------------------------
# DMuon-2 Appendix A: with mutually orthogonal row blocks (M1 M2^T = 0) the
# Gram is block diagonal, so NS of the whole matrix equals the stacked
# iteration of each block started from M_i / (||M||_F + eps); in the exact
# polar limit it is the stacked polar factors.
# --------------------------------------------------------------------------
def _block_orthogonal(rng, n=12, r1=3, r2=4):
    Q = _orth(rng, n, n)
    M1 = rng.standard_normal((r1, 5)) @ Q[:, :5].T
    M2 = rng.standard_normal((r2, n - 5)) @ Q[:, 5:].T
    return M1, M2


def test_block_orthogonal_polar_limit():
    rng = np.random.default_rng(8)
    M1, M2 = _block_orthogonal(rng)
    assert np.max(np.abs(M1 @ M2.T)) < 1e-12
    M = np.vstack([M1, M2])

    def polar(Y):
        u, _, vt = np.linalg.svd(Y, full_matrices=False)
        return u @ vt

    got = R.newton_schulz_ref(M, 80, abc=CUBIC)
    want = np.vstack([polar(M1), polar(M2)])
    assert _relerr(got, want) <= 1e-10


def test_block_orthogonal_finite_quintic():
    rng = np.random.default_rng(9)
    M1, M2 = _block_orthogonal(rng)
    M = np.vstack([M1, M2])
    eps = R.DEFAULT_EPS
    N = np.linalg.norm(M)
    parts = []
    for Mi in (M1, M2):
        ni = np.linalg.norm(Mi)
        t = eps / (N + eps - ni)       # Y/(||Y||+eps) == Mi/(N+eps) exactly in reals
        parts.append(R.newton_schulz_ref(Mi * t, 5, eps=eps))
    assert _relerr(R.newton_schulz_ref(M, 5, eps=eps), np.vstack(parts)) <= 1e-9
    # and a non-orthogonal split does NOT decouple
    M2b = M2 + 0.3 * M1[:1].repeat(M2.shape[0], 0)
    Mb = np.vstack([M1, M2b])
    alone = R.newton_schulz_ref(M1 * (eps / (np.linalg.norm(Mb) + eps - np.linalg.norm(M1))), 5)
    assert _relerr(R.newton_schulz_ref(Mb, 5)[:M1.shape[0]], alone) > 1e-3


# --------------------------------------------------------------------------
# Special cases
# --------------------------------------------------------------------------
def test_cubic_limit_is_library_polar_factor():
    rng = np.random.default_rng(4)
    U, V = _orth(rng, 6, 6), _orth(rng, 10, 6)
    G = (U * np.linspace(1.0, 0.08, 6)) @ V.T
    got = R.newton_schulz_ref(G, 60, abc=CUBIC)
    u, _, vt = np.linalg.svd(G, full_matrices=False)
    assert _relerr(got, u @ vt) <= 1e-12


def test_steps_zero_is_normalised_input():
    rng = np.random.default_rng(6)
    G = rng.standard_normal((3, 8))
    got = R.newton_schulz_ref(G, 0)
    assert _relerr(got, G / (np.sqrt((G ** 2).sum()) + 1e-7)) <= 1e-15


def test_zero_matrix():
    out = R.newton_schulz_ref(np.zeros((4, 6)))
    assert np.all(out == 0.0) and np.all(np.isfinite(out))
    W = np.ones((4, 6))
    w2, m2, o = R.muon_step_ref(W, np.zeros((4, 6)), np.zeros((4, 6)), lr=0.02, wd=0.01)
    assert np.allclose(w2, (1 - 0.02 * 0.01) * W, rtol=0, atol=1e-15)
    assert np.all(o == 0)


def test_row_vector_closed_form():
    g = np.array([[3.0, -4.0, 12.0]])   # ||g|| = 13
    x = 13.0 / (13.0 + 1e-7)
    f = R.scalar_polynomial_ref(np.array([x]))[0]
    assert _relerr(R.newton_schulz_ref(g), f * g / 13.0) <= 1e-14
    assert _relerr(R.newton_schulz_ref(g.T), (f * g / 13.0).T) <= 1e-14


def test_scalar_polynomial_hand_values():
    # f(1) = a + b + c; f(0) = 0; f odd
    a, b, c = QUINTIC
    assert R.scalar_polynomial_ref(np.array([1.0]), 1)[0] == pytest.approx(0.7010, abs=1e-12)
    assert R.scalar_polynomial_ref(np.array([0.0]), 5)[0] == 0.0
    x = np.array([0.3, -0.3])
    y = R.scalar_polynomial_ref(x, 5)
    assert y[0] == -y[1]
    assert R.scalar_polynomial_ref(np.array([0.5]), 1)[0] == pytest.approx(
        3.4445 * 0.5 - 4.775 * 0.125 + 2.0315 * 0.03125, abs=1e-15)


# --------------------------------------------------------------------------
# Momentum (DMuon-2 section 2.1) and the update
# --------------------------------------------------------------------------
@pytest.mark.parametrize("nesterov", [False, True])
def test_momentum_geometric_series(nesterov):
    rng = np.random.default_rng(1)
    G = rng.standard_normal((3, 4))
    mu = 0.95
    M = np.zeros_like(G)
    for t in range(1, 8):
        M, D = R.momentum_ref(G, M, mu, nesterov)
        geo = (1 - mu ** t) / (1 - mu)
        assert np.allclose(M, G * geo, rtol=1e-14, atol=0)
        want_d = G * (1 + mu * geo) if nesterov else G * geo
        assert np.allclose(D, want_d, rtol=1e-14, atol=0)


def test_momentum_mu_zero():
    G = np.arange(6.0).reshape(2, 3)
    M, D = R.momentum_ref(G, np.full((2, 3), 7.0), 0.0, True)
    assert np.array_equal(M, G) and np.array_equal(D, G)


def test_update_special_cases():
    rng = np.random.default_rng(2)
    W = rng.standard_normal((4, 4))
    O = rng.standard_normal((4, 4))
    assert np.array_equal(R.update_ref(W, O, 0.0, 0.5, 3.0), W)          # lr = 0
    # W = 0: W' = -lr*s*O (sign of the step: W_{t+1} = W_t - eta*NS)
    assert np.allclose(R.update_ref(np.zeros((4, 4)), O, 0.1, 0.3, 2.0), -0.2 * O, rtol=1e-15)
    # O = 0 over t steps: (1 - lr*wd)^t W
    w = W.copy()
    for _ in range(5):
        w = R.update_ref(w, np.zeros_like(O), 0.02, 0.01, 1.0)
    assert np.allclose(w, W * (1 - 2e-4) ** 5, rtol=1e-14)


def test_scale_rules():
    assert R.scale_ref(256, 64, 0) == 2.0
    assert R.scale_ref(64, 256, 0) == 1.0
    assert R.scale_ref(64, 256, 1) == pytest.approx(3.2)
    assert R.scale_ref(14336, 4096, 0) == pytest.approx(np.sqrt(3.5))
    assert R.scale_ref(7, 9, 2) == 1.0


def test_step_uses_stored_shape_for_scale_and_transposes():
    rng = np.random.default_rng(12)
    W = rng.standard_normal((2, 9, 4)) * 0.02
    G = rng.standard_normal((2, 9, 4))
    M0 = np.zeros_like(G)
    w2, m2, o = R.muon_step_ref(W, G, M0, mu=0.9, nesterov=True, lr=0.1, wd=0.0)
    D = G + 0.9 * G
    for i in range(2):
        assert _relerr(o[i], R.newton_schulz_ref(D[i].T).T) <= 1e-13
        assert np.allclose(w2[i], W[i] - 0.1 * 1.5 * o[i], rtol=0, atol=1e-15)


def test_golden_c1_summary():
    """Regression pin: the stored summary was written by
    tests/golden/make_golden.py, which calls only the oracle."""
    import json
    import os
    from newton_schulz_gb300 import synth
    path = os.path.join(os.path.dirname(__file__), "golden", "c1_oracle_summary.json")
    with open(path) as f:
        gold = json.load(f)
    groups = synth.config_c1_numpy()
    outs = R.muon_step_groups_ref(groups, mu=0.95, nesterov=True, lr=0.02, wd=0.01)
    for gi, (w2, m2, o) in enumerate(outs):
        g = gold["groups"][gi]
        for i in range(w2.shape[0]):
            assert np.linalg.norm(o[i]) == pytest.approx(g["O_fro"][i], rel=1e-12)
            assert np.linalg.norm(w2[i]) == pytest.approx(g["W_fro"][i], rel=1e-12)
            assert o[i].ravel()[:4].tolist() == pytest.approx(g["O_head"][i], rel=1e-10, abs=1e-14)
