"""Pins of the oracle's backward pass against what the pages and mathematics fix (no GPU).

The backward formulas restate "RankMixer 详解（1）" section 5.2 (the FFN chain
rule, Gelu' = Phi + u phi, the LayerNorm input gradient, P^T for the mixing
and (P^T + I) through the first residual, g_o / T through the mean pool).
The page prints no gradient of the block itself, so the pins are:

* central finite differences of the oracle's forward pass (pinned on its own
  by the printed worked example and closed forms) for every entry of every
  parameter and of the input, at tiny shapes: a dropped term, a wrong sign or
  a transposed weight in the backward fails them;
* closed forms and invariants: Gelu'(0) = 1/2, Gelu'(u) + Gelu'(-u) = 1, the
  LayerNorm input gradient is orthogonal to the all-ones row (shift
  invariance) and, with eps = 0, to the row itself (scale invariance).
"""
import numpy as np
import pytest

import oracle

EPS = 1e-5


def _params(T, D, F, seed, gamma_spread=0.3):
    r = np.random.default_rng(seed)
    return {
        "W1": r.standard_normal((T, D, F)) / np.sqrt(D),
        "b1": 0.1 * r.standard_normal((T, F)),
        "W2": r.standard_normal((T, F, D)) / np.sqrt(F),
        "b2": 0.1 * r.standard_normal((T, D)),
        "ln1_g": 1.0 + gamma_spread * r.standard_normal(D),
        "ln1_b": 0.1 * r.standard_normal(D),
        "ln2_g": 1.0 + gamma_spread * r.standard_normal(D),
        "ln2_b": 0.1 * r.standard_normal(D),
    }


def _fd(f, x, h=1e-5):
    """Central differences of the scalar f() with respect to every entry of x (in place)."""
    g = np.empty_like(x)
    flat = x.reshape(-1)
    gf = g.reshape(-1)
    for i in range(flat.size):
        keep = flat[i]
        flat[i] = keep + h
        fp = f()
        flat[i] = keep - h
        fm = f()
        flat[i] = keep
        gf[i] = (fp - fm) / (2 * h)
    return g


def _close(analytic, numeric, tol=2e-7):
    scale = max(1.0, float(np.max(np.abs(numeric))))
    err = float(np.max(np.abs(analytic - numeric)))
    assert err <= tol * scale, f"max |analytic - fd| = {err:.3e} (scale {scale:.3e})"


# ----------------------------------------------------------------------------
# GELU derivative
# ----------------------------------------------------------------------------

def test_gelu_grad_closed_values_and_symmetry():
    u = np.linspace(-6, 6, 241)
    g = oracle.gelu_grad(u)
    assert oracle.gelu_grad(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(g + oracle.gelu_grad(-u), 1.0, rtol=0, atol=1e-15)
    # far tails: Gelu(u) -> u (slope 1) for large u and -> 0 (slope 0) for very negative u
    assert abs(oracle.gelu_grad(np.array([12.0]))[0] - 1.0) < 1e-15
    assert abs(oracle.gelu_grad(np.array([-12.0]))[0]) < 1e-15
    # the derivative exceeds 1 just above 0 (the GELU overshoots slope 1 near u ~ 1.4)
    assert g.max() > 1.12 and g.max() < 1.13


def test_gelu_grad_matches_finite_differences_of_gelu():
    u = np.linspace(-5, 5, 101) + 0.013
    h = 1e-6
    fd = (oracle.gelu(u + h) - oracle.gelu(u - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_grad(u), fd, rtol=0, atol=1e-8)


# ----------------------------------------------------------------------------
# LayerNorm backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("D", [4, 8, 48])
def test_layernorm_backward_matches_finite_differences(D):
    r = np.random.default_rng(D)
    R = 2.0 * r.standard_normal((3, D)) + 0.7
    gamma = 1.0 + 0.3 * r.standard_normal(D)
    beta = 0.1 * r.standard_normal(D)
    Gout = r.standard_normal((3, D))
    dR, dg, db = oracle.layernorm_backward(R, gamma, Gout, EPS)
    loss = lambda: float(np.sum(Gout * oracle.layernorm(R, gamma, beta, EPS)))
    _close(dR, _fd(loss, R))
    _close(dg, _fd(loss, gamma))
    _close(db, _fd(loss, beta))


def test_layernorm_backward_invariants():
    r = np.random.default_rng(3)
    R = 3.0 * r.standard_normal((5, 16)) - 1.0
    gamma = 1.0 + 0.2 * r.standard_normal(16)
    Gout = r.standard_normal((5, 16))
    dR, _, db = oracle.layernorm_backward(R, gamma, Gout, EPS)
    # LN(r + c) = LN(r): the input gradient has no component along the all-ones row
    np.testing.assert_allclose(dR.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(db, Gout.sum(axis=0), atol=1e-12)
    # with eps = 0, LN(alpha r) = LN(r): the gradient is also orthogonal to r
    dR0, _, _ = oracle.layernorm_backward(R, gamma, Gout, 0.0)
    np.testing.assert_allclose(np.sum(dR0 * R, axis=1), 0.0, atol=1e-11)
    # ... and not with eps > 0 on a row of small variance (the eps term is kept)
    Rs = 1e-3 * R
    dRs, _, _ = oracle.layernorm_backward(Rs, gamma, Gout, EPS)
    assert np.max(np.abs(np.sum(dRs * Rs, axis=1))) > 1e-6


# ----------------------------------------------------------------------------
# Block and stack backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("B,T,q,k", [(2, 2, 2, 2), (3, 4, 2, 2), (2, 3, 1, 3)])
def test_block_backward_matches_finite_differences(B, T, q, k):
    D = T * q
    F = k * D
    p = _params(T, D, F, seed=100 + B * T)
    r = np.random.default_rng(7 + T)
    X = r.standard_normal((B, T, D))
    G = r.standard_normal((B, T, D))
    dX, g = oracle.block_backward(X, G, p, EPS)
    loss = lambda: float(np.sum(G * oracle.block_forward(X, p, EPS)))
    _close(dX, _fd(loss, X))
    names = {"W1": "dW1", "b1": "db1", "W2": "dW2", "b2": "db2",
             "ln1_g": "dln1_g", "ln1_b": "dln1_b", "ln2_g": "dln2_g", "ln2_b": "dln2_b"}
    for pk, gk in names.items():
        _close(g[gk], _fd(loss, p[pk]))


def test_block_backward_is_a_sum_over_samples():
    """Parameter gradients of a batch are the sums of the per-sample gradients;
    the input gradient of a sample depends on that sample alone."""
    T, q, k, B = 4, 2, 2, 5
    D, F = T * q, k * T * q
    p = _params(T, D, F, seed=11)
    r = np.random.default_rng(12)
    X = r.standard_normal((B, T, D))
    G = r.standard_normal((B, T, D))
    dX, g = oracle.block_backward(X, G, p, EPS)
    acc = None
    for b in range(B):
        dXb, gb = oracle.block_backward(X[b:b + 1], G[b:b + 1], p, EPS)
        np.testing.assert_allclose(dXb[0], dX[b], rtol=0, atol=1e-13)
        acc = gb if acc is None else {kk: acc[kk] + gb[kk] for kk in acc}
    for kk in g:
        np.testing.assert_allclose(g[kk], acc[kk], rtol=0, atol=1e-12)


def test_block_backward_of_the_residual_paths_alone():
    """With W2 = 0 and b2 = 0 the FFN output is zero, so X' = LN2(S) and the FFN weights
    W1, b1 receive no gradient; with G orthogonal to every LN2 input direction
    that survives (a constant row times gamma2^-1 after centring) nothing flows at all."""
    T, q, k, B = 4, 2, 2, 3
    D, F = T * q, k * T * q
    p = _params(T, D, F, seed=21)
    p["W2"][:] = 0.0
    p["b2"][:] = 0.0
    r = np.random.default_rng(22)
    X = r.standard_normal((B, T, D))
    G = r.standard_normal((B, T, D))
    _, g = oracle.block_backward(X, G, p, EPS)
    assert np.all(g["dW1"] == 0.0) and np.all(g["db1"] == 0.0)
    # G = c / gamma2 (a constant direction before the affine) is absorbed by the LN2 centring
    Gc = np.broadcast_to(1.0 / p["ln2_g"], (B, T, D)).copy()
    dX, g2 = oracle.block_backward(X, Gc, p, EPS)
    np.testing.assert_allclose(dX, 0.0, atol=1e-12)
    np.testing.assert_allclose(g2["dW2"], 0.0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 2])
def test_stack_backward_matches_finite_differences(L):
    B, T, q, k = 2, 2, 2, 2
    D, F = T * q, k * T * q
    layers = [_params(T, D, F, seed=200 + n) for n in range(L)]
    r = np.random.default_rng(31)
    X0 = r.standard_normal((B, T, D))
    dP = r.standard_normal((B, D))
    dX0, grads = oracle.stack_backward(X0, dP, layers, EPS)
    loss = lambda: float(np.sum(dP * oracle.stack_forward(X0, layers, EPS)))
    _close(dX0, _fd(loss, X0))
    for n in range(L):
        for pk, gk in (("W1", "dW1"), ("b2", "db2"), ("ln1_g", "dln1_g"), ("ln2_b", "dln2_b")):
            _close(grads[n][gk], _fd(loss, layers[n][pk]))


def test_stack_backward_pool_share():
    """The mean pool gives every token row g_o / T: with L = 1 the stack backward
    equals the block backward fed G[b, t] = dpooled[b] / T."""
    B, T, q, k = 3, 4, 2, 2
    D, F = T * q, k * T * q
    p = _params(T, D, F, seed=41)
    r = np.random.default_rng(42)
    X0 = r.standard_normal((B, T, D))
    dP = r.standard_normal((B, D))
    dX0, grads = oracle.stack_backward(X0, dP, [p], EPS)
    G = np.repeat(dP[:, None, :] / T, T, axis=1)
    dXb, gb = oracle.block_backward(X0, G, p, EPS)
    np.testing.assert_array_equal(dX0, dXb)
    for kk in gb:
        np.testing.assert_array_equal(grads[0][kk], gb[kk])
