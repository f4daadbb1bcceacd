"""Pins of the UniMixing oracle ("UniMixer: A Unified Architecture for Scaling
Laws in Recommendation Systems", section 4.3 Eq. 11-15, Appendices A-B) to
facts fixed independently of it:

* Appendix A's printed example: with the printed global matrix G and identity
  local blocks, UniMixing is the TokenMixer of the 2 x 6 input;
* the compressibility property (W_perm = G kron I) for general T, checked
  against the separately pinned TokenMixing oracle;
* Appendix B's identity between the explicit generalised Kronecker product and
  the optimised flow (Eq. 26-29, including its transposed local weights);
* Sinkhorn-Knopp's 2 x 2 closed form (the limit keeps the cross ratio
  P11 P22 / (P12 P21) of exp(C) and is doubly stochastic), its doubly
  stochastic and symmetric limit, the row-then-column order, and its
  invariance to a constant shift of the raw weights;
* the stack with UniMixing set to the block permutation equals the RankMixer
  stack with TokenMixing.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from rankmixer_feature_interaction_gb300 import synth
from tests.golden_io import load_golden


def _block_perm(T: int) -> np.ndarray:
    """G of TokenMixing for H = T at block size D / T: input block j = t T + h
    (token t, head h) goes to output block h T + t."""
    n = T * T
    G = np.zeros((n, n))
    for j in range(n):
        t, h = divmod(j, T)
        G[h * T + t, j] = 1.0
    return G


def _eye_blocks(nb: int, bs: int) -> np.ndarray:
    return np.broadcast_to(np.eye(bs), (nb, bs, bs)).copy()


def test_appendix_a_example_is_unimixing_with_printed_factors():
    fx = load_golden("mix_2x6_perm.txt")
    X = fx["input"][None]                      # one sample, T = 2, D = 6
    Y = oracle.unimixing(X, fx["G"], _eye_blocks(4, 3))
    np.testing.assert_array_equal(Y[0], fx["mixed"])


@pytest.mark.parametrize("T,q", [(2, 1), (2, 3), (4, 2), (8, 3)])
def test_block_permutation_reproduces_tokenmixing(T, q):
    D = T * q
    rng = np.random.default_rng(T * 100 + q)
    X = rng.normal(size=(3, T, D))
    G = _block_perm(T)
    np.testing.assert_array_equal(oracle.unimixing(X, G, _eye_blocks(T * T, q)), oracle.token_mix(X))
    # compressibility: the TokenMixer's permutation matrix factors as G kron I_q
    n = T * D
    P = np.zeros((n, n))
    for j in range(n):
        e = np.zeros(n)
        e[j] = 1.0
        P[:, j] = oracle.token_mix(e.reshape(1, T, D)).reshape(-1)
    np.testing.assert_array_equal(P, np.kron(G, np.eye(q)))


@pytest.mark.parametrize("nb,bs", [(4, 3), (6, 2), (5, 4)])
def test_optimised_flow_equals_generalised_kronecker_product(nb, bs):
    rng = np.random.default_rng(nb * 10 + bs)
    WG = rng.normal(size=(nb, nb))
    WB = rng.normal(size=(nb, bs, bs))
    x = rng.normal(size=(nb * bs,))
    # Eq. 26: block (i, j) of the explicit matrix is WG[i, j] WB_j, acting on column vectors
    K = np.zeros((nb * bs, nb * bs))
    for i in range(nb):
        for j in range(nb):
            K[i * bs:(i + 1) * bs, j * bs:(j + 1) * bs] = WG[i, j] * WB[j]
    explicit = K @ x
    # Eq. 27-29: the optimised flow with x_j WB_j^T equals it
    flow = oracle.unimixing(x[None], WG, np.transpose(WB, (0, 2, 1)))[0]
    np.testing.assert_allclose(flow, explicit, rtol=0, atol=1e-12)


def test_unimixing_special_cases_and_linearity():
    rng = np.random.default_rng(5)
    nb, bs = 6, 4
    X = rng.normal(size=(2, nb * bs))
    np.testing.assert_array_equal(oracle.unimixing(X, np.eye(nb), _eye_blocks(nb, bs)), X)
    Yu = oracle.unimixing(X, np.full((nb, nb), 1.0 / nb), _eye_blocks(nb, bs))
    mean_block = X.reshape(2, nb, bs).mean(axis=1)
    np.testing.assert_allclose(Yu.reshape(2, nb, bs), np.broadcast_to(mean_block[:, None], (2, nb, bs)), atol=1e-14)
    WG, WB = rng.normal(size=(nb, nb)), rng.normal(size=(nb, bs, bs))
    X2 = rng.normal(size=X.shape)
    lhs = oracle.unimixing(2.0 * X - 3.0 * X2, WG, WB)
    rhs = 2.0 * oracle.unimixing(X, WG, WB) - 3.0 * oracle.unimixing(X2, WG, WB)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)


@pytest.mark.parametrize("tau", [1.0, 0.3, 0.05])
def test_sinkhorn_2x2_cross_ratio_and_closed_form(tau):
    rng = np.random.default_rng(int(tau * 100))
    W = rng.normal(size=(2, 2))
    a = np.exp(W[0, 0] / tau)
    c = np.exp(W[1, 1] / tau)
    b = np.exp((W[0, 1] + W[1, 0]) / (2 * tau))
    # every round rescales rows and columns, which keeps P11 P22 / (P12 P21) = a c / b^2
    for iters in (1, 5, 50):
        P = oracle.sinkhorn(W, tau, iters)
        np.testing.assert_allclose(P[0, 0] * P[1, 1] / (P[0, 1] * P[1, 0]), a * c / b ** 2, rtol=1e-9)
    if tau >= 0.3:     # the doubly stochastic limit with that cross ratio (slow to reach at small tau)
        p = np.sqrt(a * c) / (np.sqrt(a * c) + b)
        np.testing.assert_allclose(oracle.sinkhorn(W, tau, 2000), [[p, 1 - p], [1 - p, p]], rtol=0, atol=1e-12)


def test_sinkhorn_limit_doubly_stochastic_symmetric_and_order():
    rng = np.random.default_rng(11)
    W = rng.normal(size=(3, 6, 6))
    P = oracle.sinkhorn(W, 0.5, 500)
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, atol=1e-12)
    np.testing.assert_allclose(P.sum(axis=-2), 1.0, atol=1e-12)
    np.testing.assert_allclose(P, np.transpose(P, (0, 2, 1)), atol=1e-10)
    # a round ends with the column step: columns sum to 1 after one round, rows need not
    P1 = oracle.sinkhorn(W, 0.5, 1)
    np.testing.assert_allclose(P1.sum(axis=-2), 1.0, atol=1e-14)
    assert np.abs(P1.sum(axis=-1) - 1.0).max() > 1e-6
    # no rounds: the exponential of the symmetrised, tempered weights
    P0 = oracle.sinkhorn(W, 0.5, 0)
    np.testing.assert_allclose(P0, np.exp((W + np.transpose(W, (0, 2, 1))) / 1.0), rtol=1e-14)


def test_sinkhorn_shift_invariance():
    rng = np.random.default_rng(13)
    W = rng.normal(size=(5, 5))
    np.testing.assert_allclose(oracle.sinkhorn(W + 3.7, 0.2, 30), oracle.sinkhorn(W, 0.2, 30), rtol=1e-12,
                               atol=1e-15)


@pytest.mark.parametrize("T,q,k,L", [(2, 3, 2, 2), (4, 2, 2, 1)])
def test_stack_with_block_permutation_equals_tokenmixing_stack(T, q, k, L):
    D = T * q
    layers = [synth.to_f64(p) for p in synth.make_stack(T, D, k, L, 21, "f32", "cpu")]
    for p in layers:
        p["WG"] = _block_perm(T)
        p["WB"] = _eye_blocks(T * T, q)
    X0 = synth.make_input(5, T, D, 22, "f32", "cpu").double().numpy()
    pooled_u, XL_u = oracle.stack_forward_unimix(X0, layers, return_XL=True)
    pooled, XL = oracle.stack_forward(X0, layers, return_XL=True)
    np.testing.assert_allclose(XL_u, XL, atol=1e-12)
    np.testing.assert_allclose(pooled_u, pooled, atol=1e-12)
