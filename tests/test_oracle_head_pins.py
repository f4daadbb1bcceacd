"""Pins of the oracle's prediction head and feature tokenization (no GPU).

Head ("RankMixer 详解（1）" sections 5.1-5.2, worked example section 6.4): the
page prints o_output, the head's w and b (4 decimals), the logit z, the
probability p, the loss l and dl/dz (6 decimals, from full precision) for a
sample with label 1.  The pins check the oracle against those numbers within
the error the printed rounding allows, against finite differences of its own
loss, and against the symmetries of the logistic loss.

Tokenization ("RankMixer" section 3.2 Eq. 2; "RankMixer 详解（1）" section 2.4):
slice t of the concatenated embedding, projected by token t's linear layer.
Pinned by an identity projection (the slices themselves), a brute-force
restatement in numpy, token independence and finite differences of the
backward.
"""
import numpy as np
import pytest

import oracle
from tests.golden_io import load_golden


@pytest.fixture(scope="module")
def wx():
    return load_golden("worked_example_T4.txt")


def test_head_reproduces_the_printed_worked_example(wx):
    o, w, b = wx["o"], wx["head_w"][0], wx["head_b"][0, 0]
    y = wx["label"][0]
    r = oracle.head(o, w, b, y)
    # z from 4-decimal o, w, b: each rounding moves z by at most 5e-5 times the other factor
    bound = 5e-5 * (np.abs(w).sum() + np.abs(o).sum() + 1.0)
    assert abs(r["z"][0] - wx["z"][0, 0]) <= bound
    # from the printed z (6 decimals) the printed p, l and dl/dz follow to their rounding
    rz = oracle.head(np.zeros((1, 1)), np.zeros(1), wx["z"][0, 0], y)
    assert abs(rz["p"][0] - wx["p_hat"][0, 0]) <= 1e-6
    assert abs(rz["loss"][0] - wx["loss"][0, 0]) <= 1e-6
    assert abs(rz["dz"][0] - wx["dl_dz"][0, 0]) <= 1e-6
    # dl/do = dl/dz * w ([WT] section 5.2, the head's share before the pool)
    np.testing.assert_allclose(r["dO"][0], r["dz"][0] * w, rtol=0, atol=1e-15)


def test_head_loss_symmetry_and_limits():
    z = np.array([-40.0, -3.0, -0.5, 0.0, 0.7, 5.0, 40.0])
    O = z[:, None]
    one = oracle.head(O, np.ones(1), 0.0, np.ones_like(z))
    zero = oracle.head(-O, np.ones(1), 0.0, np.zeros_like(z))
    np.testing.assert_allclose(one["loss"], zero["loss"], rtol=0, atol=1e-15)   # l(z, 1) = l(-z, 0)
    np.testing.assert_allclose(one["p"] + oracle.head(-O, np.ones(1), 0.0)["p"], 1.0, atol=1e-15)
    assert one["loss"][3] == pytest.approx(np.log(2.0), abs=1e-15)                 # p = 1/2
    assert one["loss"][0] == pytest.approx(40.0, abs=1e-12)                        # no overflow at |z| = 40
    assert one["loss"][-1] == pytest.approx(np.exp(-40.0), rel=1e-9)


def test_head_gradient_matches_finite_differences():
    r = np.random.default_rng(5)
    O = r.standard_normal((4, 6))
    w = r.standard_normal(6) * 0.5
    y = np.array([1.0, 0.0, 1.0, 0.0])
    g = oracle.head(O, w, 0.3, y)
    h = 1e-6
    for i in range(4):
        for j in range(6):
            Op, Om = O.copy(), O.copy()
            Op[i, j] += h
            Om[i, j] -= h
            fd = (oracle.head(Op, w, 0.3, y)["loss"][i] - oracle.head(Om, w, 0.3, y)["loss"][i]) / (2 * h)
            assert abs(fd - g["dO"][i, j]) <= 1e-8


@pytest.mark.parametrize("B,T,d,D", [(3, 4, 5, 8), (2, 2, 8, 8), (1, 3, 4, 6)])
def test_tokenize_against_slices_and_brute_force(B, T, d, D):
    r = np.random.default_rng(B * 100 + T)
    E = r.standard_normal((B, T * d))
    W = r.standard_normal((T, d, D))
    bias = r.standard_normal((T, D))
    X0 = oracle.tokenize(E, W, bias)
    ref = np.stack([E[:, t * d:(t + 1) * d] @ W[t] + bias[t] for t in range(T)], axis=1)
    np.testing.assert_allclose(X0, ref, rtol=1e-13, atol=1e-13)
    if d == D:   # identity projection, zero bias: the tokens are the slices themselves
        Xi = oracle.tokenize(E, np.broadcast_to(np.eye(d), (T, d, d)).copy(), np.zeros((T, D)))
        np.testing.assert_array_equal(Xi, E.reshape(B, T, d))
    # token t depends on slice t and W[t] only
    E2 = E.copy()
    E2[:, :d] += 1.0
    X2 = oracle.tokenize(E2, W, bias)
    np.testing.assert_array_equal(X2[:, 1:], X0[:, 1:])
    assert not np.allclose(X2[:, 0], X0[:, 0])


def test_tokenize_backward_matches_finite_differences():
    r = np.random.default_rng(9)
    B, T, d, D = 2, 3, 4, 5
    E = r.standard_normal((B, T * d))
    W = r.standard_normal((T, d, D))
    bias = r.standard_normal((T, D))
    G = r.standard_normal((B, T, D))
    dE, dW, db = oracle.tokenize_backward(E, W, G)
    loss = lambda: float(np.sum(G * oracle.tokenize(E, W, bias)))
    h = 1e-6
    for arr, grad in ((E, dE), (W, dW), (bias, db)):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + h
            lp = loss()
            flat[i] = keep - h
            lm = loss()
            flat[i] = keep
            assert abs((lp - lm) / (2 * h) - gflat[i]) <= 1e-7
