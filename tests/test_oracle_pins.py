"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test ties one oracle function to something other than itself: a worked
example printed on the pages (fixtures under tests/golden/, each citing its
page and section), a closed form, an invariant, or a library routine in a
special case.  A plausible slip in the oracle -- a dropped term, a swapped
index, a transposed operand, the wrong variance divisor -- fails at least one.
"""
import math

import numpy as np
import pytest
from scipy.special import ndtr

import oracle

from tests.golden_io import load_golden

RNG = np.random.default_rng(20260101)


# ----------------------------------------------------------------------------
# TokenMixing ("RankMixer" section 3.3.1 Eq. 3-4)
# ----------------------------------------------------------------------------

def test_mix_A1D4_layout():
    """"RankMixer详解" section 五: 4 tokens x 8 dims, 4 heads of 2 -> rows A_h B_h C_h D_h."""
    fx = load_golden("mix_A1D4.txt", numeric=False)
    T, D, H = 4, 8, 4
    q = D // H
    X = np.arange(T * D, dtype=np.float64).reshape(T, D) + 1.0  # unique value per coordinate

    def block(label):  # "C3" -> token C (index 2), head 3 (index 2)
        t = "ABCD".index(label[0])
        h = int(label[1:]) - 1
        return X[t, h * q:(h + 1) * q]

    # the fixture's input rows must be the split of X into heads
    for t, row in enumerate(fx["input"]):
        np.testing.assert_array_equal(np.concatenate([block(l) for l in row]), X[t])
    expected = np.stack([np.concatenate([block(l) for l in row]) for row in fx["mixed"]])
    np.testing.assert_array_equal(oracle.token_mix(X, H), expected)


def test_mix_2x6_example_and_permutation_matrix():
    """"UniMixer" Appendix A: the 2x6 example, its 12x12 W_perm and W_perm = G kron I_3."""
    fx = load_golden("mix_2x6_perm.txt")
    X = fx["input"]
    np.testing.assert_array_equal(oracle.token_mix(X, 2), fx["mixed"])
    n = X.size
    P = np.zeros((n, n))
    for j in range(n):
        e = np.zeros(n)
        e[j] = 1.0
        P[:, j] = oracle.token_mix(e.reshape(X.shape), 2).reshape(-1)
    np.testing.assert_array_equal(P, fx["W_perm"])
    np.testing.assert_array_equal(fx["W_perm"], np.kron(fx["G"], np.eye(3)))


def _perm_matrix(T, D, H):
    n = T * D
    P = np.zeros((n, n))
    for j in range(n):
        e = np.zeros(n)
        e[j] = 1.0
        P[:, j] = oracle.token_mix(e.reshape(T, D), H).reshape(-1)
    return P


@pytest.mark.parametrize("T,q", [(2, 1), (2, 3), (4, 2), (8, 3), (4, 48), (16, 48), (32, 48)])
def test_mix_is_involution_when_H_equals_T(T, q):
    """"UniMixer" section 4 (symmetry of W_perm when T = H): Mix(Mix(X)) = X."""
    D = T * q
    X = RNG.standard_normal((3, T, D))
    M = oracle.token_mix(X)
    assert not np.array_equal(M, X) or T == 1
    np.testing.assert_array_equal(oracle.token_mix(M), X)


@pytest.mark.parametrize("T,D,H", [(2, 6, 2), (4, 8, 4), (3, 6, 3)])
def test_perm_matrix_properties_H_equals_T(T, D, H):
    """"UniMixer" section 4: W_perm is one-hot per row and column, doubly stochastic,
    symmetric for T = H, and W_perm = G kron I_{D/T}; "RankMixer 详解（1）" section 5.2: P^T P = I."""
    P = _perm_matrix(T, D, H)
    assert set(np.unique(P)) == {0.0, 1.0}
    np.testing.assert_array_equal(P.sum(0), np.ones(T * D))
    np.testing.assert_array_equal(P.sum(1), np.ones(T * D))
    np.testing.assert_array_equal(P, P.T)
    np.testing.assert_array_equal(P.T @ P, np.eye(T * D))
    q = D // T
    G = P[::q, ::q]
    np.testing.assert_array_equal(P, np.kron(G, np.eye(q)))


def test_perm_matrix_not_symmetric_when_H_differs_from_T():
    """"UniMixer" section 4: for T != H the permutation is not symmetric."""
    P = _perm_matrix(2, 6, 3)
    np.testing.assert_array_equal(P.T @ P, np.eye(12))
    assert not np.array_equal(P, P.T)


@pytest.mark.parametrize("T", [2, 4, 7])
def test_mix_equals_transpose_when_head_has_one_coordinate(T):
    """"RankMixer 详解（1）" section 3.1: with D = H = T the mixing is the plain transpose."""
    X = RNG.standard_normal((T, T))
    np.testing.assert_array_equal(oracle.token_mix(X), X.T)


# ----------------------------------------------------------------------------
# LayerNorm ("RankMixer 详解（1）" section 3.3)
# ----------------------------------------------------------------------------

def test_layernorm_centring_example():
    fx = load_golden("layernorm_shift.txt")
    out = oracle.layernorm(fx["rows"], eps=0.0)
    c = fx["centred"][0]
    # both rows centre to the printed vector, so their normalised rows coincide
    np.testing.assert_allclose(out[0], out[1], atol=1e-13)
    np.testing.assert_allclose(out[0], c / np.std(c), atol=1e-13)


def test_layernorm_invariants():
    """Before the affine: row mean 0 and biased variance sigma^2 / (sigma^2 + eps)."""
    eps = 1e-5
    R = RNG.standard_normal((50, 96)) * RNG.uniform(0.01, 3.0, size=(50, 1)) + RNG.standard_normal((50, 1))
    out = oracle.layernorm(R, eps=eps)
    np.testing.assert_allclose(out.mean(1), 0.0, atol=1e-12)
    var = np.var(R, axis=1)  # numpy's biased variance
    np.testing.assert_allclose(np.var(out, axis=1), var / (var + eps), rtol=1e-11)
    # affine part: gamma * normalised + beta
    g = 1.0 + 0.1 * RNG.standard_normal(96)
    b = 0.1 * RNG.standard_normal(96)
    np.testing.assert_allclose(oracle.layernorm(R, g, b, eps), out * g + b, atol=1e-12)
    # shift invariance and (eps = 0) scale invariance
    np.testing.assert_allclose(oracle.layernorm(R + 7.25, eps=eps), out, atol=1e-9)
    np.testing.assert_allclose(oracle.layernorm(3.0 * R, eps=0.0), oracle.layernorm(R, eps=0.0), atol=1e-11)


# ----------------------------------------------------------------------------
# GELU ("RankMixer 详解（1）" sections 4.1, 4.2)
# ----------------------------------------------------------------------------

def test_gelu_printed_values():
    fx = load_golden("gelu_values.txt")
    g = oracle.gelu(np.array([1.0, -1.0, 2.0, 0.0]))
    assert abs(g[0] - fx["gelu_1"][0, 0]) <= 5e-5
    assert abs(g[1] - fx["gelu_minus_1"][0, 0]) <= 5e-5
    C = g[2] - 2 * g[0] + g[3]
    assert abs(C - fx["C_1_1"][0, 0]) <= 5e-5


def test_gelu_is_u_times_normal_cdf():
    u = np.linspace(-8, 8, 2001)
    np.testing.assert_allclose(oracle.gelu(u), u * ndtr(u), rtol=1e-13, atol=1e-15)
    # odd-part identity Gelu(u) - Gelu(-u) = u, used by the closed-form PFFN pins below
    np.testing.assert_allclose(oracle.gelu(u) - oracle.gelu(-u), u, atol=1e-13)


# ----------------------------------------------------------------------------
# Worked example ("RankMixer 详解（1）" section 6, T = H = D = 4, k = 2, eps = 1e-5)
# ----------------------------------------------------------------------------

@pytest.fixture(scope="module")
def wx():
    return load_golden("worked_example_T4.txt")


def test_worked_example_mix_residual(wx):
    X0 = wx["X0"]
    # two 4-decimal roundings of the inputs plus one of the printed sum
    np.testing.assert_allclose(X0 + oracle.token_mix(X0), wx["X0_plus_mix"], atol=1.5e-4)


def test_worked_example_S0(wx):
    X0 = wx["X0"]
    Y = X0 + oracle.token_mix(X0)
    mu, var, first = wx["row1_mean_var_first"][0]
    assert abs(Y[0].mean() - mu) <= 1e-4 and abs(np.var(Y[0]) - var) <= 1e-4
    S0 = oracle.layernorm(Y, eps=1e-5)
    assert abs(S0[0, 0] - first) <= 2e-4
    np.testing.assert_allclose(S0, wx["S0"], atol=3e-4)


def test_worked_example_gelu_of_u1(wx):
    a = oracle.gelu(wx["u1"][0])
    np.testing.assert_allclose(a[[0, 3]], wx["gelu_u1_first_fourth"][0], atol=1.2e-4)


def test_worked_example_X1_and_pool(wx):
    X1 = oracle.layernorm(wx["S0"] + wx["V"], eps=1e-5)
    np.testing.assert_allclose(X1, wx["X1"], atol=3e-4)
    o = oracle.mean_pool(wx["X1"][None])[0]
    np.testing.assert_allclose(o, wx["o"][0], atol=1e-4)
    z = o @ wx["head_w"][0] + wx["head_b"][0, 0]
    assert abs(z - wx["z"][0, 0]) <= 5e-4


# ----------------------------------------------------------------------------
# Per-token FFN ("RankMixer" section 3.3.2 Eq. 6-9): closed forms from the GELU
# odd-part identity.  With W1_t = [A_t, -A_t], b1_t = [c_t, -c_t], W2_t = [I; -I]:
#   v_t = Gelu(s A_t + c_t) - Gelu(-(s A_t + c_t)) + b2_t = s A_t + c_t + b2_t;
# with W1_t = [I, -I], b1 = 0, W2_t = [A_t; -A_t]:  v_t = s A_t + b2_t.
# A_t is random, non-symmetric and distinct per token, so a transposed
# operand, a wrong token index or a dropped bias all change the result.
# ----------------------------------------------------------------------------

def _identity_trick_layer1(T, D, rng):
    A = rng.standard_normal((T, D, D)) / math.sqrt(D)
    c = 0.1 * rng.standard_normal((T, D))
    W1 = np.concatenate([A, -A], axis=2)            # [T, D, 2D]
    b1 = np.concatenate([c, -c], axis=1)            # [T, 2D]
    I = np.broadcast_to(np.eye(D), (T, D, D))
    W2 = np.concatenate([I, -I], axis=1)            # [T, 2D, D]
    b2 = 0.1 * rng.standard_normal((T, D))
    return A, c, W1, b1, W2, b2


@pytest.mark.parametrize("B,T,D", [(3, 4, 8), (2, 5, 6), (2, 16, 48)])
def test_pffn_closed_form_first_layer_matrix(B, T, D):
    rng = np.random.default_rng(B * 1000 + T * 10 + D)
    A, c, W1, b1, W2, b2 = _identity_trick_layer1(T, D, rng)
    S = rng.standard_normal((B, T, D))
    expect = np.einsum("btd,tde->bte", S, A) + c[None] + b2[None]
    np.testing.assert_allclose(oracle.pffn(S, W1, b1, W2, b2), expect, atol=1e-11)


@pytest.mark.parametrize("B,T,D", [(3, 4, 8), (2, 3, 5)])
def test_pffn_closed_form_second_layer_matrix(B, T, D):
    rng = np.random.default_rng(7 + B + T + D)
    A = rng.standard_normal((T, D, D)) / math.sqrt(D)
    I = np.broadcast_to(np.eye(D), (T, D, D))
    W1 = np.concatenate([I, -I], axis=2)
    b1 = np.zeros((T, 2 * D))
    W2 = np.concatenate([A, -A], axis=1)
    b2 = 0.1 * rng.standard_normal((T, D))
    S = rng.standard_normal((B, T, D))
    expect = np.einsum("btd,tde->bte", S, A) + b2[None]
    np.testing.assert_allclose(oracle.pffn(S, W1, b1, W2, b2), expect, atol=1e-11)


def test_pffn_tokens_are_independent():
    """Changing token t's weights changes only row t of the output (parameter isolation)."""
    rng = np.random.default_rng(3)
    B, T, D, F = 2, 4, 6, 12
    W1 = rng.standard_normal((T, D, F)); b1 = rng.standard_normal((T, F))
    W2 = rng.standard_normal((T, F, D)); b2 = rng.standard_normal((T, D))
    S = rng.standard_normal((B, T, D))
    V = oracle.pffn(S, W1, b1, W2, b2)
    W1b = W1.copy(); W1b[2] += 0.5
    V2 = oracle.pffn(S, W1b, b1, W2, b2)
    changed = np.any(V2 != V, axis=(0, 2))
    assert changed.tolist() == [False, False, True, False]


# ----------------------------------------------------------------------------
# Block and stack ("RankMixer" section 3.1 Eq. 1)
# ----------------------------------------------------------------------------

def _ln_params(D, rng):
    return dict(ln1_g=1 + 0.1 * rng.standard_normal(D), ln1_b=0.1 * rng.standard_normal(D),
                ln2_g=1 + 0.1 * rng.standard_normal(D), ln2_b=0.1 * rng.standard_normal(D))


@pytest.mark.parametrize("B,T,q", [(3, 4, 2), (2, 8, 3)])
def test_block_wiring_with_closed_form_pffn(B, T, q):
    """S = LN1(Mix(X) + X) with the LN1 affine; X' = LN2(PFFN(S) + S) with the LN2 affine,
    PFFN in closed form, so the residual must be S (not X) and the LN pairs not swapped."""
    D = T * q
    rng = np.random.default_rng(B + T + q)
    A, c, W1, b1, W2, b2 = _identity_trick_layer1(T, D, rng)
    p = dict(W1=W1, b1=b1, W2=W2, b2=b2, **_ln_params(D, rng))
    X = rng.standard_normal((B, T, D))
    Xo, S = oracle.block_forward(X, p, eps=1e-5, return_S=True)
    S_expect = oracle.layernorm(oracle.token_mix(X) + X, p["ln1_g"], p["ln1_b"], 1e-5)
    np.testing.assert_allclose(S, S_expect, atol=1e-12)
    V = np.einsum("btd,tde->bte", S, A) + c[None] + b2[None]
    np.testing.assert_allclose(Xo, oracle.layernorm(V + S, p["ln2_g"], p["ln2_b"], 1e-5), atol=1e-10)


def test_stack_is_composition_then_mean_pool():
    rng = np.random.default_rng(11)
    B, T, D, F = 3, 4, 8, 16
    layers = []
    for _ in range(2):
        layers.append(dict(W1=rng.standard_normal((T, D, F)) / math.sqrt(D), b1=0.1 * rng.standard_normal((T, F)),
                           W2=rng.standard_normal((T, F, D)) / math.sqrt(F), b2=0.1 * rng.standard_normal((T, D)),
                           **_ln_params(D, rng)))
    X = rng.standard_normal((B, T, D))
    pooled, XL = oracle.stack_forward(X, layers, return_XL=True)
    X1 = oracle.block_forward(X, layers[0])
    X2 = oracle.block_forward(X1, layers[1])
    np.testing.assert_allclose(XL, X2, atol=1e-13)
    np.testing.assert_allclose(pooled, X2.mean(axis=1), atol=1e-13)


# ----------------------------------------------------------------------------
# Sparse-MoE PFFN ("RankMixer" section 3.4 Eq. 10)
# ----------------------------------------------------------------------------

def test_moe_all_gates_closed_gives_zero():
    rng = np.random.default_rng(5)
    B, T, D, E, Fe = 2, 3, 4, 3, 6
    S = rng.standard_normal((B, T, D))
    V, G = oracle.moe_pffn(S, np.zeros((T, D, E)), -np.ones((T, E)),
                           rng.standard_normal((T, E, D, Fe)), rng.standard_normal((T, E, Fe)),
                           rng.standard_normal((T, E, Fe, D)), rng.standard_normal((T, E, D)), return_gates=True)
    assert np.all(G == 0.0) and np.all(V == 0.0)


def test_moe_closed_form_with_known_gates():
    """Gates ReLU(bg) from a zero router matrix; experts in closed form s A_te + c_te + b2_te."""
    rng = np.random.default_rng(6)
    B, T, D, E = 3, 4, 5, 4
    A = rng.standard_normal((T, E, D, D)) / math.sqrt(D)
    c = 0.1 * rng.standard_normal((T, E, D))
    eW1 = np.concatenate([A, -A], axis=3)
    eb1 = np.concatenate([c, -c], axis=2)
    I = np.broadcast_to(np.eye(D), (T, E, D, D))
    eW2 = np.concatenate([I, -I], axis=2)
    eb2 = 0.1 * rng.standard_normal((T, E, D))
    bg = rng.standard_normal((T, E))
    S = rng.standard_normal((B, T, D))
    V, G = oracle.moe_pffn(S, np.zeros((T, D, E)), bg, eW1, eb1, eW2, eb2, return_gates=True)
    g = np.maximum(bg, 0.0)
    np.testing.assert_array_equal(G, np.broadcast_to(g, (B, T, E)))
    expert = np.einsum("btd,tedf->btef", S, A) + c[None] + eb2[None]
    np.testing.assert_allclose(V, np.einsum("te,btef->btf", g, expert), atol=1e-11)


def test_moe_router_is_linear_then_relu():
    rng = np.random.default_rng(8)
    B, T, D, E, Fe = 4, 3, 6, 5, 4
    S = rng.standard_normal((B, T, D))
    Wg = rng.standard_normal((T, D, E))
    bg = rng.standard_normal((T, E))
    _, G = oracle.moe_pffn(S, Wg, bg, np.zeros((T, E, D, Fe)), np.zeros((T, E, Fe)),
                           np.zeros((T, E, Fe, D)), np.zeros((T, E, D)), return_gates=True)
    h = np.einsum("btd,tde->bte", S, Wg) + bg[None]
    np.testing.assert_allclose(G, np.maximum(h, 0.0), atol=1e-12)
    assert (G == 0).any() and (G > 0).any()


def test_moe_single_open_expert_is_a_dense_pffn():
    rng = np.random.default_rng(9)
    B, T, D, Fe = 2, 3, 4, 8
    S = rng.standard_normal((B, T, D))
    W1 = rng.standard_normal((T, 1, D, Fe)); b1 = rng.standard_normal((T, 1, Fe))
    W2 = rng.standard_normal((T, 1, Fe, D)); b2 = rng.standard_normal((T, 1, D))
    V = oracle.moe_pffn(S, np.zeros((T, D, 1)), np.ones((T, 1)), W1, b1, W2, b2)
    np.testing.assert_allclose(V, oracle.pffn(S, W1[:, 0], b1[:, 0], W2[:, 0], b2[:, 0]), atol=1e-12)


# ----------------------------------------------------------------------------
# DTSI-MoE training forward ("RankMixer" section 3.4 Eq. 10-11; "6.4 Rankmixer:
# 硬件效率优化" section 6.4.4): V from h_train's gates, the regulariser from
# h_infer's.  Pinned against the (separately pinned) inference MoE oracle run
# with each router, and against the definition of L_reg and A_j as sums of the
# inference gates that oracle returns.
# ----------------------------------------------------------------------------

def _moe_case(B, T, D, E, Fe, seed):
    r = np.random.default_rng(seed)
    S = r.standard_normal((B, T, D))
    Wt = r.standard_normal((T, D, E)) / np.sqrt(D)
    Wi = r.standard_normal((T, D, E)) / np.sqrt(D)
    bt = 0.2 * r.standard_normal((T, E))
    bi = -0.5 + 0.1 * r.standard_normal((T, E))
    eW1 = r.standard_normal((T, E, D, Fe)) / np.sqrt(D)
    eb1 = 0.1 * r.standard_normal((T, E, Fe))
    eW2 = r.standard_normal((T, E, Fe, D)) / np.sqrt(Fe)
    eb2 = 0.1 * r.standard_normal((T, E, D))
    return S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2


def test_moe_train_forward_uses_the_training_router_and_regularises_the_inference_one():
    S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2 = _moe_case(5, 3, 8, 4, 6, 71)
    r = oracle.moe_pffn_train(S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2)
    V_train, G_train = oracle.moe_pffn(S, Wt, bt, eW1, eb1, eW2, eb2, return_gates=True)
    V_infer, G_infer = oracle.moe_pffn(S, Wi, bi, eW1, eb1, eW2, eb2, return_gates=True)
    np.testing.assert_array_equal(r["V"], V_train)
    np.testing.assert_array_equal(r["G_train"], G_train)
    np.testing.assert_allclose(r["G_infer"], G_infer, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["lreg"], G_infer.sum(axis=(1, 2)), rtol=1e-14)
    np.testing.assert_allclose(r["A"], G_infer.sum(axis=(0, 1)), rtol=1e-14)
    assert not np.allclose(r["V"], V_infer)            # the forward does not follow h_infer
    # the regulariser is a sum of ReLU outputs: zero exactly when every inference gate is closed
    z = oracle.moe_pffn_train(S, Wt, bt, Wi, bi - 100.0, eW1, eb1, eW2, eb2)
    assert np.all(z["lreg"] == 0.0) and np.all(z["A"] == 0.0)
    np.testing.assert_array_equal(z["V"], r["V"])
