"""RankMixer CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain double-precision restatement of the RankMixer block forward
(``rankmixer_oracle.c``), loaded through ctypes.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA library and never
imports it.

Sources: "RankMixer: Scaling Up Ranking Models in Industrial Recommenders",
section 3.1 Eq. 1, section 3.3 Eq. 3-9, section 3.4 Eq. 10; "UniMixer: A Unified
Architecture for Scaling Laws in Recommendation Systems", section 4.3 Eq. 11-15
and Appendices A-B (UniMixing); "RankMixer 详解（1）",
sections 3.1, 3.3, 4.1, 5.1 and 5.2 (the backward pass).  Every function below forwards to the C loop
nest of the same name; the docstrings say which passage each follows.

Parity status: every function is pinned by a test under ``tests/`` (printed
worked examples, closed forms, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rankmixer_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over samples).  Returns the .so path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.oracle_token_mix.argtypes = [dp, dp, i, i, i, i]
            lib.oracle_layernorm.argtypes = [dp, dp, dp, ctypes.c_double, dp, i, i]
            lib.oracle_gelu.argtypes = [dp, dp, ctypes.c_size_t]
            lib.oracle_pffn.argtypes = [dp, dp, dp, dp, dp, dp, i, i, i, i]
            lib.oracle_block_forward.argtypes = [dp] * 11 + [ctypes.c_double, i, i, i, i]
            lib.oracle_mean_pool.argtypes = [dp, dp, i, i, i]
            lib.oracle_stack_forward.argtypes = [dp] * 11 + [ctypes.c_double, i, i, i, i, i]
            lib.oracle_moe_pffn.argtypes = [dp] * 9 + [i, i, i, i, i]
            lib.oracle_gelu_grad.argtypes = [dp, dp, ctypes.c_size_t]
            lib.oracle_layernorm_backward.argtypes = [dp, dp, dp, ctypes.c_double, dp, dp, dp, i, i]
            lib.oracle_block_backward.argtypes = [dp] * 11 + [ctypes.c_double] + [dp] * 8 + [i, i, i, i]
            lib.oracle_stack_backward.argtypes = [dp] * 11 + [ctypes.c_double] + [dp] * 8 + [i, i, i, i, i]
            lib.oracle_head.argtypes = [dp, dp, ctypes.c_double, dp, dp, dp, dp, dp, dp, i, i]
            lib.oracle_tokenize.argtypes = [dp, dp, dp, dp, i, i, i, i]
            lib.oracle_tokenize_backward.argtypes = [dp] * 6 + [i, i, i, i]
            lib.oracle_moe_pffn_train.argtypes = [dp] * 14 + [i, i, i, i, i]
            lib.oracle_sinkhorn.argtypes = [dp, dp, i, i, ctypes.c_double, i]
            lib.oracle_unimixing.argtypes = [dp, dp, dp, dp, i, i, i]
            lib.oracle_stack_forward_unimix.argtypes = [dp] * 13 + [i, ctypes.c_double, i, i, i, i, i]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [i]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def token_mix(X, H: int | None = None) -> np.ndarray:
    """TokenMixing ("RankMixer", section 3.3.1 Eq. 3-4; "RankMixer 详解（1）" section 3.1):
    out[b, h, t*q + r] = X[b, t, h*q + r] with q = D/H.  X is [B, T, D] (or [T, D])."""
    X = _f64(X)
    squeeze = X.ndim == 2
    if squeeze:
        X = X[None]
    B, T, D = X.shape
    H = T if H is None else H
    if D % H:
        raise ValueError("D must be divisible by H")
    out = np.empty((B, H, T * (D // H)), dtype=np.float64)
    _load().oracle_token_mix(_p(X), _p(out), B, T, D, H)
    return out[0] if squeeze else out


def layernorm(R, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """Row LayerNorm with biased variance ("RankMixer 详解（1）" section 3.3)."""
    R = _f64(R)
    D = R.shape[-1]
    rows = R.size // D
    g = _f64(np.ones(D) if gamma is None else gamma)
    b = _f64(np.zeros(D) if beta is None else beta)
    out = np.empty_like(R)
    _load().oracle_layernorm(_p(R), _p(g), _p(b), float(eps), _p(out), rows, D)
    return out


def gelu(u) -> np.ndarray:
    """Gelu(u) = u * Phi(u) ("RankMixer 详解（1）" section 4.1)."""
    u = _f64(u)
    out = np.empty_like(u)
    _load().oracle_gelu(_p(u), _p(out), u.size)
    return out


def pffn(S, W1, b1, W2, b2) -> np.ndarray:
    """Per-token FFN ("RankMixer" section 3.3.2 Eq. 6-9): V[b,t] = Gelu(S[b,t] W1[t] + b1[t]) W2[t] + b2[t].
    S [B,T,D], W1 [T,D,F], b1 [T,F], W2 [T,F,D], b2 [T,D]."""
    S, W1, b1, W2, b2 = map(_f64, (S, W1, b1, W2, b2))
    B, T, D = S.shape
    F = W1.shape[-1]
    V = np.empty_like(S)
    _load().oracle_pffn(_p(S), _p(W1), _p(b1), _p(W2), _p(b2), _p(V), B, T, D, F)
    return V


def block_forward(X, p: dict, eps: float = 1e-5, return_S: bool = False):
    """One RankMixer block ("RankMixer" section 3.1 Eq. 1):
    S = LN1(TokenMixing(X) + X); X' = LN2(PFFN(S) + S).  ``p`` holds one layer:
    W1 [T,D,F], b1 [T,F], W2 [T,F,D], b2 [T,D], ln1_g, ln1_b, ln2_g, ln2_b [D]."""
    X = _f64(X)
    B, T, D = X.shape
    a = {k: _f64(p[k]) for k in ("W1", "b1", "W2", "b2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")}
    F = a["W1"].shape[-1]
    Xo = np.empty_like(X)
    S = np.empty_like(X)
    _load().oracle_block_forward(_p(X), _p(Xo), _p(S), _p(a["W1"]), _p(a["b1"]), _p(a["W2"]), _p(a["b2"]),
                                 _p(a["ln1_g"]), _p(a["ln1_b"]), _p(a["ln2_g"]), _p(a["ln2_b"]),
                                 float(eps), B, T, D, F)
    return (Xo, S) if return_S else Xo


def mean_pool(X) -> np.ndarray:
    """o = (1/T) sum_t X[b, t, :] ("RankMixer" section 3.1; "RankMixer 详解（1）" section 5.1)."""
    X = _f64(X)
    B, T, D = X.shape
    o = np.empty((B, D), dtype=np.float64)
    _load().oracle_mean_pool(_p(X), _p(o), B, T, D)
    return o


def stack_forward(X0, layers: list, eps: float = 1e-5, return_XL: bool = False):
    """L stacked blocks with per-layer weights, then mean pooling ("RankMixer" section 3.1)."""
    X0 = _f64(X0)
    B, T, D = X0.shape
    L = len(layers)
    cat = {k: _f64(np.stack([np.asarray(l[k], dtype=np.float64) for l in layers]))
           for k in ("W1", "b1", "W2", "b2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")}
    F = cat["W1"].shape[-1]
    pooled = np.empty((B, D), dtype=np.float64)
    XL = np.empty_like(X0) if return_XL else None
    xl_ptr = _p(XL) if return_XL else ctypes.POINTER(ctypes.c_double)()
    _load().oracle_stack_forward(_p(X0), _p(pooled), xl_ptr, _p(cat["W1"]), _p(cat["b1"]), _p(cat["W2"]),
                                 _p(cat["b2"]), _p(cat["ln1_g"]), _p(cat["ln1_b"]), _p(cat["ln2_g"]),
                                 _p(cat["ln2_b"]), float(eps), B, T, D, F, L)
    return (pooled, XL) if return_XL else pooled


def sinkhorn(W, tau: float, iters: int) -> np.ndarray:
    """Constrained UniMixing weights ("UniMixer", section 4.3 Eq. 15): for each
    n x n matrix in ``W`` ([..., n, n]), Sinkhorn-Knopp of (W + W^T) / (2 tau):
    elementwise exp, then ``iters`` rounds of row then column normalisation."""
    W = _f64(W)
    n = W.shape[-1]
    if W.shape[-2] != n:
        raise ValueError("square matrices expected")
    count = W.size // (n * n)
    out = np.empty_like(W)
    _load().oracle_sinkhorn(_p(W), _p(out), count, n, float(tau), int(iters))
    return out


def unimixing(X, WG, WB) -> np.ndarray:
    """UniMixing ("UniMixer", section 4.3 Eq. 12-14): flatten each sample of X
    ([B, ...], L values), cut it into nb = L / bs blocks x_j, h_j = x_j WB[j],
    out_i = sum_j WG[i, j] h_j.  WG [nb, nb], WB [nb, bs, bs] (constrained
    weights); returns X's shape."""
    X = _f64(X)
    WG, WB = _f64(WG), _f64(WB)
    B = X.shape[0]
    L = X.size // B
    nb, bs = WB.shape[0], WB.shape[-1]
    if nb * bs != L or WG.shape != (nb, nb) or WB.shape != (nb, bs, bs):
        raise ValueError("UniMixing shapes: WG [nb, nb], WB [nb, bs, bs] with nb * bs = L")
    Y = np.empty_like(X)
    _load().oracle_unimixing(_p(X), _p(Y), _p(WG), _p(WB), B, L, bs)
    return Y


def stack_forward_unimix(X0, layers: list, eps: float = 1e-5, return_XL: bool = False):
    """``stack_forward`` with UniMixing ("UniMixer", section 4.3 Eq. 14) in place of
    TokenMixing in every layer: each layer dict also holds the constrained
    weights WG [nb, nb] and WB [nb, bs, bs] (nb * bs = T * D)."""
    X0 = _f64(X0)
    B, T, D = X0.shape
    L = len(layers)
    keys = ("W1", "b1", "W2", "b2", "ln1_g", "ln1_b", "ln2_g", "ln2_b", "WG", "WB")
    cat = {k: _f64(np.stack([np.asarray(l[k], dtype=np.float64) for l in layers])) for k in keys}
    F = cat["W1"].shape[-1]
    nb, bs = cat["WB"].shape[1], cat["WB"].shape[-1]
    if nb * bs != T * D or cat["WG"].shape[1:] != (nb, nb):
        raise ValueError("UniMixing shapes: WG [nb, nb], WB [nb, bs, bs] with nb * bs = T * D")
    pooled = np.empty((B, D), dtype=np.float64)
    XL = np.empty_like(X0) if return_XL else None
    xl_ptr = _p(XL) if return_XL else ctypes.POINTER(ctypes.c_double)()
    _load().oracle_stack_forward_unimix(_p(X0), _p(pooled), xl_ptr, _p(cat["W1"]), _p(cat["b1"]), _p(cat["W2"]),
                                        _p(cat["b2"]), _p(cat["ln1_g"]), _p(cat["ln1_b"]), _p(cat["ln2_g"]),
                                        _p(cat["ln2_b"]), _p(cat["WG"]), _p(cat["WB"]), bs, float(eps), B, T, D,
                                        F, L)
    return (pooled, XL) if return_XL else pooled


def moe_pffn(S, Wg, bg, eW1, eb1, eW2, eb2, return_gates: bool = False):
    """Sparse-MoE PFFN with ReLU routing ("RankMixer" section 3.4 Eq. 10), all experts
    evaluated densely.  S [B,T,D], Wg [T,D,E], bg [T,E], eW1 [T,E,D,Fe], eb1 [T,E,Fe],
    eW2 [T,E,Fe,D], eb2 [T,E,D]."""
    S, Wg, bg, eW1, eb1, eW2, eb2 = map(_f64, (S, Wg, bg, eW1, eb1, eW2, eb2))
    B, T, D = S.shape
    E = Wg.shape[-1]
    Fe = eW1.shape[-1]
    V = np.empty_like(S)
    G = np.empty((B, T, E), dtype=np.float64)
    _load().oracle_moe_pffn(_p(S), _p(Wg), _p(bg), _p(eW1), _p(eb1), _p(eW2), _p(eb2), _p(V), _p(G),
                            B, T, D, E, Fe)
    return (V, G) if return_gates else V


GRAD_KEYS = ("dW1", "db1", "dW2", "db2", "dln1_g", "dln1_b", "dln2_g", "dln2_b")
_PARAM_KEYS = ("W1", "b1", "W2", "b2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def gelu_grad(u) -> np.ndarray:
    """Gelu'(u) = Phi(u) + u phi(u) ("RankMixer 详解（1）" section 5.2)."""
    u = _f64(u)
    out = np.empty_like(u)
    _load().oracle_gelu_grad(_p(u), _p(out), u.size)
    return out


def layernorm_backward(R, gamma, Gout, eps: float = 1e-5):
    """Row LayerNorm backward ("RankMixer 详解（1）" section 5.2): returns (dR, dgamma, dbeta)
    for LN input rows R and output gradient Gout (the affine gradients summed over rows)."""
    R, Gout = _f64(R), _f64(Gout)
    D = R.shape[-1]
    g = _f64(gamma)
    dR = np.empty_like(R)
    dg = np.empty(D)
    db = np.empty(D)
    _load().oracle_layernorm_backward(_p(R), _p(g), _p(Gout), float(eps), _p(dR), _p(dg), _p(db), R.size // D, D)
    return dR, dg, db


def _grad_arrays(T, D, F, lead=()):
    shapes = {"dW1": (T, D, F), "db1": (T, F), "dW2": (T, F, D), "db2": (T, D),
              "dln1_g": (D,), "dln1_b": (D,), "dln2_g": (D,), "dln2_b": (D,)}
    return {k: np.empty(tuple(lead) + shapes[k]) for k in GRAD_KEYS}


def block_backward(X, G, p: dict, eps: float = 1e-5):
    """Backward of one block ("RankMixer 详解（1）" section 5.2) for the loss whose gradient at the
    block output is G.  Returns (dX, grads) with grads keyed by GRAD_KEYS, each summed over
    the batch: dW1 [T,D,F], db1 [T,F], dW2 [T,F,D], db2 [T,D], dln*_g / dln*_b [D]."""
    X, G = _f64(X), _f64(G)
    B, T, D = X.shape
    a = {k: _f64(p[k]) for k in _PARAM_KEYS}
    F = a["W1"].shape[-1]
    dX = np.empty_like(X)
    g = _grad_arrays(T, D, F)
    _load().oracle_block_backward(_p(X), _p(G), _p(dX), *[_p(a[k]) for k in _PARAM_KEYS], float(eps),
                                  *[_p(g[k]) for k in GRAD_KEYS], B, T, D, F)
    return dX, g


def stack_backward(X0, dpooled, layers: list, eps: float = 1e-5):
    """Backward of L stacked blocks and the mean pool ("RankMixer 详解（1）" section 5.2):
    returns (dX0, [grads of layer 0, ..., grads of layer L-1])."""
    X0, dpooled = _f64(X0), _f64(dpooled)
    B, T, D = X0.shape
    L = len(layers)
    cat = {k: _f64(np.stack([np.asarray(l[k], dtype=np.float64) for l in layers])) for k in _PARAM_KEYS}
    F = cat["W1"].shape[-1]
    dX0 = np.empty_like(X0)
    g = _grad_arrays(T, D, F, (L,))
    _load().oracle_stack_backward(_p(X0), _p(dpooled), _p(dX0), *[_p(cat[k]) for k in _PARAM_KEYS], float(eps),
                                  *[_p(g[k]) for k in GRAD_KEYS], B, T, D, F, L)
    return dX0, [{k: g[k][n] for k in GRAD_KEYS} for n in range(L)]


def head(O, w, b: float, y=None):
    """Prediction head ("RankMixer 详解（1）" sections 5.1-5.2): z = o w + b, p = sigmoid(z),
    and with labels y the per-sample BCE loss, dl/dz = p - y and dl/do = (p - y) w.
    Returns a dict with z, p (and loss, dz, dO when y is given)."""
    O, w = _f64(O), _f64(w)
    B, D = O.shape
    out = {"z": np.empty(B), "p": np.empty(B)}
    null = ctypes.POINTER(ctypes.c_double)()
    if y is None:
        _load().oracle_head(_p(O), _p(w), float(b), null, _p(out["z"]), _p(out["p"]), null, null, null, B, D)
        return out
    y = _f64(y)
    out.update(loss=np.empty(B), dz=np.empty(B), dO=np.empty_like(O))
    _load().oracle_head(_p(O), _p(w), float(b), _p(y), _p(out["z"]), _p(out["p"]), _p(out["loss"]), _p(out["dz"]),
                        _p(out["dO"]), B, D)
    return out


def tokenize(E, W, bias) -> np.ndarray:
    """Feature tokenization ("RankMixer" Eq. 2; "RankMixer 详解（1）" section 2.4): X0[b, t] =
    E[b, t d:(t + 1) d] W[t] + bias[t].  E [B, T d], W [T, d, D], bias [T, D] -> X0 [B, T, D]."""
    E, W, bias = _f64(E), _f64(W), _f64(bias)
    T, d, D = W.shape
    B = E.shape[0]
    X0 = np.empty((B, T, D))
    _load().oracle_tokenize(_p(E), _p(W), _p(bias), _p(X0), B, T, d, D)
    return X0


def tokenize_backward(E, W, dX0):
    """Gradients of the tokenization for dX0 [B, T, D]: returns (dE [B, T d], dW [T, d, D], db [T, D])."""
    E, W, dX0 = _f64(E), _f64(W), _f64(dX0)
    T, d, D = W.shape
    B = E.shape[0]
    dE, dW, db = np.empty_like(E), np.empty_like(W), np.empty((T, D))
    _load().oracle_tokenize_backward(_p(E), _p(W), _p(dX0), _p(dE), _p(dW), _p(db), B, T, d, D)
    return dE, dW, db


def moe_pffn_train(S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2) -> dict:
    """Training forward of the Sparse-MoE PFFN with dense-training / sparse-inference routers
    ("RankMixer" section 3.4 Eq. 10-11; "6.4 Rankmixer: 硬件效率优化" section 6.4.4): V from the
    training router's gates G_train; the inference router's gates G_infer, the per-sample
    regulariser lreg = sum over tokens and experts of G_infer, and the per-expert activation
    A = sum over samples and tokens of G_infer."""
    S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2 = map(_f64, (S, Wt, bt, Wi, bi, eW1, eb1, eW2, eb2))
    B, T, D = S.shape
    E = Wt.shape[-1]
    Fe = eW1.shape[-1]
    out = {"V": np.empty_like(S), "G_train": np.empty((B, T, E)), "G_infer": np.empty((B, T, E)),
           "lreg": np.empty(B), "A": np.empty(E)}
    _load().oracle_moe_pffn_train(_p(S), _p(Wt), _p(bt), _p(Wi), _p(bi), _p(eW1), _p(eb1), _p(eW2), _p(eb2),
                                  _p(out["V"]), _p(out["G_train"]), _p(out["G_infer"]), _p(out["lreg"]),
                                  _p(out["A"]), B, T, D, E, Fe)
    return out
