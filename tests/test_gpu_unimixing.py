"""GPU parity of UniMixing ("UniMixer: A Unified Architecture for Scaling Laws in
Recommendation Systems", section 4.3 Eq. 11-15) against the oracle: the
Sinkhorn-Knopp constrained weights, the mixing alone, and the block and stack
forward with UniMixing in place of TokenMixing.  Every expected value comes from
the oracle run on the raw weights (its own constrained weights), never from the
library."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer
from tests.helpers import assert_bf16_rounding, check

pytestmark = pytest.mark.gpu

DEV = "cuda"
ITERS = 20


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _constrained(WG, WB, tau, iters=ITERS):
    return oracle.sinkhorn(_np(WG), tau, iters), oracle.sinkhorn(_np(WB), tau, iters)


def _block_perm(T: int) -> np.ndarray:
    G = np.zeros((T * T, T * T))
    for j in range(T * T):
        t, h = divmod(j, T)
        G[h * T + t, j] = 1.0
    return G


@pytest.mark.parametrize("dtype,T,D,bs,tau", [
    ("bf16", 8, 512, 64, 1.0),
    ("bf16", 32, 1536, 48, 0.05),    # the 1B shape at the pages' final temperature
    ("f32", 4, 8, 2, 0.3),
])
def test_constrained_weights_match_oracle(dtype, T, D, bs, tau):
    layers = synth.make_stack(T, D, 2, 1, 3, dtype, DEV)
    m = RankMixer(T, D, 2, layers, dtype=dtype, max_batch=16)
    WG, WB = synth.make_unimix_weights(T, D, bs, 4, DEV)
    m.set_unimixing(0, WG, WB, tau=tau, iters=ITERS)
    gWG, gWB = m.unimixing_weights(0)
    torch.cuda.synchronize()
    oWG, oWB = _constrained(WG, WB, tau)
    check(gWG, oWG, "f32", f"WG T={T} D={D} bs={bs} tau={tau}")
    check(gWB, oWB, "f32", f"WB T={T} D={D} bs={bs} tau={tau}")
    # doubly stochastic in the columns after the last (column) step
    np.testing.assert_allclose(_np(gWG).sum(axis=0), 1.0, atol=1e-4)
    np.testing.assert_allclose(_np(gWB).sum(axis=1), 1.0, atol=1e-4)


@pytest.mark.parametrize("dtype,path,T,D,bs,B,tau", [
    ("bf16", "auto", 8, 512, 64, 301, 1.0),     # tensor-core global product, ragged N, fast local step
    ("bf16", "auto", 8, 512, 32, 129, 0.05),    # nb = 128, sparse weights
    ("bf16", "auto", 32, 1536, 48, 40, 0.3),    # the 1B shape (nb = 1024, bs = D / T)
    ("bf16", "auto", 4, 24, 6, 50, 1.0),        # bs not a multiple of 4, nb = 16: generic kernels
    ("f32", "auto", 4, 8, 2, 64, 1.0),          # the tiny float32 configuration
    ("f32", "auto", 8, 64, 8, 100, 0.3),
])
def test_unimixing_op_matches_oracle(dtype, path, T, D, bs, B, tau):
    layers = synth.make_stack(T, D, 2, 1, 5, dtype, DEV)
    m = RankMixer(T, D, 2, layers, dtype=dtype, max_batch=B, gemm_path=path)
    WG, WB = synth.make_unimix_weights(T, D, bs, 6 + bs, DEV)
    m.set_unimixing(0, WG, WB, tau=tau, iters=ITERS)
    X = synth.make_input(B, T, D, 7, dtype, DEV)
    Y = m.unimixing(0, X, out_dtype="f32")
    Yc = m.unimixing(0, X)                     # the context dtype
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    oWG, oWB = _constrained(WG, WB, tau)
    ref = oracle.unimixing(_np(X), oWG, oWB)
    check(Y, ref, dtype, f"unimixing {dtype} T={T} D={D} bs={bs} B={B} tau={tau}")
    if dtype == "bf16":
        assert_bf16_rounding(Yc, Y, "unimixing output")
    else:
        assert torch.equal(Yc, Y)


@pytest.mark.parametrize("dtype,T,D,k,B,bs", [
    ("bf16", 8, 512, 2, 200, 64),
    ("bf16", 16, 768, 4, 130, 48),     # the 100M width, bs = D / T
    ("f32", 4, 8, 2, 64, 2),
])
def test_stack_and_block_with_unimixing_match_oracle(dtype, T, D, k, B, bs):
    L = 2
    layers = synth.make_stack(T, D, k, L, 9, dtype, DEV)
    m = RankMixer(T, D, k, layers, dtype=dtype, max_batch=B)
    WG, WB = synth.make_unimix_weights(T, D, bs, 10, DEV)
    tau = 0.3
    m.set_unimixing(0, WG, WB, tau=tau, iters=ITERS)          # layer 1 keeps TokenMixing
    X0 = synth.make_input(B, T, D, 11, dtype, DEV)
    pooled, XL = m.stack_forward(X0, return_XL=True, xl_dtype="f32")
    X1 = m.block_forward(0, X0, out_dtype="f32")
    if dtype == "bf16":
        _, XLb = m.stack_forward(X0, return_XL=True)
        X1b = m.block_forward(0, X0)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    if dtype == "bf16":
        assert_bf16_rounding(XLb, XL, "X_L with UniMixing")
        assert_bf16_rounding(X1b, X1, "block 0 with UniMixing")
    oWG, oWB = _constrained(WG, WB, tau)
    ref = synth.to_f64(layers)
    ref[0]["WG"], ref[0]["WB"] = oWG, oWB
    q = D // T
    ref[1]["WG"] = _block_perm(T)                              # TokenMixing, as a UniMixing special case
    ref[1]["WB"] = np.broadcast_to(np.eye(q), (T * T, q, q)).copy()
    assert q == bs      # the oracle stack takes one block size for every layer
    o_pooled, o_XL = oracle.stack_forward_unimix(_np(X0), ref, return_XL=True)
    check(pooled, o_pooled, dtype if dtype == "f32" else "bf16", f"pooled {dtype} T={T} D={D}")
    check(XL, o_XL, dtype, f"X_L {dtype} T={T} D={D}")
    _, o_X1 = oracle.stack_forward_unimix(_np(X0), ref[:1], return_XL=True)
    check(X1, o_X1, dtype, f"block 0 {dtype} T={T} D={D}")


def test_full_size_stack_sampled():
    """The 1B shape at B = 4096 with UniMixing in both layers (bs = 48), checked
    on a sample of rows against the oracle."""
    T, D, k, B, bs = 32, 1536, 4, 4096, 48
    layers = synth.make_stack(T, D, k, 2, 13, "bf16", DEV)
    m = RankMixer(T, D, k, layers, dtype="bf16", max_batch=B)
    raw = [synth.make_unimix_weights(T, D, bs, 14 + n, DEV) for n in range(2)]
    for n, (WG, WB) in enumerate(raw):
        m.set_unimixing(n, WG, WB, tau=0.3, iters=ITERS)
    X0 = synth.make_input(B, T, D, 15, "bf16", DEV)
    pooled = m.stack_forward(X0)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    idx = np.array([0, 1, 777, 2048, 4095])
    ref = synth.to_f64(layers)
    for n, (WG, WB) in enumerate(raw):
        ref[n]["WG"], ref[n]["WB"] = _constrained(WG, WB, 0.3)
    o_pooled = oracle.stack_forward_unimix(_np(X0[idx]), ref)
    check(pooled[idx], o_pooled, "bf16", "pooled, 1B shape with UniMixing, sampled rows")


def test_unimixing_argument_errors():
    T, D = 4, 64
    layers = synth.make_stack(T, D, 2, 1, 17, "bf16", DEV)
    m = RankMixer(T, D, 2, layers, dtype="bf16", max_batch=8)
    WG, WB = synth.make_unimix_weights(T, D, 16, 18, DEV)
    X = synth.make_input(8, T, D, 19, "bf16", DEV)
    with pytest.raises(_lib.RankMixerError) as e:              # TokenMixing layer
        m.unimixing(0, X)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:              # bs does not divide T D
        _lib.rm_set_unimixing(m.ctx, 0, WG.data_ptr(), WB.data_ptr(), 7, 1.0, 5, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:              # tau <= 0
        _lib.rm_set_unimixing(m.ctx, 0, WG.data_ptr(), WB.data_ptr(), 16, 0.0, 5, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:              # layer out of range
        _lib.rm_set_unimixing(m.ctx, 1, WG.data_ptr(), WB.data_ptr(), 16, 1.0, 5, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    # the allocation-free entry point runs TokenMixing layers only
    m.set_unimixing(0, WG, WB, tau=1.0, iters=5)
    Y = torch.empty_like(X)
    with pytest.raises(_lib.RankMixerError) as e:
        _lib.rm_block_forward_noalloc(m.ctx, 0, X.data_ptr(), Y.data_ptr(), X.shape[0], 0)
    assert e.value.status == _lib.RM_ERR_UNSUPPORTED
    # training contexts refuse UniMixing layers in their training calls
    mt = RankMixer(T, D, 2, layers, dtype="bf16", max_batch=8, training=True)
    mt.set_unimixing(0, WG, WB, tau=1.0, iters=5)
    with pytest.raises(_lib.RankMixerError) as e:
        mt.stack_forward_train(X)
    assert e.value.status == _lib.RM_ERR_UNSUPPORTED


_LOCAL_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
from rankmixer_feature_interaction_gb300 import synth
from rankmixer_feature_interaction_gb300.api import RankMixer
out = {{}}
for T, D, bs, B, Bcap in {shapes}:
    layers = synth.make_stack(T, D, 2, 2, 21, "bf16", "cuda")
    m = RankMixer(T, D, 2, layers, dtype="bf16", max_batch=Bcap)
    for n in range(2):
        WG, WB = synth.make_unimix_weights(T, D, bs, 22 + n, "cuda")
        m.set_unimixing(n, WG, WB, tau=0.3, iters=5)
    X = synth.make_input(B, T, D, 24, "bf16", "cuda")
    Y = m.unimixing(0, X, out_dtype="f32")                            # bf16 samples in
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")   # layer 1: fp16 samples in
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    key = f"{{T}}_{{D}}_{{bs}}_{{B}}"
    out["Y_" + key] = Y.cpu().numpy()
    out["XL_" + key] = XL.cpu().numpy()
    out["pooled_" + key] = pooled.float().cpu().numpy()
    m.close()
np.savez(sys.argv[1], **out)
print("ok")
"""

# (T, D, bs, B, max_batch): every tensor-core block size, a partial last group of
# blocks (nb = 25), ragged sample tiles, many items per CTA at the 1B shape
_LOCAL_SHAPES = [(8, 512, 64, 301, 301), (8, 512, 32, 129, 200), (32, 1536, 48, 700, 700), (5, 240, 48, 77, 100),
                 (4, 64, 16, 33, 33), (16, 768, 48, 130, 130)]


def test_staged_local_step_bit_identical_to_register_kernel(tmp_path):
    """The local step staged through shared memory by bulk copies and the
    register-prefetch kernel (RM_UNIMIX_LOCAL=regs) form the same products in
    the same order: the mixing output and the stack built on it agree bit for bit."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    got = {}
    for mode in ("staged", "regs"):
        env = {k: v for k, v in os.environ.items() if k != "RM_UNIMIX_LOCAL"}
        if mode == "regs":
            env["RM_UNIMIX_LOCAL"] = "regs"
        path = str(tmp_path / f"local_{mode}.npz")
        r = subprocess.run([sys.executable, "-c", _LOCAL_CHILD.format(root=root, shapes=_LOCAL_SHAPES), path],
                           env=env, cwd=root, capture_output=True, text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
        got[mode] = dict(np.load(path))
    for key in got["staged"]:
        a, b = got["staged"][key], got["regs"][key]
        assert a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32)), key
