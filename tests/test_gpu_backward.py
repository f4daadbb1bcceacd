"""GPU parity of the block backward pass against the oracle ("RankMixer 详解（1）" section 5.2).

The same seeded block input X, output gradient G and parameters go to both
sides (the oracle receives them as rounded to the library's dtype, in
float64).  Every returned gradient is compared element by element with the
bars of the forward pass: max relative error <= 1e-4 on the float32 path and
max error <= 2e-2 * RMS (of that gradient) on the bf16 path.  Shapes span
several 128 x 256 tiles with ragged batch tails; the full-width shapes of the
100M and 1B configurations run at a batch the oracle finishes in seconds, and
the benchmark batch is checked on sampled samples (dX of a sample depends on
that sample alone) and by the additivity of the parameter gradients over
sub-batches.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer
from tests.helpers import check

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAMES = {"dW1": "dW1", "db1": "db1", "dW2": "dW2", "db2": "db2",
         "dln1_g": "dln1_g", "dln1_b": "dln1_b", "dln2_g": "dln2_g", "dln2_b": "dln2_b"}


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _oracle_grads(g: dict) -> dict:
    return {"dW1": g["dW1"], "db1": g["db1"], "dW2": g["dW2"], "db2": g["db2"],
            "dln1_g": g["dln1_g"], "dln1_b": g["dln1_b"], "dln2_g": g["dln2_g"], "dln2_b": g["dln2_b"]}


def _model(T, D, k, L, B, seed, dtype, path="auto", max_batch=None):
    layers = synth.make_stack(T, D, k, L, seed, dtype, DEV)
    m = RankMixer(T, D, k, layers, dtype=dtype, max_batch=max_batch or B, gemm_path=path, training=True)
    return m, layers


def _check_all(dX, g, odX, og, dtype, tag):
    check(dX, odX, dtype, f"{tag} dX")
    for k_ in NAMES:
        check(g[k_], og[k_], dtype, f"{tag} {k_}")


@pytest.mark.parametrize("u_scale", [1.0])
def test_device_gelu_grad_matches_the_definition(u_scale):
    """Gelu and Gelu' of the backward epilogues against float64 u Phi(u) and Phi(u) + u phi(u)."""
    u = torch.cat([torch.linspace(-12, 12, 100001), torch.tensor([0.0, -0.0, 1.0, -1.0, 30.0, -30.0])]) * u_scale
    out = torch.empty(2 * u.numel(), dtype=torch.float32, device=DEV)
    ud = u.to(DEV)
    _lib.rm_debug_gelu_grad(ud.data_ptr(), out.data_ptr(), u.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    o = out.cpu().double().numpy().reshape(-1, 2)
    uu = u.double().numpy()
    ov, og = oracle.gelu(uu), oracle.gelu_grad(uu)
    # erf to 1.5e-7 (Abramowitz & Stegun 7.1.26) plus float32 rounding
    assert np.max(np.abs(o[:, 1] - og)) <= 4e-7
    assert np.max(np.abs(o[:, 0] - ov) / np.maximum(1.0, np.abs(uu))) <= 4e-7
    assert o[np.argmin(np.abs(uu)), 1] == 0.5


@pytest.mark.parametrize("dtype,path,T,D,k,B", [
    ("f32", "auto", 4, 8, 2, 64),            # the tiny float32 configuration
    ("f32", "auto", 4, 64, 2, 37),           # float32, ragged batch
    ("bf16", "simt", 4, 256, 4, 300),        # bf16 on CUDA cores
    ("bf16", "auto", 4, 256, 4, 300),        # bf16 on tcgen05: 3 row tiles (ragged), 4 / 1 column tiles
    ("bf16", "auto", 2, 512, 2, 129),        # one row past a tile, K = B not a multiple of 64
    ("bf16", "auto", 4, 256, 4, 1),          # a single sample
])
def test_block_backward_matches_oracle(dtype, path, T, D, k, B):
    m, layers = _model(T, D, k, 1, B, 11 + D + B, dtype, path)
    if path == "auto" and dtype == "bf16":
        assert m.path == "tcgen05"
    X = synth.make_input(B, T, D, 12 + D + B, dtype, DEV)
    G = synth.make_output_grad((B, T, D), 13 + D + B, device=DEV)
    dX, g = m.block_backward(0, X, G)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    odX, og = oracle.block_backward(_np(X), _np(G), synth.to_f64(layers[0]))
    _check_all(dX, g, odX, _oracle_grads(og), dtype, f"{dtype}/{path} T={T} D={D} B={B}")


def test_block_backward_small_gradients_keep_their_precision():
    """A loss gradient of scale 1e-7 (a batch-averaged loss) is carried in bf16, whose
    range covers it: the relative error is the same as at scale 1."""
    T, D, k, B = 4, 256, 4, 200
    m, layers = _model(T, D, k, 1, B, 21, "bf16")
    X = synth.make_input(B, T, D, 22, "bf16", DEV)
    G = synth.make_output_grad((B, T, D), 23, scale=1e-7, device=DEV)
    dX, g = m.block_backward(0, X, G)
    torch.cuda.synchronize()
    odX, og = oracle.block_backward(_np(X), _np(G), synth.to_f64(layers[0]))
    _check_all(dX, g, odX, _oracle_grads(og), "bf16", "G scale 1e-7")


def test_tensor_core_and_cuda_core_backward_agree():
    T, D, k, B = 4, 256, 4, 260
    layers = synth.make_stack(T, D, k, 1, 31, "bf16", DEV)
    X = synth.make_input(B, T, D, 32, "bf16", DEV)
    G = synth.make_output_grad((B, T, D), 33, device=DEV)
    out = {}
    for path in ("auto", "simt"):
        m = RankMixer(T, D, k, layers, dtype="bf16", max_batch=B, gemm_path=path, training=True)
        out[path] = m.block_backward(0, X, G)
        torch.cuda.synchronize()
        m.close()
    check(out["auto"][0], _np(out["simt"][0]), "bf16", "tc vs simt dX")
    for k_ in NAMES:
        check(out["auto"][1][k_], _np(out["simt"][1][k_]), "bf16", f"tc vs simt {k_}")


@pytest.mark.parametrize("name,B", [("rankmixer_100m", 48), ("rankmixer_1b", 12)])
def test_block_backward_full_width_shapes(name, B):
    c = synth.CONFIGS[name]
    T, D, k = c["T"], c["D"], c["k"]
    m, layers = _model(T, D, k, 1, B, 41, "bf16", max_batch=256)
    assert m.path == "tcgen05"
    X = synth.make_input(B, T, D, 42, "bf16", DEV)
    G = synth.make_output_grad((B, T, D), 43, device=DEV)
    dX, g = m.block_backward(0, X, G)
    torch.cuda.synchronize()
    odX, og = oracle.block_backward(_np(X), _np(G), synth.to_f64(layers[0]))
    _check_all(dX, g, odX, _oracle_grads(og), "bf16", f"{name} B={B}")


def test_block_backward_bench_batch_sampled_and_additive():
    """The 1B shape at B = 4096: dX of sampled samples against the oracle run on
    those samples alone, and the parameter gradients of the whole batch against
    the sums of the two halves' (each a separate call)."""
    c = synth.CONFIGS["rankmixer_1b"]
    T, D, k, B = c["T"], c["D"], c["k"], c["B"]
    m, layers = _model(T, D, k, 1, B, 51, "bf16")
    X = synth.make_input(B, T, D, 52, "bf16", DEV)
    G = synth.make_output_grad((B, T, D), 53, device=DEV)
    dX, g = m.block_backward(0, X, G)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(layers[0])
    for b in (0, 1, 2047, 4095):
        odX, _ = oracle.block_backward(_np(X[b:b + 1]), _np(G[b:b + 1]), p64)
        check(dX[b:b + 1], odX, "bf16", f"1b B=4096 dX sample {b}")
    h = B // 2
    _, g0 = m.block_backward(0, X[:h].contiguous(), G[:h].contiguous())
    _, g1 = m.block_backward(0, X[h:].contiguous(), G[h:].contiguous())
    torch.cuda.synchronize()
    for k_ in NAMES:
        check(g[k_], _np(g0[k_]) + _np(g1[k_]), "bf16", f"1b B=4096 {k_} = halves", tol=1e-3)


@pytest.mark.parametrize("dtype,T,D,k,B,L", [("f32", 4, 8, 2, 64, 2), ("bf16", 4, 256, 4, 130, 2)])
def test_stack_backward_matches_oracle(dtype, T, D, k, B, L):
    m, layers = _model(T, D, k, L, B, 61 + L, dtype)
    X0 = synth.make_input(B, T, D, 62, dtype, DEV)
    dP = synth.make_output_grad((B, D), 63, device=DEV)
    dX0, gs = m.stack_backward(X0, dP)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    odX0, ogs = oracle.stack_backward(_np(X0), _np(dP), synth.to_f64(layers))
    check(dX0, odX0, dtype, f"stack {dtype} dX0")
    for n in range(L):
        for k_ in NAMES:
            check(gs[n][k_], ogs[n][k_], dtype, f"stack {dtype} layer {n} {k_}")


def test_backward_needs_a_training_context():
    T, D, k, B = 4, 8, 2, 4
    layers = synth.make_stack(T, D, k, 1, 71, "f32", DEV)
    m = RankMixer(T, D, k, layers, dtype="f32", max_batch=B)
    X = synth.make_input(B, T, D, 72, "f32", DEV)
    G = synth.make_output_grad((B, T, D), 73, device=DEV)
    with pytest.raises(_lib.RankMixerError) as e:
        m.block_backward(0, X, G)
    assert e.value.status == _lib.RM_ERR_UNSUPPORTED
    mt = RankMixer(T, D, k, layers, dtype="f32", max_batch=B, training=True)
    with pytest.raises(_lib.RankMixerError) as e:
        mt.block_backward(0, X, G, dX=G)                    # dX_in overlapping dX_out
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError):
        mt.block_backward(0, torch.cat([X, X]), torch.cat([G, G]))   # B above max_batch


@pytest.mark.parametrize("dtype,T,D,k,B,L", [("f32", 4, 8, 2, 64, 2), ("bf16", 4, 256, 4, 130, 2),
                                             ("bf16", 16, 768, 4, 40, 2)])
def test_training_forward_pooled_matches_oracle(dtype, T, D, k, B, L):
    m, layers = _model(T, D, k, L, B, 81 + D, dtype)
    X0 = synth.make_input(B, T, D, 82, dtype, DEV)
    pooled = m.stack_forward_train(X0)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    check(pooled, oracle.stack_forward(_np(X0), synth.to_f64(layers)), dtype, f"training forward {dtype} pooled")


def test_saved_backward_equals_the_one_call_backward():
    """stack_forward_train + stack_backward_saved gives the one-call stack_backward's
    gradients bit for bit (the same kernels on the same inputs)."""
    T, D, k, B, L = 4, 256, 4, 150, 2
    m, layers = _model(T, D, k, L, B, 91, "bf16")
    X0 = synth.make_input(B, T, D, 92, "bf16", DEV)
    dP = synth.make_output_grad((B, D), 93, device=DEV)
    dX_a, g_a = m.stack_backward(X0, dP)
    m.stack_forward_train(X0)
    dX_b, g_b = m.stack_backward_saved(dP)
    torch.cuda.synchronize()
    assert torch.equal(dX_a, dX_b)
    for n in range(L):
        for k_ in NAMES:
            assert torch.equal(g_a[n][k_], g_b[n][k_]), (n, k_)


def test_saved_backward_needs_its_training_forward():
    T, D, k, B = 4, 8, 2, 8
    m, _ = _model(T, D, k, 2, B, 95, "f32")
    X0 = synth.make_input(B, T, D, 96, "f32", DEV)
    dP = synth.make_output_grad((B, D), 97, device=DEV)
    with pytest.raises(_lib.RankMixerError) as e:          # nothing saved yet
        m.stack_backward_saved(dP)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    m.stack_forward_train(X0)
    with pytest.raises(_lib.RankMixerError) as e:          # another batch size
        m.stack_backward_saved(dP[:4].contiguous())
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    m.stack_backward_saved(dP)
    torch.cuda.synchronize()
    with pytest.raises(_lib.RankMixerError) as e:          # the activations were consumed
        m.stack_backward_saved(dP)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG


def test_gradients_into_one_flat_buffer_equal_separate_buffers():
    """The benchmark's replicas write all gradients into one flat buffer (one all-reduce);
    the views get the same values as separate tensors."""
    T, D, k, B, L = 4, 256, 4, 100, 2
    m, _ = _model(T, D, k, L, B, 401, "bf16")
    X0 = synth.make_input(B, T, D, 402, "bf16", DEV)
    dP = synth.make_output_grad((B, D), 403, device=DEV)
    _, g_sep = m.stack_backward(X0, dP)
    flat = torch.full((m.flat_grad_numel(),), float("nan"), dtype=torch.float32, device=DEV)
    _, g_flat = m.stack_backward(X0, dP, grads=m.alloc_grads(flat=flat))
    torch.cuda.synchronize()
    for n in range(L):
        for k_ in NAMES:
            assert torch.equal(g_sep[n][k_], g_flat[n][k_]), (n, k_)
