"""GPU parity of the steps either side of the block stack: feature tokenization
("RankMixer" section 3.2 Eq. 2) and the prediction head ("RankMixer 详解（1）"
sections 5.1-5.2), and the end-to-end scoring call that chains tokenization,
the stack and the head, against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer, head_forward
from tests.golden_io import load_golden
from tests.helpers import check

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _tokenizer(T, d, D, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn((T, d, D), generator=g) / np.sqrt(d)).to(synth.TORCH_DTYPE[dtype]).to(DEV)
    b = (0.1 * torch.randn((T, D), generator=g)).to(synth.TORCH_DTYPE[dtype]).to(DEV)
    return W, b


def test_head_matches_oracle_and_the_worked_example():
    g = torch.Generator().manual_seed(3)
    B, D = 1000, 1536
    O = torch.randn((B, D), generator=g).to(DEV)
    w = (torch.randn(D, generator=g) / np.sqrt(D)).to(DEV)
    y = (torch.rand(B, generator=g) < 0.3).float().to(DEV)
    out = head_forward(O, w, 0.2, y, mean_loss=True)
    torch.cuda.synchronize()
    ref = oracle.head(_np(O), _np(w), 0.2, _np(y))
    check(out["p"], ref["p"], "f32", "head p")
    check(out["loss"], ref["loss"], "f32", "head loss")
    check(out["dpooled"], ref["dO"] / B, "f32", "head dpooled (batch mean)")
    # the printed worked example ("RankMixer 详解（1）" section 6.4), label 1
    wx = load_golden("worked_example_T4.txt")
    o1 = torch.tensor(wx["o"], dtype=torch.float32, device=DEV)
    w1 = torch.tensor(wx["head_w"][0], dtype=torch.float32, device=DEV)
    r1 = head_forward(o1, w1, float(wx["head_b"][0, 0]), torch.ones(1, device=DEV), mean_loss=False)
    torch.cuda.synchronize()
    assert abs(r1["p"].item() - wx["p_hat"][0, 0]) <= 1e-4
    assert abs(r1["loss"].item() - wx["loss"][0, 0]) <= 2e-4


def test_head_rejects_inconsistent_outputs():
    O = torch.zeros((4, 8), device=DEV)
    w = torch.zeros(8, device=DEV)
    with pytest.raises(_lib.RankMixerError) as e:       # a loss without labels
        _lib.rm_head_forward(O.data_ptr(), w.data_ptr(), 0.0, None, None, O.data_ptr(), None, 4, 8, True, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype,path,T,d,D,B", [
    ("bf16", "auto", 4, 128, 256, 300),      # tensor cores: 3 row tiles (ragged), K = d
    ("bf16", "auto", 32, 64, 1536, 200),     # the 1B width
    ("bf16", "simt", 4, 40, 256, 70),        # d not a multiple of 64: CUDA cores
    ("f32", "auto", 4, 6, 8, 64),            # the tiny float32 configuration
])
def test_tokenize_matches_oracle(dtype, path, T, d, D, B):
    layers = synth.make_stack(T, D, 2, 1, 7, dtype, DEV)
    m = RankMixer(T, D, 2, layers, dtype=dtype, max_batch=B, gemm_path=path)
    W, b = _tokenizer(T, d, D, 8 + d, dtype)
    m.set_tokenizer(W, b)
    E = synth.make_input(B, T, d, 9, dtype, DEV).reshape(B, T * d).contiguous()
    X0 = m.tokenize(E)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    check(X0, oracle.tokenize(_np(E), _np(W), _np(b)), dtype, f"tokenize {dtype}/{path} T={T} d={d} D={D} B={B}")


@pytest.mark.parametrize("dtype,T,d,D,k,B", [("bf16", 4, 128, 256, 2, 150), ("f32", 4, 6, 8, 2, 64)])
def test_score_end_to_end_matches_oracle(dtype, T, d, D, k, B):
    layers = synth.make_stack(T, D, k, 2, 11, dtype, DEV)
    m = RankMixer(T, D, k, layers, dtype=dtype, max_batch=B)
    W, b = _tokenizer(T, d, D, 12, dtype)
    m.set_tokenizer(W, b)
    E = synth.make_input(B, T, d, 13, dtype, DEV).reshape(B, T * d).contiguous()
    hw = (torch.randn(D, generator=torch.Generator().manual_seed(14)) / np.sqrt(D)).to(DEV)
    p = m.score(E, hw, 0.1)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    X0 = oracle.tokenize(_np(E), _np(W), _np(b))
    pooled = oracle.stack_forward(X0, synth.to_f64(layers))
    ref = oracle.head(pooled, _np(hw), 0.1)["p"]
    check(p, ref, dtype, f"score {dtype} p")


def test_score_needs_a_tokenizer():
    T, D = 4, 8
    layers = synth.make_stack(T, D, 2, 1, 15, "f32", DEV)
    m = RankMixer(T, D, 2, layers, dtype="f32", max_batch=4)
    E = torch.zeros((4, T * 6), device=DEV)
    with pytest.raises(_lib.RankMixerError) as e:
        m.score(E, torch.zeros(D, device=DEV), 0.0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype,path,T,d,D,B,gscale", [
    ("bf16", "auto", 4, 256, 256, 300, 1.0),      # tensor cores: dW (MN x MN, K = B ragged), dE (N = d)
    ("bf16", "auto", 4, 256, 256, 120, 1e-6),     # a small gradient keeps its precision (per-token scale)
    ("bf16", "auto", 32, 512, 1536, 64, 1.0),     # the 1B width with the bench's slice length
    ("bf16", "simt", 4, 40, 256, 70, 1.0),        # d not a multiple of 64
    ("f32", "auto", 4, 6, 8, 64, 1.0),
])
def test_tokenize_backward_matches_oracle(dtype, path, T, d, D, B, gscale):
    layers = synth.make_stack(T, D, 2, 1, 17, dtype, DEV)
    m = RankMixer(T, D, 2, layers, dtype=dtype, max_batch=B, gemm_path=path)
    W, b = _tokenizer(T, d, D, 18 + d, dtype)
    m.set_tokenizer(W, b)
    E = synth.make_input(B, T, d, 19, dtype, DEV).reshape(B, T * d).contiguous()
    G = synth.make_output_grad((B, T, D), 20, scale=gscale, device=DEV)
    out = m.tokenize_backward(E, G)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    dE, dW, db = oracle.tokenize_backward(_np(E), _np(W), _np(G))
    tag = f"tokenize backward {dtype}/{path} T={T} d={d} D={D} B={B} scale={gscale:g}"
    check(out["dE"], dE, dtype, tag + " dE")
    check(out["dW"], dW, dtype, tag + " dW")
    check(out["db"], db, dtype, tag + " db")
