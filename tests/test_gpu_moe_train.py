"""GPU parity of the dense-training / sparse-inference Sparse-MoE PFFN forward
("RankMixer" section 3.4 Eq. 10-11; "6.4 Rankmixer: 硬件效率优化" section 6.4.4)
against the oracle: V on the training router's gates, the inference router's
gates, the per-sample regulariser and the per-expert activation."""
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


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def _model(T, D, E, Fe, B, seed, dtype, train_active=None, same_router=False):
    layers = synth.make_stack(T, D, 2, 1, seed, dtype, DEV, E=E, Fe=Fe, active=2.0)
    if same_router:
        layers[0]["Wg_train"], layers[0]["bg_train"] = layers[0]["Wg"], layers[0]["bg"]
    else:
        active = 0.75 * E if train_active is None else train_active     # most experts open under h_train
        layers[0].update(synth.make_train_router(T, D, E, seed + 1, dtype, DEV, active=active))
    m = RankMixer(T, D, 2, layers, dtype=dtype, max_batch=B, n_experts=E, expert_hidden=Fe)
    return m, layers[0]


@pytest.mark.parametrize("dtype,T,D,E,Fe,B", [("f32", 4, 16, 4, 12, 40), ("bf16", 4, 256, 8, 256, 300),
                                              ("bf16", 2, 512, 6, 128, 129)])
def test_moe_train_forward_matches_oracle(dtype, T, D, E, Fe, B):
    m, p = _model(T, D, E, Fe, B, 301 + D, dtype)
    S = synth.make_input(B, T, D, 302, dtype, DEV)
    out = m.moe_pffn_forward_train(0, S)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(p)
    ref = oracle.moe_pffn_train(_np(S), p64["Wg_train"], p64["bg_train"], p64["Wg"], p64["bg"], p64["eW1"],
                                p64["eb1"], p64["eW2"], p64["eb2"])
    # the gates decide which experts run: compare them first (float32 path tolerance for both dtypes)
    check(out["G_train"], ref["G_train"], "f32", f"moe-train {dtype} G_train", tol=1e-4 if dtype == "f32" else 5e-3)
    check(out["G_infer"], ref["G_infer"], "f32", f"moe-train {dtype} G_infer", tol=1e-4 if dtype == "f32" else 5e-3)
    check(out["V"], ref["V"], dtype, f"moe-train {dtype} V")
    check(out["lreg"], ref["lreg"], "f32", f"moe-train {dtype} lreg", tol=1e-4 if dtype == "f32" else 5e-3)
    check(out["A"], ref["A"], "f32", f"moe-train {dtype} A", tol=1e-4 if dtype == "f32" else 5e-3)
    # dense training: the training router opens more experts than the inference one
    assert (out["G_train"] > 0).float().mean() > (out["G_infer"] > 0).float().mean()


def test_moe_train_forward_with_one_router_equals_inference_forward():
    T, D, E, Fe, B = 4, 256, 8, 256, 200
    m, _ = _model(T, D, E, Fe, B, 311, "bf16", same_router=True)
    S = synth.make_input(B, T, D, 312, "bf16", DEV)
    out = m.moe_pffn_forward_train(0, S)
    V_inf, G_inf = m.moe_pffn_forward(0, S, return_gates=True)
    torch.cuda.synchronize()
    assert torch.equal(out["V"], V_inf)
    assert torch.equal(out["G_train"], G_inf)
    assert torch.allclose(out["G_infer"], G_inf, rtol=0, atol=1e-5)


def test_moe_train_forward_needs_a_training_router():
    T, D, E, Fe, B = 2, 16, 4, 8, 8
    layers = synth.make_stack(T, D, 2, 1, 321, "f32", DEV, E=E, Fe=Fe)
    m = RankMixer(T, D, 2, layers, dtype="f32", max_batch=B, n_experts=E, expert_hidden=Fe)
    S = synth.make_input(B, T, D, 322, "f32", DEV)
    with pytest.raises(_lib.RankMixerError) as e:
        m.moe_pffn_forward_train(0, S)
    assert e.value.status == _lib.RM_ERR_UNSUPPORTED
