"""GPU parity of the CUDA library against the CPU oracle (needs an sm_103a GPU).

Every test feeds the same seeded values to both sides (the oracle receives the
values as rounded to the library's dtype, in float64) and compares element by
element: bit-exact for the mixing permutation, max relative error <= 1e-4 on
the float32 path, max error <= 2e-2 * RMS on the bf16 path.  Full-size
workloads run on the GPU in the benchmark's launch configuration and are
compared on sampled samples the oracle computes one by one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer, debug_mix_residual, token_mix
from tests.helpers import assert_bf16_rounding, check

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _build(T, D, k, L, B, seed, dtype, path="auto", max_batch=None, E=0, Fe=0, moe_mask=0, active=2.0):
    layers = synth.make_stack(T, D, k, L, seed, dtype, DEV, E=E, Fe=Fe, active=active)
    m = RankMixer(T, D, k, layers, dtype=dtype, max_batch=max_batch or B, n_experts=E, expert_hidden=Fe,
                  moe_layer_mask=moe_mask, gemm_path=path)
    X = synth.make_input(B, T, D, seed + 1, dtype, DEV)
    return m, layers, X


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


# ----------------------------------------------------------------------------
# TokenMixing: bit-exact
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,T,D,H", [(3, 4, 8, 4), (5, 2, 6, 2), (7, 2, 6, 3), (2, 4, 12, 6), (2, 16, 768, 16),
                                     (3, 32, 1536, 32), (1, 5, 15, 5)])
def test_token_mix_bit_exact(dtype, B, T, D, H):
    X = synth.make_input(B, T, D, 100 + B + T + D + H, dtype, DEV)
    Y = token_mix(X, H)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(Y), oracle.token_mix(_np(X), H))


@pytest.mark.parametrize("B,T,D", [(3, 4, 256), (7, 8, 512), (5, 16, 768), (2, 32, 1536), (4, 2, 256)])
def test_fused_mixing_gather_bit_exact(B, T, D):
    """The gather inside the fused mix + LN1 kernel (the hot path's mixing), read out
    before LN1: y = Mix(X) + X.  From a bf16 layer input y is the float32 sum of two
    bf16 values, i.e. the exact sum rounded once to float32."""
    X = synth.make_input(B, T, D, 300 + T + D, "bf16", DEV)
    Y = debug_mix_residual(X)                      # [T, B, D]
    torch.cuda.synchronize()
    x = _np(X)
    want = (oracle.token_mix(x) + x).astype(np.float32)
    np.testing.assert_array_equal(Y.permute(1, 0, 2).cpu().numpy(), want)


@pytest.mark.parametrize("B,T,D", [(3, 4, 256), (5, 16, 768), (2, 32, 1536)])
def test_fused_mixing_gather_from_fp16_rows_bit_exact(B, T, D):
    """The same kernel reading a later layer's input (fp16 rows, token-major) with its LN2
    finalisation set to the identity: y is the fp16 sum of the two gathered values
    (round to nearest even of the exact sum)."""
    g = torch.Generator().manual_seed(400 + T)
    Z = (3 * torch.randn((T, B, D), generator=g)).to(torch.float16).to(DEV)
    Y = debug_mix_residual(Z, from_z=True)
    torch.cuda.synchronize()
    z = Z.permute(1, 0, 2).to("cpu", torch.float64).numpy()          # [B, T, D]
    want = (oracle.token_mix(z) + z).astype(np.float16).astype(np.float32)
    np.testing.assert_array_equal(Y.permute(1, 0, 2).cpu().numpy(), want)


@pytest.mark.parametrize("form", [0, 1])
def test_device_gelu_matches_the_definition(form):
    """The epilogue GELU (erf by Abramowitz & Stegun 7.1.26) against u * Phi(u) in float64:
    form 0 is the scalar form of the CUDA-core GEMMs, form 1 the packed form of the
    tensor-core epilogues."""
    from scipy.special import ndtr
    u = torch.cat([torch.linspace(-12, 12, 200001), torch.tensor([0.0, -0.0, 1.0, -1.0, 30.0, -30.0, 1e-8, -1e-8])])
    out = torch.empty_like(u, device=DEV)
    ud = u.to(DEV)
    _lib.rm_debug_gelu(ud.data_ptr(), out.data_ptr(), u.numel(), form, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    x = u.double().numpy()
    ref = x * ndtr(x)
    g = out.cpu().double().numpy()
    err = np.abs(g - ref) / np.maximum(1.0, np.abs(x))
    assert err.max() <= 4e-7, f"max scaled error {err.max():.3e}"


# ----------------------------------------------------------------------------
# Tiny float32 configuration (T=4, D=8, H=4: the A1..D4 layout), 1e-4
# ----------------------------------------------------------------------------

def test_tiny_fp32_block_and_stack():
    c = synth.CONFIGS["tiny_fp32"]
    m, layers, X = _build(c["T"], c["D"], c["k"], c["L"], c["B"], 7, "f32")
    assert m.path == "simt"
    Xo, S = m.block_forward(0, X, return_S=True)
    pooled, XL = m.stack_forward(X, return_XL=True)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(layers)
    Xo_ref, S_ref = oracle.block_forward(_np(X), p64[0], return_S=True)
    pooled_ref, XL_ref = oracle.stack_forward(_np(X), p64, return_XL=True)
    check(S, S_ref, "f32", "S (LN1)")
    check(Xo, Xo_ref, "f32", "block X_out")
    check(XL, XL_ref, "f32", "stack X_L")
    check(pooled, pooled_ref, "f32", "pooled")


# ----------------------------------------------------------------------------
# bf16 shapes that span several tiles and a ragged batch tail, both GEMM paths
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("path", ["tcgen05", "simt"])
@pytest.mark.parametrize("T,D,k,L,B", [(4, 256, 2, 2, 300), (8, 512, 4, 1, 260), (2, 64, 1, 1, 129),
                                       (2, 192, 2, 1, 300),    # pair tiles with BN = 128 (GEMM1) and 64 (GEMM2)
                                       (16, 768, 4, 1, 77)])
def test_bf16_block_and_stack(path, T, D, k, L, B):
    m, layers, X = _build(T, D, k, L, B, 11 + T + D, "bf16", path=path)
    assert m.path == path
    Xo32, S32 = m.block_forward(0, X, return_S=True, out_dtype="f32")
    Xo, S = m.block_forward(0, X, return_S=True)
    pooled32, XL32 = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    pooled, XL = m.stack_forward(X, return_XL=True)
    pooled_only = m.stack_forward(X)          # the pool without X_L takes its own (fp16-pair) path
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(layers)
    Xo_ref, S_ref = oracle.block_forward(_np(X), p64[0], return_S=True)
    check(S32, S_ref, "bf16", "S (LN1)")
    check(Xo32, Xo_ref, "bf16", "block X_out")
    assert_bf16_rounding(S, S32, "S")
    assert_bf16_rounding(Xo, Xo32, "block X_out")
    pooled_ref, XL_ref = oracle.stack_forward(_np(X), p64, return_XL=True)
    check(XL32, XL_ref, "bf16", "stack X_L")
    assert_bf16_rounding(XL, XL32, "stack X_L")
    assert torch.equal(pooled, pooled32)      # the X_L dtype does not change the pooled output
    check(pooled, pooled_ref, "bf16", "pooled")
    check(pooled_only, pooled_ref, "bf16", "pooled (without X_L)")


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_stack_matches_chained_blocks(path):
    """Chaining rm_block_forward feeds each block its input rounded to bf16, the stack
    keeps X_n on the device in fp16: the two are different computations, so each is
    held to the oracle on its own inputs -- every chained block against the oracle's
    block on the bf16 input it actually received, the stack against the oracle's
    stack -- and the pooled output must be the token mean of X_L."""
    T, D, k, L, B = 4, 256, 2, 3, 200
    m, layers, X = _build(T, D, k, L, B, 5, "bf16", path=path)
    p64 = synth.to_f64(layers)
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    Xn = X
    for n in range(L):
        out32 = m.block_forward(n, Xn, out_dtype="f32")
        out = m.block_forward(n, Xn)
        torch.cuda.synchronize()
        check(out32, oracle.block_forward(_np(Xn), p64[n]), "bf16", f"chained block {n}")
        assert_bf16_rounding(out, out32, f"chained block {n}")
        Xn = out
    torch.testing.assert_close(pooled, XL.mean(dim=1), rtol=0, atol=2e-3)
    pr, xr = oracle.stack_forward(_np(X), p64, return_XL=True)
    check(XL, xr, "bf16", "stack X_L (L=3)")
    check(pooled, pr, "bf16", "pooled (L=3)")


def test_tcgen05_agrees_with_simt():
    T, D, k, B = 8, 512, 4, 333
    layers = synth.make_stack(T, D, k, 1, 9, "bf16", DEV)
    X = synth.make_input(B, T, D, 10, "bf16", DEV)
    a = RankMixer(T, D, k, layers, max_batch=B, gemm_path="tcgen05").block_forward(0, X, out_dtype="f32")
    b = RankMixer(T, D, k, layers, max_batch=B, gemm_path="simt").block_forward(0, X, out_dtype="f32")
    torch.cuda.synchronize()
    check(a, _np(b), "bf16", "tcgen05 vs simt", tol=1e-2)


def test_deterministic_reruns():
    T, D, k, L, B = 8, 512, 4, 2, 300
    m, _, X = _build(T, D, k, L, B, 21, "bf16")
    p1, x1 = m.stack_forward(X, return_XL=True)
    p2, x2 = m.stack_forward(X, return_XL=True)
    torch.cuda.synchronize()
    assert torch.equal(p1, p2) and torch.equal(x1, x2)


@pytest.mark.parametrize("B", [300, 40])      # the CTA-pair and the weights-as-M layer kernels eagerly
def test_graph_captured_stack_replays_the_eager_result(B):
    """The stack forward captured into a CUDA graph (after one eager call has made the
    lazy allocations) replays the eager result bit for bit: under capture each layer's FFN
    runs as two launches, which give the fused launch's bits."""
    T, D, k, L = 8, 512, 2, 2
    m, _, X = _build(T, D, k, L, B, 25, "bf16")
    ref = m.stack_forward(X).clone()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.stack_forward(X)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res = m.stack_forward(X)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(res, ref)
    assert m.sync_status() == _lib.RM_OK
    assert torch.equal(m.stack_forward(X), ref)   # eager again after the captures


@pytest.mark.parametrize("B", [100, 2500])      # one shot; three pipelined chunks (512, 1024, 964)
def test_host_entry_matches_device_entry(B):
    """The host entry runs large batches as chunks.  Every sample's arithmetic is the same
    whatever the batch (the tile shapes and k-loops do not depend on it), so the chunked
    call equals the device call bit for bit; both are also held to the oracle."""
    T, D, k, L = 8, 512, 4, 2
    m, layers, X = _build(T, D, k, L, B, 23, "bf16")
    dev = m.stack_forward(X)
    Xh = X.cpu().pin_memory()
    host = m.stack_forward_host(Xh)
    host2 = m.stack_forward_host(Xh)          # a second call reuses the staging buffers
    torch.cuda.synchronize()
    assert torch.equal(host, host2) and torch.equal(dev.cpu(), host)
    rng = np.random.default_rng(B)
    idx = np.unique(np.concatenate([[0, B - 1], rng.choice(B, size=min(24, B), replace=False)]))
    ref = oracle.stack_forward(_np(X[idx]), synth.to_f64(layers))
    check(host[idx], ref, "bf16", f"host entry B={B}")
    check(dev.cpu()[idx], ref, "bf16", f"device entry B={B}")


# ----------------------------------------------------------------------------
# Edge cases
# ----------------------------------------------------------------------------

def test_batch_of_one_and_full_capacity():
    T, D, k, L = 4, 256, 2, 2
    m, layers, X = _build(T, D, k, L, 257, 31, "bf16", max_batch=257)
    p64 = synth.to_f64(layers)
    for B in (1, 257):
        pooled, XL = m.stack_forward(X[:B].contiguous(), return_XL=True, xl_dtype="f32")
        torch.cuda.synchronize()
        pr, xr = oracle.stack_forward(_np(X[:B]), p64, return_XL=True)
        check(XL, xr, "bf16", f"X_L B={B}")
        check(pooled, pr, "bf16", f"pooled B={B}")


@pytest.mark.parametrize("dtype,T,D,k", [("bf16", 4, 12, 2), ("f32", 4, 12, 3), ("bf16", 6, 96, 2),
                                         ("f32", 3, 48, 1), ("bf16", 32, 32, 1)])
def test_odd_shapes_take_the_simt_path(dtype, T, D, k):
    """q odd, D not a multiple of 64, q = 1 (plain transpose): CUDA-core GEMMs."""
    B = 37
    m, layers, X = _build(T, D, k, 2, B, 41 + D, dtype)
    assert m.path == "simt"
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    torch.cuda.synchronize()
    pr, xr = oracle.stack_forward(_np(X), synth.to_f64(layers), return_XL=True)
    check(XL, xr, dtype, "X_L")
    check(pooled, pr, dtype, "pooled")
    if dtype == "bf16":
        _, XLb = m.stack_forward(X, return_XL=True)
        assert_bf16_rounding(XLb, XL, "X_L")


def test_invalid_arguments_are_reported():
    T, D, k = 4, 256, 2
    m, layers, X = _build(T, D, k, 1, 16, 3, "bf16")
    with pytest.raises(_lib.RankMixerError) as e:
        m.block_forward(1, X)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:
        m.stack_forward(synth.make_input(17, T, D, 1, "bf16", DEV))
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:
        _lib.rm_block_forward(m.ctx, 0, X.data_ptr(), X.data_ptr(), None, _lib.RM_BF16, 16, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:
        _lib.rm_stack_forward(m.ctx, X.data_ptr() + 2, m.stack_forward(X).data_ptr(), None, _lib.RM_BF16, 16, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    Y = torch.empty_like(X)
    with pytest.raises(_lib.RankMixerError) as e:          # unknown output dtype
        _lib.rm_block_forward(m.ctx, 0, X.data_ptr(), Y.data_ptr(), None, 7, 16, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    with pytest.raises(_lib.RankMixerError) as e:
        RankMixer(T, D, k, layers, gemm_path="tcgen05", dtype="f32")
    assert e.value.status in (_lib.RM_ERR_UNSUPPORTED, _lib.RM_ERR_INVALID_ARG)
    with pytest.raises(_lib.RankMixerError) as e:
        m.moe_pffn_forward(0, X)
    assert e.value.status == _lib.RM_ERR_UNSUPPORTED
    # the context stays usable
    m.stack_forward(X)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK


def test_bounded_wait_reports_timeout_and_context_survives():
    T, D, k = 4, 256, 2
    m, layers, X = _build(T, D, k, 1, 16, 3, "bf16")
    m.debug_wait_timeout(2000)
    assert m.sync_status() == _lib.RM_ERR_TIMEOUT
    assert m.sync_status() == _lib.RM_OK      # cleared
    out = m.block_forward(0, X, out_dtype="f32")
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    check(out, oracle.block_forward(_np(X), synth.to_f64(layers)[0]), "bf16", "block after timeout")


def test_profiler_counts_launches():
    T, D, k, L, B = 4, 256, 2, 2, 64
    m, _, X = _build(T, D, k, L, B, 3, "bf16")
    m.profile(True)
    m.stack_forward(X)
    st = m.profile_read()
    m.profile(False)
    # both FFN GEMMs of a layer run as one fused launch ("pffn") or as two
    assert st["mix_ln1"][0] == L and st["pool"][0] == 1
    assert st["gemm1"][0] + st["pffn"][0] == L and st["gemm2"][0] + st["pffn"][0] == L
    assert all(ms >= 0 for _, ms in st.values())


# ----------------------------------------------------------------------------
# Full-size workloads, sampled parity
# ----------------------------------------------------------------------------

def _sampled_stack_parity(name, B, n_samples, seed, max_batch=None, model=None):
    c = synth.CONFIGS[name]
    T, D, k, L = c["T"], c["D"], c["k"], c["L"]
    if model is None:
        m, layers, _ = _build(T, D, k, L, 1, seed, "bf16", max_batch=max_batch or B)
        p64 = synth.to_f64(layers)
    else:
        m, layers, p64 = model
    X = synth.make_input(B, T, D, seed + B, "bf16", DEV)
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    _, XLb = m.stack_forward(X, return_XL=True)
    pooled_only = m.stack_forward(X)          # the serving call: no X_L
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    assert_bf16_rounding(XLb, XL, f"{name} B={B} X_L")
    del XLb
    rng = np.random.default_rng(seed + B)
    idx = np.unique(np.concatenate([[0, B - 1], rng.choice(B, size=min(n_samples, B), replace=False)]))
    pr, xr = oracle.stack_forward(_np(X[idx]), p64, return_XL=True)
    check(XL[torch.as_tensor(idx, device=XL.device)], xr, "bf16", f"{name} B={B} X_L")
    check(pooled[torch.as_tensor(idx, device=pooled.device)], pr, "bf16", f"{name} B={B} pooled")
    check(pooled_only[torch.as_tensor(idx, device=pooled.device)], pr, "bf16", f"{name} B={B} pooled (without X_L)")
    assert torch.isfinite(pooled).all() and torch.isfinite(pooled_only).all()
    return m


def test_rankmixer_100m_full_size_sampled():
    _sampled_stack_parity("rankmixer_100m", 2048, 24, 1000)


@pytest.fixture(scope="module")
def model_1b():
    c = synth.CONFIGS["rankmixer_1b"]
    layers = synth.make_stack(c["T"], c["D"], c["k"], c["L"], 2000, "bf16", DEV)
    m = RankMixer(c["T"], c["D"], c["k"], layers, max_batch=8192)
    assert m.path == "tcgen05"
    p64 = synth.to_f64(layers)
    yield m, layers, p64
    m.close()


def test_rankmixer_1b_full_size_sampled(model_1b):
    _sampled_stack_parity("rankmixer_1b", 4096, 8, 2000, model=model_1b)


@pytest.mark.parametrize("B", [1, 8, 64, 256, 1024, 8192])
def test_rankmixer_1b_serving_sweep_sampled(model_1b, B):
    _sampled_stack_parity("rankmixer_1b", B, 3, 2000, model=model_1b)


# ----------------------------------------------------------------------------
# Sparse-MoE PFFN
# ----------------------------------------------------------------------------

def _moe_oracle(S64, p64, t_slice=None):
    return oracle.moe_pffn(S64, p64["Wg"], p64["bg"], p64["eW1"], p64["eb1"], p64["eW2"], p64["eb2"],
                           return_gates=True)


@pytest.mark.parametrize("dtype,path,T,D,E,Fe,B", [("bf16", "auto", 4, 256, 4, 256, 300),
                                                   ("bf16", "simt", 4, 256, 4, 256, 300),
                                                   ("bf16", "auto", 2, 128, 8, 384, 129),
                                                   ("f32", "auto", 3, 18, 4, 24, 50)])
def test_moe_pffn_small(dtype, path, T, D, E, Fe, B):
    m, layers, _ = _build(T, D, 2, 1, B, 61 + D, dtype, path=path, E=E, Fe=Fe, active=E / 4)
    S = synth.make_input(B, T, D, 62, dtype, DEV)
    V, G = m.moe_pffn_forward(0, S, return_gates=True)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(layers[0])
    V_ref, G_ref = _moe_oracle(_np(S), p64)
    assert 0.1 < (G_ref > 0).mean() < 0.5, "router bias should open about a quarter of the experts"
    np.testing.assert_allclose(_np(G), G_ref, atol=2e-4 if dtype == "bf16" else 1e-5, rtol=1e-3)
    check(V, V_ref, dtype, "MoE V")


@pytest.mark.parametrize("dtype,T,D,E,Fe,B", [("bf16", 2, 256, 4, 256, 600),    # CTA-pair expert tiles (B >= 512)
                                               ("bf16", 2, 128, 12, 128, 131),    # two 8-expert router slices
                                               ("bf16", 4, 36, 4, 64, 37),       # rows not in 16-byte chunks
                                               ("f32", 2, 8, 9, 16, 50)])        # fp32, E > 8, B % 4 != 0
def test_moe_router_shapes_and_determinism(dtype, T, D, E, Fe, B):
    m, layers, _ = _build(T, D, 2, 1, B, 90 + D + E, dtype, E=E, Fe=Fe, active=E / 4)
    S = synth.make_input(B, T, D, 91, dtype, DEV)
    V1 = torch.full(S.shape, float("nan"), dtype=torch.float32, device=DEV)   # every row must be written
    V1, G = m.moe_pffn_forward(0, S, V1, return_gates=True)
    V2 = torch.full(S.shape, float("nan"), dtype=torch.float32, device=DEV)
    V2 = m.moe_pffn_forward(0, S, V2)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    p64 = synth.to_f64(layers[0])
    V_ref, G_ref = _moe_oracle(_np(S), p64)
    np.testing.assert_allclose(_np(G), G_ref, atol=2e-4 if dtype == "bf16" else 1e-5, rtol=1e-3)
    check(V1, V_ref, dtype, f"MoE V (E={E}, D={D})")
    # rows inside an expert group may be ordered differently from run to run; the values may not
    assert torch.equal(V1, V2), "MoE PFFN is not deterministic"
    closed = (G_ref > 0).sum(-1) == 0
    assert closed.any(), "the case should have (sample, token) pairs with every expert closed"
    assert (V1[torch.from_numpy(closed).to(DEV)] == 0).all()


def test_moe_all_experts_closed_gives_exact_zero():
    T, D, E, Fe, B = 4, 256, 4, 256, 70
    layers = synth.make_stack(T, D, 2, 1, 93, "bf16", DEV, E=E, Fe=Fe)
    layers[0]["bg"] = torch.full_like(layers[0]["bg"], -1e3)     # ReLU closes every gate
    m = RankMixer(T, D, 2, layers, max_batch=B, n_experts=E, expert_hidden=Fe)
    S = synth.make_input(B, T, D, 94, "bf16", DEV)
    V = torch.full(S.shape, float("nan"), dtype=torch.float32, device=DEV)
    V, G = m.moe_pffn_forward(0, S, V, return_gates=True)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    assert (G == 0).all() and (V == 0).all()


def test_moe_layer_inside_block():
    T, D, E, Fe, B = 4, 256, 4, 256, 200
    m, layers, X = _build(T, D, 2, 2, B, 71, "bf16", E=E, Fe=Fe, moe_mask=0b10, active=1.0)
    p64 = synth.to_f64(layers)
    X1 = m.block_forward(0, X)                        # dense layer, bf16 output (the next block's input)
    X1f = m.block_forward(0, X, out_dtype="f32")
    X2, S2 = m.block_forward(1, X1, return_S=True, out_dtype="f32")   # MoE layer, from the bf16 X1
    X2b = m.block_forward(1, X1)
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")   # both layers, X1 kept on the device
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    assert_bf16_rounding(X1, X1f, "dense layer")
    assert_bf16_rounding(X2b, X2, "MoE layer X_out")

    def moe_block(x, p):
        S = oracle.layernorm(oracle.token_mix(x) + x, p["ln1_g"], p["ln1_b"], 1e-5)
        V = oracle.moe_pffn(S, p["Wg"], p["bg"], p["eW1"], p["eb1"], p["eW2"], p["eb2"])
        return oracle.layernorm(V + S, p["ln2_g"], p["ln2_b"], 1e-5), S

    X1_ref = oracle.block_forward(_np(X), p64[0])
    check(X1f, X1_ref, "bf16", "dense layer")
    X2_ref, S2_ref = moe_block(_np(X1), p64[1])
    check(S2, S2_ref, "bf16", "MoE layer S")
    check(X2, X2_ref, "bf16", "MoE layer X_out")
    XL_ref, _ = moe_block(X1_ref, p64[1])
    check(XL, XL_ref, "bf16", "stack with a MoE layer, X_L")
    check(pooled, XL_ref.mean(axis=1), "bf16", "stack with a MoE layer, pooled")


def test_moe_1b_full_size_sampled():
    c = synth.CONFIGS["moe_1b"]
    T, D, E, Fe, B = c["T"], c["D"], c["E"], c["Fe"], c["B"]
    p = synth.make_experts(T, D, E, Fe, 3000, "bf16", DEV, active=c["active"])
    dense = synth.make_layer(T, D, c["k"], 3001, "bf16", DEV)
    dense.update(p)
    m = RankMixer(T, D, c["k"], [dense], max_batch=B, n_experts=E, expert_hidden=Fe)
    S = synth.make_input(B, T, D, 3002, "bf16", DEV)
    V, G = m.moe_pffn_forward(0, S, return_gates=True)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    active = (G > 0).float().sum(-1).mean().item()
    assert 1.7 < active < 2.3, f"mean active experts {active}"
    rng = np.random.default_rng(5)
    pairs = [(int(rng.integers(B)), int(rng.integers(T))) for _ in range(6)] + [(0, 0), (B - 1, T - 1)]
    for b, t in pairs:
        pt = {k: _np(v[t:t + 1]) for k, v in p.items()}
        V_ref, G_ref = oracle.moe_pffn(_np(S[b:b + 1, t:t + 1]), pt["Wg"], pt["bg"], pt["eW1"], pt["eb1"],
                                       pt["eW2"], pt["eb2"], return_gates=True)
        np.testing.assert_allclose(_np(G[b:b + 1, t:t + 1]), G_ref, atol=2e-4, rtol=1e-3)
        check(V[b:b + 1, t:t + 1], V_ref, "bf16", f"MoE V (b={b}, t={t})")


# ----------------------------------------------------------------------------
# Every tile dispatch of the dense GEMMs (RM_GEMM_PAIR is read once per process)
# ----------------------------------------------------------------------------

_DISPATCH_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
import oracle
from rankmixer_feature_interaction_gb300 import synth
from rankmixer_feature_interaction_gb300.api import RankMixer
from tests.helpers import check
for T, D, k, L, B in {shapes}:
    layers = synth.make_stack(T, D, k, L, 123, "bf16", "cuda")
    m = RankMixer(T, D, k, layers, max_batch=B, gemm_path="tcgen05")
    X = synth.make_input(B, T, D, 124, "bf16", "cuda")
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    p64 = synth.to_f64(layers)
    ref_pool, ref_XL = oracle.stack_forward(X.cpu().double().numpy(), p64, return_XL=True)
    check(XL, ref_XL, "bf16", f"X_L {{(T, D, k, L, B)}}")
    check(pooled, ref_pool, "bf16", f"pooled {{(T, D, k, L, B)}}")
    m.close()
print("ok")
"""

# shapes that reach every tile form: CTA pairs with BN 256 / 128 (GEMM1) and 64 (GEMM2), one-CTA
# tiles (129..255 rows), the weights-as-M path (1..64 rows, and up to 256 when widened)
_DISPATCH_SHAPES = [(4, 256, 2, 2, 300), (2, 192, 2, 1, 300), (8, 512, 2, 2, 1100), (4, 256, 2, 2, 13),
                    (4, 256, 2, 2, 40), (4, 512, 2, 1, 150), (32, 768, 1, 1, 20)]
_TUNING_KEYS = ("RM_GEMM_PAIR", "RM_GEMM_KSUB", "RM_GEMM1_EPW", "RM_GEMM2_BN", "RM_GEMM_SMALL_BN", "RM_GEMM_SWAP_MAX",
                "RM_PDL", "RM_NVTX", "RM_GEMM_FUSED", "RM_HID_HINT")


@pytest.mark.parametrize("tuning", [{},                                            # the defaults
                                    {"RM_GEMM_PAIR": "0"},                          # one CTA per tile
                                    {"RM_GEMM2_BN": "128"},                         # narrower second-GEMM tiles
                                    {"RM_GEMM_SMALL_BN": "128"},                    # narrower one-CTA tiles
                                    {"RM_GEMM_SWAP_MAX": "0"},                      # no weights-as-M path
                                    {"RM_GEMM_SWAP_MAX": "256"},                    # weights-as-M up to 256 rows
                                    {"RM_GEMM_FUSED": "0"},                         # the two FFN GEMMs apart
                                    {"RM_PDL": "0"},                                # plain stream order
                                    {"RM_NVTX": "1"},                               # NVTX ranges around launches
                                    {"RM_GEMM_PAIR": "2"},                          # pairs for GEMM2 only
                                    {"RM_GEMM_KSUB": "1"},                          # one k-block per stage
                                    {"RM_GEMM1_EPW": "16"},                         # 16 GELU epilogue warps
                                    {"RM_GEMM1_EPW": "8", "RM_GEMM_KSUB": "2"},     # 8 warps at short K
                                    {"RM_GEMM1_EPW": "16", "RM_GEMM_KSUB": "1"},
                                    {"RM_HID_HINT": "1"}])                          # evict-first hidden-row stores
def test_every_gemm_tile_dispatch(tuning):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in _TUNING_KEYS}
    env.update(tuning)
    r = subprocess.run([sys.executable, "-c", _DISPATCH_CHILD.format(root=root, shapes=_DISPATCH_SHAPES)], env=env,
                       cwd=root, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


def test_pipelined_host_entry():
    """Batches enqueued back to back through the pipelined host entry (copy of batch n + 1
    while batch n computes, two in flight) give each batch the device call's result, bit
    for bit; tickets can be waited for late, twice, or not at all before their slot is
    reused."""
    T, D, k, L, B = 8, 512, 4, 2, 300
    m, layers, _ = _build(T, D, k, L, B, 29, "bf16")
    Xs = [synth.make_input(B, T, D, 300 + i, "bf16", DEV) for i in range(5)]
    want = [m.stack_forward(X).cpu() for X in Xs]
    Xh = [X.cpu().pin_memory() for X in Xs]
    outs = [torch.empty((B, D), dtype=torch.float32).pin_memory() for _ in Xs]
    tickets = []
    for i in range(len(Xs)):
        tickets.append(m.stack_forward_host_async(Xh[i], outs[i]))
        if i >= 1:
            m.host_wait(tickets[i - 1])
            assert torch.equal(outs[i - 1], want[i - 1]), f"batch {i - 1}"
    m.host_wait(tickets[-1])
    m.host_wait(tickets[-1])                  # twice: returns at once
    m.host_wait(tickets[0])                   # long since waited for
    assert torch.equal(outs[-1], want[-1])
    t = m.stack_forward_host_async(Xh[0], outs[0])     # a new batch into a reused slot, never waited
    t2 = m.stack_forward_host_async(Xh[1], outs[1])
    m.host_wait(t2)
    m.host_wait(t)
    assert torch.equal(outs[0], want[0]) and torch.equal(outs[1], want[1])
    with pytest.raises(_lib.RankMixerError) as e:
        m.host_wait(t2 + 5)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    assert m.sync_status() == _lib.RM_OK



# ----------------------------------------------------------------------------
# Both FFN GEMMs of a layer in one launch (B >= 256 on the tensor-core path) run
# the per-tile arithmetic of the two separate launches: every output bit agrees
# ----------------------------------------------------------------------------

_FUSED_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer
out = {{}}
for T, D, k, L, B, Bcap in {shapes}:
    layers = synth.make_stack(T, D, k, L, 411, "bf16", "cuda")
    m = RankMixer(T, D, k, layers, max_batch=Bcap)
    m.profile(True)
    X = synth.make_input(B, T, D, 412, "bf16", "cuda")
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    Xo, S = m.block_forward(0, X, return_S=True, out_dtype="f32")
    # a smaller batch on the same context, then the full one again (the counters of the
    # row blocks past a batch keep pace)
    Xs = X[: max(256, B // 2)].contiguous()
    ps_, XLs = m.stack_forward(Xs, return_XL=True, xl_dtype="f32")
    pooled2 = m.stack_forward(X)
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    prof = m.profile_read()
    key = f"{{T}}_{{D}}_{{B}}"
    out["XL_" + key] = XL.cpu().numpy()
    out["pooled_" + key] = pooled.float().cpu().numpy()
    out["Xo_" + key] = Xo.cpu().numpy()
    out["S_" + key] = S.float().cpu().numpy()
    out["XLs_" + key] = XLs.cpu().numpy()
    out["pooled2_" + key] = pooled2.float().cpu().numpy()
    print(key, "pffn launches", prof["pffn"][0], "gemm1 launches", prof["gemm1"][0])
    m.close()
# one context through batches that alternate between the CTA-pair and the weights-as-M
# layer kernels (the two share the dependency counters and their epochs)
layers = synth.make_stack(8, 512, 2, 2, 413, "bf16", "cuda")
m = RankMixer(8, 512, 2, layers, max_batch=600)
X = synth.make_input(600, 8, 512, 414, "bf16", "cuda")
for i, B in enumerate((600, 40, 300, 20, 64, 600)):
    out[f"seq_{{i}}_{{B}}"] = m.stack_forward(X[:B].contiguous()).float().cpu().numpy()
torch.cuda.synchronize()
assert m.sync_status() == 0
m.close()
np.savez(sys.argv[1], **out)
print("ok")
"""

# (T, D, k, L, B, max_batch): ragged row blocks, a context larger than the batch, both model widths
_FUSED_SHAPES = [(4, 256, 2, 3, 300, 300), (8, 512, 2, 2, 1100, 1500), (16, 768, 4, 2, 512, 512),
                 (32, 1536, 1, 2, 300, 600),
                 # weights as M (17 <= B <= 64): ragged batches, a context larger than the batch
                 (8, 512, 2, 2, 37, 64), (16, 768, 4, 2, 17, 300), (32, 1536, 4, 2, 64, 64), (4, 256, 2, 3, 20, 600)]


def test_fused_layer_gemm_bit_identical_to_two_launches(tmp_path):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    got, logs = {}, {}
    for mode in ("1", "0"):
        env = {k: v for k, v in os.environ.items() if k not in _TUNING_KEYS}
        env["RM_GEMM_FUSED"] = mode
        path = str(tmp_path / f"fused_{mode}.npz")
        r = subprocess.run([sys.executable, "-c", _FUSED_CHILD.format(root=root, shapes=_FUSED_SHAPES), path],
                           env=env, cwd=root, capture_output=True, text=True, timeout=900)
        assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
        got[mode] = dict(np.load(path))
        logs[mode] = r.stdout
    # the fused launch ran when enabled, and only the separate GEMMs when not
    assert "pffn launches 0" not in logs["1"] and "gemm1 launches 0" in logs["1"], logs["1"]
    assert "pffn launches 0" in logs["0"], logs["0"]
    for key in got["1"]:
        a, b = got["1"][key], got["0"][key]
        assert a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32)), key
