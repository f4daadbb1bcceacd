"""Device allocation failures, injected on the host (no GPU fault is involved).

Every device allocation of the library goes through one allocator whose next
allocation can be made to fail (rm_debug_fail_alloc, or RM_FAULT_INJECT=alloc:N).
For context creation and for every call that allocates a workspace on first
use, each allocation in turn is made to fail: the call must return
RM_ERR_OOM, release what it took (rm_debug_alloc_stats counts the live
allocations), and leave the context usable -- the same call then succeeds
and computes the same result as on a context that never saw a failure.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer

pytestmark = pytest.mark.gpu

DEV = "cuda"
T, D, k, L, B, E, Fe = 4, 256, 2, 2, 64, 4, 256


def _live():
    return _lib.rm_debug_alloc_stats()[1:]


def _allocations(fn) -> int:
    made0 = _lib.rm_debug_alloc_stats()[0]
    fn()
    torch.cuda.synchronize()
    return _lib.rm_debug_alloc_stats()[0] - made0


def _expect_oom(fn, what):
    with pytest.raises(_lib.RankMixerError) as e:
        fn()
    assert e.value.status == _lib.RM_ERR_OOM, f"{what}: {e.value}"
    assert "injected failure" in str(e.value), what


@pytest.fixture(autouse=True)
def _disarm():
    yield
    _lib.rm_debug_fail_alloc(-1)


def _layers(seed=5):
    return synth.make_stack(T, D, k, L, seed, "bf16", DEV, E=E, Fe=Fe)


def _create(layers, **kw):
    return RankMixer(T, D, k, layers, max_batch=B, n_experts=E, expert_hidden=Fe, **kw)


def test_create_unwinds_every_allocation_failure():
    layers = _layers()
    kw = dict(moe_layer_mask=0b10, training=True)
    _create(layers, **kw).close()                 # loads the kernels once
    live0 = _live()
    n = _allocations(lambda: _create(layers, **kw).close())
    assert n >= 20, n
    assert _live() == live0
    for i in range(n):
        _lib.rm_debug_fail_alloc(i)
        _expect_oom(lambda: _create(layers, **kw), f"rm_create, allocation {i}")
        assert _live() == live0, f"rm_create leaked after a failure at allocation {i}"
    _lib.rm_debug_fail_alloc(-1)
    m = _create(layers, **kw)
    X = synth.make_input(B, T, D, 6, "bf16", DEV)
    m.stack_forward(X)
    torch.cuda.synchronize()
    assert m.sync_status() == _lib.RM_OK
    m.close()
    assert _live() == live0


def test_environment_variable_arms_the_injection():
    """RM_FAULT_INJECT=alloc:N is read at the library's first allocation of a process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    child = (
        "import sys; sys.path.insert(0, %r)\n"
        "from rankmixer_feature_interaction_gb300 import _lib, synth\n"
        "from rankmixer_feature_interaction_gb300.api import RankMixer\n"
        "layers = synth.make_stack(4, 256, 2, 1, 5, 'bf16', 'cuda')\n"
        "try:\n"
        "    RankMixer(4, 256, 2, layers, max_batch=8)\n"
        "    print('created')\n"
        "except _lib.RankMixerError as e:\n"
        "    print('status', e.status, 'injected' in str(e))\n"
        "RankMixer(4, 256, 2, layers, max_batch=8).close()\n"
        "print('second ok')\n" % root)
    env = dict(os.environ, RM_FAULT_INJECT="alloc:3")
    r = subprocess.run([sys.executable, "-c", child], env=env, cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert f"status {_lib.RM_ERR_OOM} True" in r.stdout and "second ok" in r.stdout, r.stdout


def _lazy_calls(layers):
    """(name, context kwargs, setup(m), call(m) -> result tensors) for each call that
    allocates a workspace on first use."""
    X = synth.make_input(B, T, D, 7, "bf16", DEV)
    G = synth.make_output_grad((B, T, D), 8, device=DEV)
    dP = synth.make_output_grad((B, D), 9, device=DEV)
    d = 64
    g = torch.Generator(device=DEV).manual_seed(10)
    Wt = (torch.randn((T, d, D), generator=g, device=DEV) / d ** 0.5).to(torch.bfloat16)
    bt = (0.1 * torch.randn((T, D), generator=g, device=DEV)).to(torch.bfloat16)
    Em = torch.randn((B, T * d), generator=g, device=DEV).to(torch.bfloat16)
    hw = torch.randn(D, generator=g, device=DEV) / D ** 0.5
    WG, WB = synth.make_unimix_weights(T, D, D // T, 11, DEV)
    tr = synth.make_train_router(T, D, E, 12, "bf16", DEV, active=3.0)
    layers_t = [dict(p) for p in layers]
    layers_t[0].update(tr)

    def block_backward(m):
        dX, gr = m.block_backward(0, X, G)
        return [dX, gr["dW1"], gr["dW2"]]

    def stack_backward(m):
        dX0, grs = m.stack_backward(X, dP)
        return [dX0, grs[0]["dW1"], grs[1]["dW2"]]

    def host_entry(m):
        return [m.stack_forward_host(X.cpu().pin_memory())]

    def score(m):
        return [m.score(Em, hw, 0.1)]

    def tokenize_backward(m):
        out = m.tokenize_backward(Em, G)
        return [out["dE"], out["dW"], out["db"]]

    def set_unimixing(m):
        m.set_unimixing(0, WG, WB, tau=0.5, iters=5)
        return [m.stack_forward(X)]

    def moe_train(m):
        # without a gates_infer buffer the call keeps the inference-router gates in a
        # context-owned buffer, allocated at the first such call
        V = torch.empty((B, T, D), dtype=torch.float32, device=DEV)
        lreg = torch.empty(B, dtype=torch.float32, device=DEV)
        A = torch.empty(E, dtype=torch.float32, device=DEV)
        _lib.rm_moe_pffn_forward_train(m.ctx, 0, X.data_ptr(), V.data_ptr(), None, None, lreg.data_ptr(),
                                       A.data_ptr(), B, torch.cuda.current_stream().cuda_stream)
        return [V, lreg, A]

    def set_tok(m):
        m.set_tokenizer(Wt, bt)

    return [
        ("block backward", layers, dict(training=True), None, block_backward),
        ("stack backward", layers, dict(training=True), None, stack_backward),
        ("host entry", layers, {}, None, host_entry),
        ("score", layers, {}, set_tok, score),
        ("tokenize backward", layers, {}, set_tok, tokenize_backward),
        ("UniMixing", layers, {}, None, set_unimixing),
        ("MoE training forward", layers_t, {}, None, moe_train),
    ]


def test_lazy_workspaces_survive_every_allocation_failure():
    """Each allocation of each lazily allocating call fails once on a fresh context: the
    call returns RM_ERR_OOM, the retry completes the workspace and computes the result of
    a context that never saw a failure, and closing the context frees everything.  Then
    on one context every retry fails at its first new allocation until the workspace is
    complete (a failed call keeps the buffers it got)."""
    layers = _layers()
    live0 = _live()

    def same(got, want, name):
        for a, b in zip(got, want):
            a64 = a.detach().to("cpu", torch.float64).numpy()
            b64 = b.detach().to("cpu", torch.float64).numpy()
            scale = max(float(np.sqrt(np.mean(b64 ** 2))), 1e-30)
            assert np.max(np.abs(a64 - b64)) <= 1e-5 * scale, f"{name}: result after failures differs"

    for name, lay, kw, setup, call in _lazy_calls(layers):
        ref_m = _create(lay, **kw)
        if setup:
            setup(ref_m)
        n = _allocations(lambda: call(ref_m))
        want = [t.clone() for t in call(ref_m)]
        torch.cuda.synchronize()
        ref_m.close()
        assert n >= 1, name
        for i in range(n):
            m = _create(lay, **kw)
            if setup:
                setup(m)
            _lib.rm_debug_fail_alloc(i)
            _expect_oom(lambda: call(m), f"{name}, allocation {i}")
            _lib.rm_debug_fail_alloc(-1)
            got = call(m)
            torch.cuda.synchronize()
            assert m.sync_status() == _lib.RM_OK, name
            same(got, want, f"{name}, failure at allocation {i}")
            m.close()
            assert _live() == live0, f"{name}: allocations leaked after a failure at allocation {i}"
        if name == "UniMixing":
            continue          # rm_set_unimixing replaces the layer's weights whole on every call
        m = _create(lay, **kw)
        if setup:
            setup(m)
        for attempt in range(n + 1):
            _lib.rm_debug_fail_alloc(0)
            try:
                got = call(m)
                break
            except _lib.RankMixerError as e:
                assert e.status == _lib.RM_ERR_OOM, f"{name}: {e}"
        _lib.rm_debug_fail_alloc(-1)
        assert attempt >= 1, f"{name}: the first call allocated nothing"
        torch.cuda.synchronize()
        same(got, want, f"{name}, progressive failures")
        m.close()
        assert _live() == live0, f"{name}: allocations leaked"
