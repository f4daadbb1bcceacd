"""rm_block_forward_noalloc: the block forward for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the model -- a serving loop
whose device memory belongs to a pool or framework allocator, a plugin with a
fixed memory budget, or code that must not risk the synchronisation an
allocation can cause.  This entry point keeps its intermediates in a static
device array compiled into the library instead of a workspace.  These tests
call it through the C ABI twice in a row and check each result against
rm_block_forward's (the same kernels on the same values: bit for bit, which
is within every tolerance the other parity tests use), and check that the
largest batch the refusal message names runs while one sample more is
refused.  The file is named to be collected last.
"""
import re

import pytest
import torch

from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer

pytestmark = pytest.mark.gpu


def _noalloc(m: RankMixer, layer: int, X: torch.Tensor) -> torch.Tensor:
    out = torch.empty_like(X)
    _lib.rm_block_forward_noalloc(m.ctx, layer, X.data_ptr(), out.data_ptr(), X.shape[0],
                                  torch.cuda.current_stream().cuda_stream)
    return out


@pytest.mark.parametrize("dtype,T,D,k,L,B,path", [("bf16", 16, 768, 4, 2, 64, "tcgen05"),
                                                  ("bf16", 4, 256, 2, 1, 100, "simt"),
                                                  ("f32", 4, 8, 2, 1, 64, "simt")])
def test_noalloc_matches_block_forward_on_two_calls(dtype, T, D, k, L, B, path):
    layers = synth.make_stack(T, D, k, L, 77, dtype, "cuda")
    m = RankMixer(T, D, k, layers, dtype=dtype, max_batch=B, gemm_path=path)
    assert m.path == path
    for call, seed in enumerate((78, 79)):        # two calls in a row, different inputs
        layer = call % L
        X = synth.make_input(B, T, D, seed, dtype, "cuda")
        got = _noalloc(m, layer, X)
        ref = m.block_forward(layer, X)
        torch.cuda.synchronize()
        assert m.sync_status() == _lib.RM_OK
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref), f"noalloc call {call + 1} differs from rm_block_forward"
    m.close()


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_noalloc_batch_limit_and_batches_beyond_max_batch(path):
    T, D, k = 16, 768, 4
    layers = synth.make_stack(T, D, k, 1, 80, "bf16", "cuda")
    m = RankMixer(T, D, k, layers, max_batch=8, gemm_path=path)
    X = synth.make_input(400, T, D, 81, "bf16", "cuda")
    with pytest.raises(_lib.RankMixerError) as e:
        _noalloc(m, 0, X)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    assert "static scratch" in str(e.value)
    limit = int(re.search(r"B <= (\d+)", str(e.value)).group(1))
    assert 150 < limit < 400
    with pytest.raises(_lib.RankMixerError) as e:          # one sample past the named limit
        _noalloc(m, 0, X[:limit + 1].contiguous())
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    # batches above the context's max_batch (8) run with the right row strides: equal to
    # rm_block_forward on a context with room for them
    big = RankMixer(T, D, k, layers, max_batch=limit, gemm_path=path)
    for B in (150, limit):
        Xb = X[:B].contiguous()
        got = _noalloc(m, 0, Xb)
        ref = big.block_forward(0, Xb)
        torch.cuda.synchronize()
        assert m.sync_status() == _lib.RM_OK
        assert torch.equal(got, ref), f"B={B}: noalloc differs from rm_block_forward"
    big.close()
    m.close()
