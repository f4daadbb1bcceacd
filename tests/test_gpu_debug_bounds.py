"""The bounds-checked build (librankmixer_debug.so, -DRM_DEBUG_BOUNDS).

In that build every launcher of the forward path checks the sizes, strides
and alignments it is given against the buffers they describe, and the mixing
and GEMM-epilogue kernels guard their global-memory accesses: a guard that
fires latches an error word (reported by rm_sync_status) and skips the
access.  The guards change no arithmetic, so on valid inputs the debug build
must give the normal build's results bit for bit, with no guard firing.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from rankmixer_feature_interaction_gb300 import _lib, synth
from rankmixer_feature_interaction_gb300.api import RankMixer
lib = _lib.load()
maps = open("/proc/self/maps").read()
print("loaded", "librankmixer_debug.so" in maps, "librankmixer.so" in maps)
out = {{}}
# (dtype, path, T, D, k, L, B): CTA pairs, one-CTA tiles, weights-as-M tiles, the SIMT path, float32
for dt, path, T, D, k, L, B in [("bf16", "tcgen05", 4, 256, 2, 2, 300), ("bf16", "tcgen05", 4, 256, 2, 2, 150),
                                ("bf16", "tcgen05", 4, 256, 2, 2, 13), ("bf16", "tcgen05", 32, 1536, 1, 2, 40),
                                ("bf16", "simt", 2, 64, 1, 1, 129), ("f32", "auto", 4, 8, 2, 1, 64)]:
    layers = synth.make_stack(T, D, k, L, 77, dt, "cuda")
    m = RankMixer(T, D, k, layers, dtype=dt, max_batch=B, gemm_path=path)
    X = synth.make_input(B, T, D, 78, dt, "cuda")
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    Xo = m.block_forward(0, X, out_dtype="f32")
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    key = f"{{dt}}_{{path}}_{{T}}_{{D}}_{{B}}"
    out["pooled_" + key] = pooled.float().cpu().numpy()
    out["XL_" + key] = XL.cpu().numpy()
    out["Xo_" + key] = Xo.cpu().numpy()
    m.close()
# UniMixing in both layers (the staged tensor-core local step; bf16 and fp16 samples in)
for T, D, bs, B in [(8, 512, 64, 37), (8, 512, 32, 100)]:
    layers = synth.make_stack(T, D, 2, 2, 82, "bf16", "cuda")
    m = RankMixer(T, D, 2, layers, max_batch=B)
    for n in range(2):
        WG, WB = synth.make_unimix_weights(T, D, bs, 83 + n, "cuda")
        m.set_unimixing(n, WG, WB, tau=0.3, iters=5)
    X = synth.make_input(B, T, D, 85, "bf16", "cuda")
    pooled, XL = m.stack_forward(X, return_XL=True, xl_dtype="f32")
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    out[f"unimix_XL_{{T}}_{{D}}_{{bs}}_{{B}}"] = XL.cpu().numpy()
    m.close()
# the Sparse-MoE PFFN: one-CTA and CTA-pair expert tiles
for B in (300, 600):
    T, D, E, Fe = 2, 256, 4, 256
    p = synth.make_experts(T, D, E, Fe, 79, "bf16", "cuda")
    dense = synth.make_layer(T, D, 2, 80, "bf16", "cuda")
    dense.update(p)
    m = RankMixer(T, D, 2, [dense], max_batch=B, n_experts=E, expert_hidden=Fe)
    S = synth.make_input(B, T, D, 81, "bf16", "cuda")
    V = m.moe_pffn_forward(0, S)
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    out[f"moe_{{B}}"] = V.cpu().numpy()
    m.close()
np.savez(sys.argv[1], **out)
print("ok")
"""


def _run(tmp_path, variant):
    env = {k: v for k, v in os.environ.items() if not k.startswith("RM_")}
    if variant == "debug":
        env["RM_LIBRARY"] = "debug"
    path = str(tmp_path / f"{variant}.npz")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT), path], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-3000:]
    return r.stdout, dict(np.load(path))


def test_bounds_checked_build_matches_the_normal_build(tmp_path):
    from rankmixer_feature_interaction_gb300 import build
    build.build(debug_bounds=True)
    out_dbg, got = _run(tmp_path, "debug")
    out_std, want = _run(tmp_path, "normal")
    assert "loaded True False" in out_dbg, out_dbg
    assert "loaded False True" in out_std, out_std
    assert got.keys() == want.keys()
    for key in want:
        a, b = got[key], want[key]
        assert a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32)), key
