"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/rankmixer.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from rankmixer_feature_interaction_gb300 import _lib
from rankmixer_feature_interaction_gb300 import build as rm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rankmixer.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        rm_build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:RM_API\s+)?(?:rm_status\s+|const\s+char\s*\*\s*|int\s+)(rm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("rm_create", "rm_destroy", "rm_block_forward", "rm_stack_forward", "rm_moe_pffn_forward",
                 "rm_token_mix", "rm_last_error"):
        assert must in names
    assert set(names) == set(_lib.EXPORTED), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} missing from librankmixer.so"
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(rm_\w+)\b", out))
    assert set(declared_functions()) <= exported
    assert exported <= set(declared_functions()), f"undeclared exports: {exported - set(declared_functions())}"


def test_abi_version(lib):
    assert _lib.rm_abi_version() == 4


def _cfg(**kw):
    base = dict(T=4, D=8, H=4, k=2, L=1, n_experts=0, expert_hidden=0, moe_layer_mask=0, dtype=_lib.RM_F32,
                ln_eps=1e-5, max_batch=16, gemm_path=_lib.RM_PATH_AUTO, training=0)
    base.update(kw)
    return _lib.rm_config(**base)


def _create_status(lib, cfg, layers=True):
    out = ctypes.c_void_p()
    arr = (_lib.rm_layer_params * max(cfg.L if cfg is not None else 1, 1))() if layers else None
    return lib.rm_create(ctypes.byref(cfg) if cfg is not None else None, arr, 0, ctypes.byref(out)), out.value


def test_create_rejects_bad_configs_on_host(lib):
    st, ctx = _create_status(lib, None)
    assert st == _lib.RM_ERR_INVALID_ARG and ctx is None
    st, _ = _create_status(lib, _cfg(H=2))                     # H != T: needs the [T][D] shape for the residual
    assert st == _lib.RM_ERR_UNSUPPORTED
    assert "H (2) must equal T (4)" in _lib.rm_last_error()
    st, _ = _create_status(lib, _cfg(D=9))                     # D % H != 0
    assert st == _lib.RM_ERR_INVALID_ARG
    st, _ = _create_status(lib, _cfg(max_batch=0))
    assert st == _lib.RM_ERR_INVALID_ARG
    st, _ = _create_status(lib, _cfg(dtype=7))
    assert st == _lib.RM_ERR_INVALID_ARG
    st, _ = _create_status(lib, _cfg(ln_eps=-1.0))
    assert st == _lib.RM_ERR_INVALID_ARG
    st, _ = _create_status(lib, _cfg(moe_layer_mask=1))        # MoE layer without experts
    assert st == _lib.RM_ERR_INVALID_ARG
    st, _ = _create_status(lib, _cfg(T=32, H=32, D=4096, dtype=_lib.RM_BF16))   # sample too big for one CTA
    assert st == _lib.RM_ERR_UNSUPPORTED
    st, _ = _create_status(lib, _cfg(), layers=False)
    assert st == _lib.RM_ERR_INVALID_ARG


def test_token_mix_rejects_bad_arguments_on_host(lib):
    assert lib.rm_token_mix(None, None, 1, 4, 8, 4, _lib.RM_F32, None) == _lib.RM_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(1024)
    p = ctypes.addressof(buf)
    assert lib.rm_token_mix(p, p + 512, 1, 4, 8, 3, _lib.RM_F32, None) == _lib.RM_ERR_INVALID_ARG   # D % H
    assert lib.rm_token_mix(p, p + 64, 1, 4, 8, 4, _lib.RM_F32, None) == _lib.RM_ERR_INVALID_ARG    # overlap
    assert lib.rm_token_mix(p, p + 512, 0, 4, 8, 4, _lib.RM_F32, None) == _lib.RM_ERR_INVALID_ARG   # B = 0
    assert lib.rm_token_mix(p, p + 512, 1, 4, 8, 4, 9, None) == _lib.RM_ERR_INVALID_ARG             # dtype


def test_null_context_calls(lib):
    assert lib.rm_destroy(None) == _lib.RM_OK
    info = _lib.rm_info()
    assert lib.rm_get_info(None, ctypes.byref(info)) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_block_forward(None, 0, None, None, None, _lib.RM_BF16, 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_stack_forward(None, None, None, None, _lib.RM_BF16, 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_moe_pffn_forward(None, 0, None, None, None, 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_sync_status(None, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_profile_enable(None, 1) == _lib.RM_ERR_INVALID_ARG
    assert "ctx is NULL" in _lib.rm_last_error()
    assert lib.rm_debug_gelu(None, None, 0, 2, None) == _lib.RM_ERR_INVALID_ARG      # unknown form
    assert lib.rm_debug_gelu(None, None, -1, 0, None) == _lib.RM_ERR_INVALID_ARG     # n < 0
    assert lib.rm_debug_gelu(None, None, 5, 1, None) == _lib.RM_ERR_INVALID_ARG      # NULL buffers
    grads = _lib.rm_layer_grads()
    assert lib.rm_block_backward(None, 0, None, None, None, ctypes.byref(grads), 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_stack_backward(None, None, None, None, ctypes.byref(grads), 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_stack_forward_train(None, None, None, 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_stack_backward_saved(None, None, None, ctypes.byref(grads), 1, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_debug_gelu_grad(None, None, -1, None) == _lib.RM_ERR_INVALID_ARG   # n < 0
    assert lib.rm_debug_gelu_grad(None, None, 3, None) == _lib.RM_ERR_INVALID_ARG    # NULL buffers
    assert lib.rm_set_unimixing(None, 0, None, None, 4, 1.0, 5, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_unimixing_weights(None, 0, None, None, None) == _lib.RM_ERR_INVALID_ARG
    assert lib.rm_unimixing(None, 0, None, None, _lib.RM_BF16, 1, None) == _lib.RM_ERR_INVALID_ARG
    assert "ctx is NULL" in _lib.rm_last_error()


def test_debug_mix_residual_rejects_bad_arguments_on_host(lib):
    buf = ctypes.create_string_buffer(1 << 16)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.rm_debug_mix_residual(None, 0, None, 1, 4, 256, None) == _lib.RM_ERR_INVALID_ARG   # NULL
    assert lib.rm_debug_mix_residual(p, 0, p + 8192, 1, 3, 256, None) == _lib.RM_ERR_INVALID_ARG  # D % T
    assert lib.rm_debug_mix_residual(p, 0, p + 8192, 0, 4, 256, None) == _lib.RM_ERR_INVALID_ARG  # B = 0
    assert lib.rm_debug_mix_residual(p, 0, p + 1024, 1, 4, 256, None) == _lib.RM_ERR_INVALID_ARG  # overlap
    assert lib.rm_debug_mix_residual(p + 2, 0, p + 8192, 1, 4, 256, None) == _lib.RM_ERR_INVALID_ARG   # alignment


def test_config_struct_matches_the_header(lib):
    """The binding's rm_config / rm_layer_grads mirror the header field by field."""
    text = open(HEADER, encoding="utf-8").read()
    body = re.search(r"typedef struct rm_config \{(.*?)\} rm_config;", text, flags=re.S).group(1)
    fields = re.findall(r"(\w+);", body)
    assert fields == [f for f, _ in _lib.rm_config._fields_]
    body = re.search(r"typedef struct rm_layer_grads \{(.*?)\} rm_layer_grads;", text, flags=re.S).group(1)
    names = re.findall(r"\*(\w+)", body)
    assert names == [f for f, _ in _lib.rm_layer_grads._fields_]


def test_binding_raises_with_status_and_message(lib):
    with pytest.raises(_lib.RankMixerError) as e:
        _lib.rm_token_mix(0, 0, 1, 4, 8, 4, _lib.RM_F32, 0)
    assert e.value.status == _lib.RM_ERR_INVALID_ARG
    assert "NULL" in str(e.value)


def test_allocation_hooks_answer_without_a_device(lib):
    made = ctypes.c_longlong(-1)
    live = ctypes.c_longlong(-1)
    nbytes = ctypes.c_longlong(-1)
    assert lib.rm_debug_alloc_stats(ctypes.byref(made), ctypes.byref(live), ctypes.byref(nbytes)) == _lib.RM_OK
    assert made.value >= 0 and live.value >= 0 and nbytes.value >= 0
    assert lib.rm_debug_alloc_stats(None, None, None) == _lib.RM_OK
    assert lib.rm_debug_fail_alloc(3) == _lib.RM_OK
    assert lib.rm_debug_fail_alloc(-1) == _lib.RM_OK


def test_binding_selects_the_bounds_checked_build_by_environment():
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); from rankmixer_feature_interaction_gb300 import _lib; "
            "print(_lib.LIB_NAME)" % ROOT)
    for env_value, want in ((None, "librankmixer.so"), ("debug", "librankmixer_debug.so")):
        env = {k: v for k, v in os.environ.items() if k != "RM_LIBRARY"}
        if env_value:
            env["RM_LIBRARY"] = env_value
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
        assert r.returncode == 0 and r.stdout.strip() == want, r.stdout + r.stderr
