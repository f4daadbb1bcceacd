"""ctypes binding of librankmixer.so (include/rankmixer.h), names unchanged.

Argument marshalling only: every function forwards to the C entry point of
the same name.  Loading fails loudly when the library has not been built --
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# RM_LIBRARY=debug selects the bounds-checked build librankmixer_debug.so
# (python -m rankmixer_feature_interaction_gb300.build --debug-bounds)
LIB_NAME = "librankmixer_debug.so" if os.environ.get("RM_LIBRARY") == "debug" else "librankmixer.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

# rm_status
RM_OK = 0
RM_ERR_INVALID_ARG = 1
RM_ERR_UNSUPPORTED = 2
RM_ERR_CUDA = 3
RM_ERR_OOM = 4
RM_ERR_TIMEOUT = 5
RM_ERR_DEVICE = 6
STATUS_NAMES = {0: "RM_OK", 1: "RM_ERR_INVALID_ARG", 2: "RM_ERR_UNSUPPORTED", 3: "RM_ERR_CUDA",
                4: "RM_ERR_OOM", 5: "RM_ERR_TIMEOUT", 6: "RM_ERR_DEVICE"}

# rm_dtype
RM_F32 = 0
RM_BF16 = 1

# rm_gemm_path
RM_PATH_AUTO = 0
RM_PATH_SIMT = 1
RM_PATH_TCGEN05 = 2

# rm_kernel_kind
KERNEL_KINDS = ["mix_ln1", "gemm1", "gemm2", "ln2_out", "pool", "rowstats", "moe_route", "moe_gemm1",
                "moe_gemm2", "misc", "moe_combine", "bwd_recompute", "bwd_dgrad", "bwd_wgrad", "bwd_rows",
                "tokenize", "head", "unimix", "pffn"]
RM_K_COUNT = len(KERNEL_KINDS)

EXPORTED = ["rm_create", "rm_destroy", "rm_block_forward", "rm_stack_forward", "rm_stack_forward_host",
            "rm_moe_pffn_forward", "rm_token_mix", "rm_sync_status", "rm_get_info", "rm_profile_enable",
            "rm_profile_read", "rm_debug_wait_timeout", "rm_last_error", "rm_abi_version",
            "rm_block_forward_noalloc", "rm_debug_gelu", "rm_block_backward", "rm_stack_backward",
            "rm_debug_gelu_grad", "rm_stack_forward_train", "rm_stack_backward_saved", "rm_head_forward",
            "rm_set_tokenizer", "rm_tokenize", "rm_score", "rm_moe_pffn_forward_train", "rm_tokenize_backward",
            "rm_set_unimixing", "rm_unimixing_weights", "rm_unimixing", "rm_debug_mix_residual",
            "rm_debug_fail_alloc", "rm_debug_alloc_stats", "rm_stack_forward_host_async", "rm_host_wait"]


class rm_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int), ("k", ctypes.c_int),
                ("L", ctypes.c_int), ("n_experts", ctypes.c_int), ("expert_hidden", ctypes.c_int),
                ("moe_layer_mask", ctypes.c_uint), ("dtype", ctypes.c_int), ("ln_eps", ctypes.c_float),
                ("max_batch", ctypes.c_int), ("gemm_path", ctypes.c_int), ("training", ctypes.c_int)]


class rm_layer_params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W1", "b1", "W2", "b2", "ln1_gamma", "ln1_beta", "ln2_gamma",
                                               "ln2_beta", "Wg", "bg", "eW1", "eb1", "eW2", "eb2", "Wg_train",
                                               "bg_train")]


GRAD_FIELDS = ("dW1", "db1", "dW2", "db2", "dln1_gamma", "dln1_beta", "dln2_gamma", "dln2_beta")


class rm_layer_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in GRAD_FIELDS]


class rm_info(ctypes.Structure):
    _fields_ = [("params_per_layer", ctypes.c_longlong), ("flops_per_sample", ctypes.c_longlong),
                ("weight_bytes", ctypes.c_longlong), ("workspace_bytes", ctypes.c_longlong),
                ("gemm_path", ctypes.c_int), ("num_sms", ctypes.c_int), ("device", ctypes.c_int)]


class rm_kernel_stat(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_longlong), ("total_ms", ctypes.c_double)]


class RankMixerError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load librankmixer.so (or the bounds-checked build under RM_LIBRARY=debug); raise if it
    is missing (build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_NAME} not built at {LIB_PATH}; run `python -c 'import __graft_entry__ as g; "
                           f"g.build()'` (there is no non-CUDA fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = {
        "rm_create": (st, [ctypes.POINTER(rm_config), ctypes.POINTER(rm_layer_params), i, ctypes.POINTER(vp)]),
        "rm_destroy": (st, [vp]),
        "rm_block_forward": (st, [vp, i, vp, vp, vp, i, i, vp]),
        "rm_stack_forward": (st, [vp, vp, vp, vp, i, i, vp]),
        "rm_stack_forward_host": (st, [vp, vp, vp, i, vp]),
        "rm_stack_forward_host_async": (st, [vp, vp, vp, i, vp, ctypes.POINTER(ctypes.c_longlong)]),
        "rm_host_wait": (st, [vp, ctypes.c_longlong]),
        "rm_moe_pffn_forward": (st, [vp, i, vp, vp, vp, i, vp]),
        "rm_token_mix": (st, [vp, vp, i, i, i, i, i, vp]),
        "rm_sync_status": (st, [vp, vp]),
        "rm_get_info": (st, [vp, ctypes.POINTER(rm_info)]),
        "rm_profile_enable": (st, [vp, i]),
        "rm_profile_read": (st, [vp, ctypes.POINTER(rm_kernel_stat)]),
        "rm_debug_wait_timeout": (st, [vp, i, vp]),
        "rm_last_error": (ctypes.c_char_p, []),
        "rm_abi_version": (i, []),
        "rm_block_forward_noalloc": (st, [vp, i, vp, vp, i, vp]),
        "rm_debug_gelu": (st, [vp, vp, ctypes.c_longlong, ctypes.c_int, vp]),
        "rm_block_backward": (st, [vp, i, vp, vp, vp, ctypes.POINTER(rm_layer_grads), i, vp]),
        "rm_stack_backward": (st, [vp, vp, vp, vp, ctypes.POINTER(rm_layer_grads), i, vp]),
        "rm_debug_gelu_grad": (st, [vp, vp, ctypes.c_longlong, vp]),
        "rm_stack_forward_train": (st, [vp, vp, vp, i, vp]),
        "rm_head_forward": (st, [vp, vp, ctypes.c_float, vp, vp, vp, vp, i, i, i, vp]),
        "rm_set_tokenizer": (st, [vp, vp, vp, i]),
        "rm_tokenize": (st, [vp, vp, vp, i, vp]),
        "rm_tokenize_backward": (st, [vp, vp, vp, vp, vp, vp, i, vp]),
        "rm_score": (st, [vp, vp, vp, ctypes.c_float, vp, i, vp]),
        "rm_moe_pffn_forward_train": (st, [vp, i, vp, vp, vp, vp, vp, vp, i, vp]),
        "rm_stack_backward_saved": (st, [vp, vp, vp, ctypes.POINTER(rm_layer_grads), i, vp]),
        "rm_set_unimixing": (st, [vp, i, vp, vp, i, ctypes.c_float, i, vp]),
        "rm_unimixing_weights": (st, [vp, i, vp, vp, vp]),
        "rm_unimixing": (st, [vp, i, vp, vp, i, i, vp]),
        "rm_debug_mix_residual": (st, [vp, i, vp, i, i, i, vp]),
        "rm_debug_fail_alloc": (st, [ctypes.c_longlong]),
        "rm_debug_alloc_stats": (st, [ctypes.POINTER(ctypes.c_longlong)] * 3),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    if status != RM_OK:
        msg = load().rm_last_error()
        raise RankMixerError(status, where, msg.decode() if msg else "")


# ---- thin wrappers with the C names (pointers are ints, streams are ints) ----

def rm_create(cfg: rm_config, layers, device: int = 0) -> int:
    arr = (rm_layer_params * len(layers))(*layers)
    out = ctypes.c_void_p()
    check(load().rm_create(ctypes.byref(cfg), arr, device, ctypes.byref(out)), "rm_create")
    return out.value


def rm_destroy(ctx: int) -> None:
    check(load().rm_destroy(ctx), "rm_destroy")


def rm_block_forward(ctx: int, layer: int, X_in: int, X_out: int, S_out: int | None, out_dtype: int, B: int,
                     stream: int) -> None:
    check(load().rm_block_forward(ctx, layer, X_in, X_out, S_out, out_dtype, B, stream), "rm_block_forward")


def rm_block_forward_noalloc(ctx: int, layer: int, X_in: int, X_out: int, B: int, stream: int) -> None:
    check(load().rm_block_forward_noalloc(ctx, layer, X_in, X_out, B, stream), "rm_block_forward_noalloc")


def rm_stack_forward(ctx: int, X0: int, pooled: int, XL: int | None, xl_dtype: int, B: int, stream: int) -> None:
    check(load().rm_stack_forward(ctx, X0, pooled, XL, xl_dtype, B, stream), "rm_stack_forward")


def rm_stack_forward_host(ctx: int, X0_host: int, pooled_host: int, B: int, stream: int) -> None:
    check(load().rm_stack_forward_host(ctx, X0_host, pooled_host, B, stream), "rm_stack_forward_host")


def rm_stack_forward_host_async(ctx: int, X0_host: int, pooled_host: int, B: int, stream: int) -> int:
    t = ctypes.c_longlong(-1)
    check(load().rm_stack_forward_host_async(ctx, X0_host, pooled_host, B, stream, ctypes.byref(t)),
          "rm_stack_forward_host_async")
    return t.value


def rm_host_wait(ctx: int, ticket: int) -> None:
    check(load().rm_host_wait(ctx, ticket), "rm_host_wait")


def rm_moe_pffn_forward(ctx: int, layer: int, S: int, V_out: int, gates: int | None, B: int, stream: int) -> None:
    check(load().rm_moe_pffn_forward(ctx, layer, S, V_out, gates, B, stream), "rm_moe_pffn_forward")


def rm_token_mix(X: int, Y: int, B: int, T: int, D: int, H: int, dtype: int, stream: int) -> None:
    check(load().rm_token_mix(X, Y, B, T, D, H, dtype, stream), "rm_token_mix")


def rm_sync_status(ctx: int, stream: int) -> int:
    """Returns the raw status (RM_OK, RM_ERR_TIMEOUT, ...) without raising."""
    return load().rm_sync_status(ctx, stream)


def rm_get_info(ctx: int) -> rm_info:
    info = rm_info()
    check(load().rm_get_info(ctx, ctypes.byref(info)), "rm_get_info")
    return info


def rm_profile_enable(ctx: int, on: bool) -> None:
    check(load().rm_profile_enable(ctx, 1 if on else 0), "rm_profile_enable")


def rm_profile_read(ctx: int) -> dict:
    arr = (rm_kernel_stat * RM_K_COUNT)()
    check(load().rm_profile_read(ctx, arr), "rm_profile_read")
    return {KERNEL_KINDS[k]: (arr[k].launches, arr[k].total_ms) for k in range(RM_K_COUNT)}


def rm_debug_wait_timeout(ctx: int, timeout_us: int, stream: int) -> None:
    check(load().rm_debug_wait_timeout(ctx, timeout_us, stream), "rm_debug_wait_timeout")


def rm_debug_gelu(u: int, out: int, n: int, form: int, stream: int) -> None:
    check(load().rm_debug_gelu(u, out, n, form, stream), "rm_debug_gelu")


def rm_block_backward(ctx: int, layer: int, X_in: int, dX_out: int, dX_in: int, grads: rm_layer_grads | None,
                      B: int, stream: int) -> None:
    gp = ctypes.byref(grads) if grads is not None else None
    check(load().rm_block_backward(ctx, layer, X_in, dX_out, dX_in, gp, B, stream), "rm_block_backward")


def rm_stack_backward(ctx: int, X0: int, dpooled: int, dX0: int, grads: list | None, B: int, stream: int) -> None:
    arr = (rm_layer_grads * len(grads))(*grads) if grads else None
    check(load().rm_stack_backward(ctx, X0, dpooled, dX0, arr, B, stream), "rm_stack_backward")


def rm_stack_forward_train(ctx: int, X0: int, pooled: int, B: int, stream: int) -> None:
    check(load().rm_stack_forward_train(ctx, X0, pooled, B, stream), "rm_stack_forward_train")


def rm_stack_backward_saved(ctx: int, dpooled: int, dX0: int, grads: list | None, B: int, stream: int) -> None:
    arr = (rm_layer_grads * len(grads))(*grads) if grads else None
    check(load().rm_stack_backward_saved(ctx, dpooled, dX0, arr, B, stream), "rm_stack_backward_saved")


def rm_head_forward(pooled: int, w: int, b: float, y: int | None, p: int | None, loss: int | None,
                    dpooled: int | None, B: int, D: int, mean_loss: bool, stream: int) -> None:
    check(load().rm_head_forward(pooled, w, b, y, p, loss, dpooled, B, D, 1 if mean_loss else 0, stream),
          "rm_head_forward")


def rm_moe_pffn_forward_train(ctx: int, layer: int, S: int, V: int, gates_train: int | None, gates_infer: int | None,
                              lreg: int | None, A: int | None, B: int, stream: int) -> None:
    check(load().rm_moe_pffn_forward_train(ctx, layer, S, V, gates_train, gates_infer, lreg, A, B, stream),
          "rm_moe_pffn_forward_train")


def rm_set_tokenizer(ctx: int, W: int, bias: int, d: int) -> None:
    check(load().rm_set_tokenizer(ctx, W, bias, d), "rm_set_tokenizer")


def rm_tokenize(ctx: int, E: int, X0: int, B: int, stream: int) -> None:
    check(load().rm_tokenize(ctx, E, X0, B, stream), "rm_tokenize")


def rm_tokenize_backward(ctx: int, E: int, dX0: int, dE: int | None, dW: int, db: int, B: int, stream: int) -> None:
    check(load().rm_tokenize_backward(ctx, E, dX0, dE, dW, db, B, stream), "rm_tokenize_backward")


def rm_score(ctx: int, E: int, head_w: int, head_b: float, p: int, B: int, stream: int) -> None:
    check(load().rm_score(ctx, E, head_w, head_b, p, B, stream), "rm_score")


def rm_set_unimixing(ctx: int, layer: int, WG: int, WB: int, bs: int, tau: float, iters: int, stream: int) -> None:
    check(load().rm_set_unimixing(ctx, layer, WG, WB, bs, tau, iters, stream), "rm_set_unimixing")


def rm_unimixing_weights(ctx: int, layer: int, WG_out: int | None, WB_out: int | None, stream: int) -> None:
    check(load().rm_unimixing_weights(ctx, layer, WG_out, WB_out, stream), "rm_unimixing_weights")


def rm_unimixing(ctx: int, layer: int, X: int, Y: int, out_dtype: int, B: int, stream: int) -> None:
    check(load().rm_unimixing(ctx, layer, X, Y, out_dtype, B, stream), "rm_unimixing")


def rm_debug_mix_residual(X: int, from_z: bool, Y: int, B: int, T: int, D: int, stream: int) -> None:
    check(load().rm_debug_mix_residual(X, 1 if from_z else 0, Y, B, T, D, stream), "rm_debug_mix_residual")


def rm_debug_fail_alloc(after: int) -> None:
    check(load().rm_debug_fail_alloc(after), "rm_debug_fail_alloc")


def rm_debug_alloc_stats() -> tuple[int, int, int]:
    """(allocations made since load, live allocations, live bytes)."""
    v = [ctypes.c_longlong() for _ in range(3)]
    check(load().rm_debug_alloc_stats(*[ctypes.byref(x) for x in v]), "rm_debug_alloc_stats")
    return v[0].value, v[1].value, v[2].value


def rm_debug_gelu_grad(u: int, out: int, n: int, stream: int) -> None:
    check(load().rm_debug_gelu_grad(u, out, n, stream), "rm_debug_gelu_grad")


def rm_last_error() -> str:
    m = load().rm_last_error()
    return m.decode() if m else ""


def rm_abi_version() -> int:
    return load().rm_abi_version()
