"""Torch-facing wrapper over the C ABI: allocates output tensors with torch and
passes raw pointers and the current CUDA stream to librankmixer.so.  No
arithmetic of the method happens here; every step runs in the CUDA kernels.
"""
from __future__ import annotations

import torch

from . import _lib

_DENSE_KEYS = ("W1", "b1", "W2", "b2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")
_MOE_KEYS = ("Wg", "bg", "eW1", "eb1", "eW2", "eb2")
_MOE_TRAIN_KEYS = ("Wg_train", "bg_train")
_C_NAMES = {"W1": "W1", "b1": "b1", "W2": "W2", "b2": "b2", "ln1_g": "ln1_gamma", "ln1_b": "ln1_beta",
            "ln2_g": "ln2_gamma", "ln2_b": "ln2_beta", "Wg": "Wg", "bg": "bg", "eW1": "eW1", "eb1": "eb1",
            "eW2": "eW2", "eb2": "eb2", "Wg_train": "Wg_train", "bg_train": "bg_train"}
_DTYPES = {"bf16": (torch.bfloat16, _lib.RM_BF16), "f32": (torch.float32, _lib.RM_F32)}
_PATHS = {"auto": _lib.RM_PATH_AUTO, "simt": _lib.RM_PATH_SIMT, "tcgen05": _lib.RM_PATH_TCGEN05}


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _out_dtype(name: str | None, ctx_tdtype: torch.dtype) -> tuple[torch.dtype, int]:
    """Output tensor dtype and rm_dtype code: None -> the context dtype, "f32" -> float32."""
    if name is None:
        return ctx_tdtype, (_lib.RM_F32 if ctx_tdtype == torch.float32 else _lib.RM_BF16)
    return _DTYPES[name]


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to librankmixer must be contiguous")
    return t.data_ptr()


class RankMixer:
    """A RankMixer block stack held on one GPU (one rm_ctx).

    layers: list of L dicts of contiguous tensors on `device` in `dtype` with the
    pages' layout -- W1 [T,D,kD], b1 [T,kD], W2 [T,kD,D], b2 [T,D], ln1_g/ln1_b/
    ln2_g/ln2_b [D]; with experts also Wg [T,D,E], bg [T,E], eW1 [T,E,D,Fe],
    eb1 [T,E,Fe], eW2 [T,E,Fe,D], eb2 [T,E,D].  The tensors may be freed after
    construction (the library keeps packed copies)."""

    def __init__(self, T: int, D: int, k: int, layers: list, dtype: str = "bf16", eps: float = 1e-5,
                 max_batch: int = 4096, n_experts: int = 0, expert_hidden: int = 0, moe_layer_mask: int = 0,
                 gemm_path: str = "auto", device: int = 0, training: bool = False):
        self.tdtype, cdtype = _DTYPES[dtype]
        self.T, self.D, self.k, self.L = T, D, k, len(layers)
        self.E = n_experts
        self.max_batch = max_batch
        self.device = torch.device("cuda", device)
        cfg = _lib.rm_config(T=T, D=D, H=T, k=k, L=len(layers), n_experts=n_experts, expert_hidden=expert_hidden,
                             moe_layer_mask=moe_layer_mask, dtype=cdtype, ln_eps=eps, max_batch=max_batch,
                             gemm_path=_PATHS[gemm_path], training=1 if training else 0)
        cl = []
        for p in layers:
            lp = _lib.rm_layer_params()
            for k_ in _DENSE_KEYS + (_MOE_KEYS if n_experts > 0 else ()):
                setattr(lp, _C_NAMES[k_], _ptr(p[k_]))
            if n_experts > 0 and "Wg_train" in p:
                for k_ in _MOE_TRAIN_KEYS:
                    setattr(lp, _C_NAMES[k_], _ptr(p[k_]))
            cl.append(lp)
        torch.cuda.synchronize(self.device)
        self.ctx = _lib.rm_create(cfg, cl, device)
        self.info = _lib.rm_get_info(self.ctx)

    # -- lifetime --------------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "ctx", None):
            _lib.rm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def path(self) -> str:
        return "tcgen05" if self.info.gemm_path == _lib.RM_PATH_TCGEN05 else "simt"

    # -- forward calls -----------------------------------------------------------
    def block_forward(self, layer: int, X: torch.Tensor, out: torch.Tensor | None = None, return_S: bool = False,
                      out_dtype: str | None = None):
        """X_out (and S with return_S) in the context dtype, or float32 with out_dtype="f32"."""
        B = X.shape[0]
        tdt, code = _out_dtype(out_dtype, self.tdtype)
        out = torch.empty(X.shape, dtype=tdt, device=X.device) if out is None else out
        S = torch.empty(X.shape, dtype=tdt, device=X.device) if return_S else None
        _lib.rm_block_forward(self.ctx, layer, _ptr(X), _ptr(out), _ptr(S), code, B, _stream())
        return (out, S) if return_S else out

    def stack_forward(self, X0: torch.Tensor, pooled: torch.Tensor | None = None, return_XL: bool = False,
                      xl_dtype: str | None = None):
        """pooled (float32), and X_L with return_XL in the context dtype or float32 (xl_dtype="f32")."""
        B = X0.shape[0]
        pooled = torch.empty((B, self.D), dtype=torch.float32, device=X0.device) if pooled is None else pooled
        tdt, code = _out_dtype(xl_dtype, self.tdtype)
        XL = torch.empty(X0.shape, dtype=tdt, device=X0.device) if return_XL else None
        _lib.rm_stack_forward(self.ctx, _ptr(X0), _ptr(pooled), _ptr(XL), code, B, _stream())
        return (pooled, XL) if return_XL else pooled

    def stack_forward_host(self, X0_host: torch.Tensor, pooled_host: torch.Tensor | None = None) -> torch.Tensor:
        """X0_host: CPU tensor (pinned for full speed); returns the pooled CPU float32 [B, D]."""
        B = X0_host.shape[0]
        if pooled_host is None:
            pooled_host = torch.empty((B, self.D), dtype=torch.float32, pin_memory=X0_host.is_pinned())
        _lib.rm_stack_forward_host(self.ctx, _ptr(X0_host), _ptr(pooled_host), B, _stream())
        return pooled_host

    def stack_forward_host_async(self, X0_host: torch.Tensor, pooled_host: torch.Tensor) -> int:
        """Enqueue the stack forward of a host batch (pinned CPU tensors; the copy in runs while
        the previous batch computes); returns a ticket for host_wait.  Keep both tensors alive
        and unmodified until the ticket has been waited for."""
        return _lib.rm_stack_forward_host_async(self.ctx, _ptr(X0_host), _ptr(pooled_host), X0_host.shape[0],
                                                _stream())

    def host_wait(self, ticket: int) -> None:
        """Return once the batch of `ticket` has its pooled output in its host tensor."""
        _lib.rm_host_wait(self.ctx, ticket)

    def moe_pffn_forward(self, layer: int, S: torch.Tensor, V: torch.Tensor | None = None,
                         return_gates: bool = False):
        B = S.shape[0]
        V = torch.empty(S.shape, dtype=torch.float32, device=S.device) if V is None else V
        G = torch.empty((B, self.T, self.E), dtype=torch.float32, device=S.device) if return_gates else None
        _lib.rm_moe_pffn_forward(self.ctx, layer, _ptr(S), _ptr(V), _ptr(G), B, _stream())
        return (V, G) if return_gates else V

    def moe_pffn_forward_train(self, layer: int, S: torch.Tensor, V: torch.Tensor | None = None) -> dict:
        """Dense-training / sparse-inference MoE PFFN forward: V on the training router's
        gates, plus both routers' gates, the per-sample regulariser lreg and the per-expert
        activation A of the inference router."""
        B = S.shape[0]
        V = torch.empty(S.shape, dtype=torch.float32, device=S.device) if V is None else V
        gt = torch.empty((B, self.T, self.E), dtype=torch.float32, device=S.device)
        gi = torch.empty_like(gt)
        lreg = torch.empty(B, dtype=torch.float32, device=S.device)
        A = torch.empty(self.E, dtype=torch.float32, device=S.device)
        _lib.rm_moe_pffn_forward_train(self.ctx, layer, _ptr(S), _ptr(V), _ptr(gt), _ptr(gi), _ptr(lreg), _ptr(A), B,
                                       _stream())
        return {"V": V, "G_train": gt, "G_infer": gi, "lreg": lreg, "A": A}

    # -- backward calls (contexts created with training=True) -------------------------
    def grad_numel(self) -> int:
        """Float32 values of one layer's parameter gradients."""
        T, D, F = self.T, self.D, self.k * self.D
        return 2 * T * D * F + T * F + T * D + 4 * D

    def _grad_tensors(self, dev, flat: torch.Tensor | None = None) -> tuple[dict, _lib.rm_layer_grads]:
        T, D, F = self.T, self.D, self.k * self.D
        shapes = {"dW1": (T, D, F), "db1": (T, F), "dW2": (T, F, D), "db2": (T, D), "dln1_g": (D,),
                  "dln1_b": (D,), "dln2_g": (D,), "dln2_b": (D,)}
        if flat is None:
            g = {k_: torch.empty(v, dtype=torch.float32, device=dev) for k_, v in shapes.items()}
        else:   # views into one buffer (16-byte aligned pieces), e.g. for a single all-reduce
            g, off = {}, 0
            for k_, v in shapes.items():
                n = 1
                for x in v:
                    n *= x
                g[k_] = flat[off:off + n].view(v)
                off += (n + 3) // 4 * 4
        c = _lib.rm_layer_grads(dW1=_ptr(g["dW1"]), db1=_ptr(g["db1"]), dW2=_ptr(g["dW2"]), db2=_ptr(g["db2"]),
                                dln1_gamma=_ptr(g["dln1_g"]), dln1_beta=_ptr(g["dln1_b"]),
                                dln2_gamma=_ptr(g["dln2_g"]), dln2_beta=_ptr(g["dln2_b"]))
        return g, c

    def block_backward(self, layer: int, X: torch.Tensor, G: torch.Tensor, dX: torch.Tensor | None = None):
        """Gradients of one block for the loss whose gradient at the block output is G
        (float32 [B, T, D]): returns (dX float32 [B, T, D], dict of the parameter gradients
        dW1, db1, dW2, db2, dln1_g, dln1_b, dln2_g, dln2_b, each summed over the batch)."""
        B = X.shape[0]
        dX = torch.empty(X.shape, dtype=torch.float32, device=X.device) if dX is None else dX
        g, c = self._grad_tensors(X.device)
        _lib.rm_block_backward(self.ctx, layer, _ptr(X), _ptr(G), _ptr(dX), c, B, _stream())
        return dX, g

    def alloc_grads(self, device=None, flat: torch.Tensor | None = None) -> list:
        """Gradient buffers for every layer: a list of (dict of tensors, rm_layer_grads).
        With `flat` (float32, at least L * padded grad_numel() values, see flat_grad_numel)
        the tensors are views into it, layer after layer."""
        if flat is None:
            return [self._grad_tensors(device or self.device) for _ in range(self.L)]
        per = self.flat_grad_numel() // self.L
        return [self._grad_tensors(flat.device, flat[n * per:(n + 1) * per]) for n in range(self.L)]

    def flat_grad_numel(self) -> int:
        """Values of a flat buffer holding every layer's gradients (each piece padded to 4)."""
        T, D, F = self.T, self.D, self.k * self.D
        pieces = [T * D * F, T * F, T * F * D, T * D, D, D, D, D]
        return self.L * sum((n + 3) // 4 * 4 for n in pieces)

    def stack_backward(self, X0: torch.Tensor, dpooled: torch.Tensor, dX0: torch.Tensor | None = None,
                       grads: list | None = None):
        """Gradients of the stack and the mean pool for the loss whose gradient at the pooled
        output is dpooled (float32 [B, D]): returns (dX0, [grads of layer 0 .. L-1]).  grads:
        buffers from alloc_grads() to write into (new ones when None)."""
        B = X0.shape[0]
        dX0 = torch.empty(X0.shape, dtype=torch.float32, device=X0.device) if dX0 is None else dX0
        pairs = self.alloc_grads(X0.device) if grads is None else grads
        _lib.rm_stack_backward(self.ctx, _ptr(X0), _ptr(dpooled), _ptr(dX0), [c for _, c in pairs], B, _stream())
        return dX0, [g for g, _ in pairs]

    def stack_forward_train(self, X0: torch.Tensor, pooled: torch.Tensor | None = None) -> torch.Tensor:
        """Training forward of the stack: returns pooled (float32 [B, D]) and keeps every
        layer's activations for the next stack_backward_saved call."""
        B = X0.shape[0]
        pooled = torch.empty((B, self.D), dtype=torch.float32, device=X0.device) if pooled is None else pooled
        _lib.rm_stack_forward_train(self.ctx, _ptr(X0), _ptr(pooled), B, _stream())
        return pooled

    def stack_backward_saved(self, dpooled: torch.Tensor, dX0: torch.Tensor | None = None, grads: list | None = None):
        """Backward from the last stack_forward_train's activations for the pooled-output
        gradient dpooled: returns (dX0, [grads of layer 0 .. L-1])."""
        B = dpooled.shape[0]
        dX0 = torch.empty((B, self.T, self.D), dtype=torch.float32, device=dpooled.device) if dX0 is None else dX0
        pairs = self.alloc_grads(dpooled.device) if grads is None else grads
        _lib.rm_stack_backward_saved(self.ctx, _ptr(dpooled), _ptr(dX0), [c for _, c in pairs], B, _stream())
        return dX0, [g for g, _ in pairs]

    # -- tokenization, head and scoring ------------------------------------------------
    def set_unimixing(self, layer: int, WG: torch.Tensor, WB: torch.Tensor, tau: float = 1.0,
                      iters: int = 20) -> None:
        """UniMixing ("UniMixer", section 4.3) in place of layer ``layer``'s TokenMixing.
        WG [nb, nb] and WB [nb, bs, bs] are the raw float32 weights (nb * bs = T * D);
        the context keeps their Sinkhorn-Knopp constrained form (Eq. 15)."""
        WG = WG.to(device=self.device, dtype=torch.float32).contiguous()
        WB = WB.to(device=self.device, dtype=torch.float32).contiguous()
        bs = int(WB.shape[-1])
        _lib.rm_set_unimixing(self.ctx, layer, _ptr(WG), _ptr(WB), bs, float(tau), int(iters), _stream())
        self._um_bs = getattr(self, "_um_bs", {})
        self._um_bs[layer] = bs

    def unimixing_weights(self, layer: int) -> tuple[torch.Tensor, torch.Tensor]:
        """The constrained weights (WG [nb, nb], WB [nb, bs, bs], float32) of a UniMixing layer."""
        bs = self._um_bs[layer]
        nb = self.T * self.D // bs
        WG = torch.empty((nb, nb), dtype=torch.float32, device=self.device)
        WB = torch.empty((nb, bs, bs), dtype=torch.float32, device=self.device)
        _lib.rm_unimixing_weights(self.ctx, layer, _ptr(WG), _ptr(WB), _stream())
        return WG, WB

    def unimixing(self, layer: int, X: torch.Tensor, Y: torch.Tensor | None = None,
                  out_dtype: str | None = None) -> torch.Tensor:
        """Y = UniMixing(X) of layer ``layer``: X [B, T, D] in the context dtype; Y in the
        context dtype or float32 (out_dtype="f32")."""
        tdt, code = _out_dtype(out_dtype, self.tdtype)
        Y = torch.empty(X.shape, dtype=tdt, device=X.device) if Y is None else Y
        _lib.rm_unimixing(self.ctx, layer, _ptr(X), _ptr(Y), code, X.shape[0], _stream())
        return Y

    def set_tokenizer(self, W: torch.Tensor, bias: torch.Tensor) -> None:
        """W [T, d, D], bias [T, D] in the context dtype (token t's projection of its slice)."""
        self.tok_d = int(W.shape[1])
        torch.cuda.synchronize(self.device)
        _lib.rm_set_tokenizer(self.ctx, _ptr(W), _ptr(bias), self.tok_d)

    def tokenize(self, E: torch.Tensor, X0: torch.Tensor | None = None) -> torch.Tensor:
        """E [B, T d] -> X0 [B, T, D] (context dtype)."""
        B = E.shape[0]
        X0 = torch.empty((B, self.T, self.D), dtype=E.dtype, device=E.device) if X0 is None else X0
        _lib.rm_tokenize(self.ctx, _ptr(E), _ptr(X0), B, _stream())
        return X0

    def tokenize_backward(self, E: torch.Tensor, dX0: torch.Tensor, with_dE: bool = True) -> dict:
        """Gradients of tokenize(E) for dX0 [B, T, D] (float32): dW [T, d, D], db [T, D] and
        (with_dE) dE [B, T d], all float32."""
        B = E.shape[0]
        d = self.tok_d
        dW = torch.empty((self.T, d, self.D), dtype=torch.float32, device=E.device)
        db = torch.empty((self.T, self.D), dtype=torch.float32, device=E.device)
        dE = torch.empty((B, self.T * d), dtype=torch.float32, device=E.device) if with_dE else None
        _lib.rm_tokenize_backward(self.ctx, _ptr(E), _ptr(dX0), _ptr(dE), _ptr(dW), _ptr(db), B, _stream())
        return {"dE": dE, "dW": dW, "db": db}

    def score(self, E: torch.Tensor, head_w: torch.Tensor, head_b: float, p: torch.Tensor | None = None):
        """E [B, T d] -> p [B] = sigmoid(head(pool(stack(tokenize(E)))))."""
        B = E.shape[0]
        p = torch.empty(B, dtype=torch.float32, device=E.device) if p is None else p
        _lib.rm_score(self.ctx, _ptr(E), _ptr(head_w), float(head_b), _ptr(p), B, _stream())
        return p

    # -- status / profiling --------------------------------------------------------
    def sync_status(self) -> int:
        return _lib.rm_sync_status(self.ctx, _stream())

    def profile(self, on: bool = True) -> None:
        _lib.rm_profile_enable(self.ctx, on)

    def profile_read(self) -> dict:
        return _lib.rm_profile_read(self.ctx)

    def debug_wait_timeout(self, timeout_us: int) -> None:
        _lib.rm_debug_wait_timeout(self.ctx, timeout_us, _stream())


def token_mix(X: torch.Tensor, H: int | None = None) -> torch.Tensor:
    """Y[b, h, t q + r] = X[b, t, h q + r]; X [B, T, D] (bf16 or f32) on the GPU."""
    B, T, D = X.shape
    H = T if H is None else H
    Y = torch.empty((B, H, T * (D // H)), dtype=X.dtype, device=X.device)
    dt = _lib.RM_BF16 if X.dtype == torch.bfloat16 else _lib.RM_F32
    _lib.rm_token_mix(_ptr(X), _ptr(Y), B, T, D, H, dt, _stream())
    return Y


def debug_mix_residual(X: torch.Tensor, from_z: bool = False) -> torch.Tensor:
    """Test hook: y = Mix(X) + X from the fused mixing kernel's gather (float32,
    token-major [T, B, D]).  from_z=False: X bf16 [B, T, D]; from_z=True: X fp16
    token-major [T, B, D] and y the fp16 sum widened to float32."""
    if from_z:
        T, B, D = X.shape
    else:
        B, T, D = X.shape
    Y = torch.empty((T, B, D), dtype=torch.float32, device=X.device)
    _lib.rm_debug_mix_residual(_ptr(X), from_z, _ptr(Y), B, T, D, _stream())
    return Y


def head_forward(pooled: torch.Tensor, w: torch.Tensor, b: float, y: torch.Tensor | None = None,
                 mean_loss: bool = True) -> dict:
    """The prediction head on the GPU: returns p, and with labels y the per-sample loss
    and dpooled (the gradient of the batch-mean loss when mean_loss, else of the sum)."""
    B, D = pooled.shape
    p = torch.empty(B, dtype=torch.float32, device=pooled.device)
    out = {"p": p}
    loss = dp = None
    if y is not None:
        loss = torch.empty(B, dtype=torch.float32, device=pooled.device)
        dp = torch.empty_like(pooled)
        out.update(loss=loss, dpooled=dp)
    _lib.rm_head_forward(_ptr(pooled), _ptr(w), float(b), _ptr(y), _ptr(p), _ptr(loss), _ptr(dp), B, D, mean_loss,
                         _stream())
    return out
