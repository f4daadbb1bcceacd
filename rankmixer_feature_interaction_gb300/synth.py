"""Seeded synthetic inputs and parameters for the RankMixer workloads.

Holds none of the method's arithmetic: it only draws random tensors with the
shapes and distributions of the workloads, so that the CUDA library and the
CPU oracle are fed identical values.

Distributions (second argument of N(0, x) read as the variance):
  X ~ N(0, 1); W1 ~ N(0, 1/D); W2 ~ N(0, 1/(kD)); biases ~ N(0, 0.01);
  LN gamma = 1 + N(0, 0.1), LN beta ~ N(0, 0.1);
  router Wg ~ N(0, 1/D); expert weights ~ N(0, 1/fan_in); expert biases ~ N(0, 0.01).
The router bias is set so that about 2 of E = 8 experts are open per token:
the router pre-activation s.Wg_{:,e} of an LN output row s is close to
N(0, E|s|^2 / D) with E|s|^2 / D ~= E[gamma^2] + E[beta^2] = 1.2 under the
distributions above, so bg = -z_{1-p} * sqrt(1.2) opens each expert with
probability p = active / E.

Shapes are those the RankMixer paper reports for its final models (RankMixer-
100M: T=16, D=768, L=2; RankMixer-1B: T=32, D=1536, L=2), with k = 4, H = T.
These synthetic tensors stand in for the paper's production data, which is
not available.
"""
from __future__ import annotations

import math
from statistics import NormalDist

import torch

CONFIGS = {
    # name: B, T, D, k, L, dtype (+ experts)
    "tiny_fp32": dict(B=64, T=4, D=8, k=2, L=1, dtype="f32"),
    "rankmixer_100m": dict(B=2048, T=16, D=768, k=4, L=2, dtype="bf16"),
    "rankmixer_1b": dict(B=4096, T=32, D=1536, k=4, L=2, dtype="bf16"),
    "serving_sweep_1b": dict(B=(1, 8, 64, 256, 1024, 8192), T=32, D=1536, k=4, L=2, dtype="bf16"),
    "moe_1b": dict(B=4096, T=32, D=1536, k=4, L=1, dtype="bf16", E=8, Fe=3072, active=2.0),
}

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}
GAMMA_VAR = 0.1
BETA_VAR = 0.1
BIAS_VAR = 0.01


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std: float, g: torch.Generator, device, dtype, mean: float = 0.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def make_input(B: int, T: int, D: int, seed: int, dtype: str = "bf16", device="cpu") -> torch.Tensor:
    """X0 ~ N(0, 1), [B, T, D]."""
    return _normal((B, T, D), 1.0, _gen(seed, device), device, TORCH_DTYPE[dtype])


def make_output_grad(shape: tuple, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """A seeded loss gradient at a block or pooled output: scale * N(0, 1), float32."""
    return _normal(tuple(shape), scale, _gen(seed, device), device, torch.float32)


SHARD_BLOCK = 64


def make_input_shard(global_B: int, start: int, stop: int, T: int, D: int, seed: int, dtype: str = "bf16",
                     device="cpu") -> torch.Tensor:
    """Samples [start, stop) of a seeded global batch of `global_B` inputs X0 ~ N(0, 1).

    The global batch is drawn in blocks of SHARD_BLOCK samples, block j from its
    own generator (seed, j), so a rank can draw its own shard without drawing the
    rest, and the shards of any split concatenate to the same global batch."""
    if not 0 <= start <= stop <= global_B:
        raise ValueError(f"shard [{start}, {stop}) outside a batch of {global_B}")
    parts = []
    for j in range(start // SHARD_BLOCK, (stop + SHARD_BLOCK - 1) // SHARD_BLOCK):
        b0 = j * SHARD_BLOCK
        nb = min(SHARD_BLOCK, global_B - b0)
        blk = _normal((nb, T, D), 1.0, _gen(seed * 1_000_003 + j, device), device, TORCH_DTYPE[dtype])
        parts.append(blk[max(start - b0, 0):min(stop - b0, nb)])
    if not parts:
        return torch.empty((0, T, D), dtype=TORCH_DTYPE[dtype], device=device)
    return torch.cat(parts, 0)


def router_bias(active: float, E: int) -> float:
    """Router bias opening each expert with probability active / E (see the module docstring)."""
    p = active / E
    return -NormalDist().inv_cdf(1.0 - p) * math.sqrt(1.0 + GAMMA_VAR + BETA_VAR)


def make_layer(T: int, D: int, k: int, seed: int, dtype: str = "bf16", device="cpu", E: int = 0, Fe: int = 0,
               active: float = 2.0) -> dict:
    """One layer's parameters in the pages' layout (row-vector convention)."""
    td = TORCH_DTYPE[dtype]
    g = _gen(seed, device)
    F = k * D
    p = {
        "W1": _normal((T, D, F), 1.0 / math.sqrt(D), g, device, td),
        "b1": _normal((T, F), math.sqrt(BIAS_VAR), g, device, td),
        "W2": _normal((T, F, D), 1.0 / math.sqrt(F), g, device, td),
        "b2": _normal((T, D), math.sqrt(BIAS_VAR), g, device, td),
        "ln1_g": _normal((D,), math.sqrt(GAMMA_VAR), g, device, td, mean=1.0),
        "ln1_b": _normal((D,), math.sqrt(BETA_VAR), g, device, td),
        "ln2_g": _normal((D,), math.sqrt(GAMMA_VAR), g, device, td, mean=1.0),
        "ln2_b": _normal((D,), math.sqrt(BETA_VAR), g, device, td),
    }
    if E > 0:
        p.update(make_experts(T, D, E, Fe, seed + 7919, dtype, device, active))
    return p


def make_experts(T: int, D: int, E: int, Fe: int, seed: int, dtype: str = "bf16", device="cpu",
                 active: float = 2.0) -> dict:
    td = TORCH_DTYPE[dtype]
    g = _gen(seed, device)
    return {
        "Wg": _normal((T, D, E), 1.0 / math.sqrt(D), g, device, td),
        "bg": torch.full((T, E), router_bias(active, E), device=device, dtype=torch.float32).to(td),
        "eW1": _normal((T, E, D, Fe), 1.0 / math.sqrt(D), g, device, td),
        "eb1": _normal((T, E, Fe), math.sqrt(BIAS_VAR), g, device, td),
        "eW2": _normal((T, E, Fe, D), 1.0 / math.sqrt(Fe), g, device, td),
        "eb2": _normal((T, E, D), math.sqrt(BIAS_VAR), g, device, td),
    }


def make_train_router(T: int, D: int, E: int, seed: int, dtype: str = "bf16", device="cpu",
                      active: float = 6.0) -> dict:
    """A second (training) router for the dense-training / sparse-inference MoE: Wg_train
    [T, D, E] ~ N(0, 1/D), its bias set so that about `active` of E experts open."""
    td = TORCH_DTYPE[dtype]
    g = _gen(seed, device)
    return {"Wg_train": _normal((T, D, E), 1.0 / math.sqrt(D), g, device, td),
            "bg_train": torch.full((T, E), router_bias(active, E), device=device, dtype=torch.float32).to(td)}


def make_stack(T: int, D: int, k: int, L: int, seed: int, dtype: str = "bf16", device="cpu", E: int = 0,
               Fe: int = 0, active: float = 2.0) -> list:
    return [make_layer(T, D, k, seed * 131 + n, dtype, device, E, Fe, active) for n in range(L)]


def make_unimix_weights(T: int, D: int, bs: int, seed: int, device="cpu") -> tuple:
    """Raw (unconstrained) UniMixing weights for block size bs: WG [nb, nb] and
    WB [nb, bs, bs], nb = T D / bs, every entry N(0, 1), float32."""
    nb = T * D // bs
    g = _gen(seed, device)
    WG = _normal((nb, nb), 1.0, g, device, torch.float32)
    WB = _normal((nb, bs, bs), 1.0, g, device, torch.float32)
    return WG, WB


def to_f64(p):
    """Tensor or dict/list of tensors -> numpy float64 (values exactly as rounded to their dtype)."""
    if isinstance(p, dict):
        return {k: to_f64(v) for k, v in p.items()}
    if isinstance(p, (list, tuple)):
        return [to_f64(v) for v in p]
    return p.detach().to("cpu", torch.float64).numpy()
