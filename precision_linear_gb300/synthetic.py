"""Seeded synthetic workloads: shapes and draws only, none of the method's arithmetic.

This module is the one thing the CUDA path and the CPU oracle share: both are fed
the tensors drawn here.  Every draw is a fixed torch generator stream, so a seed
names a tensor exactly on a given device type.

Shapes follow Qwen2.5-7B and Qwen2.5-32B decoder layers (the model family the
QeRL pages train); value distributions follow the workloads the pages describe:
backbone weights N(0, 0.02^2) (optionally 0.1% outliers x20), BF16 activations
N(0, 1), RMSNorm scales 1 + N(0, 0.1^2), AQN noise N(0, sigma^2), LoRA A and B
N(0, 0.02^2), adapter scale lambda = 2.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

EPS = 1e-6  # RMSNorm delta used by every workload


@dataclass(frozen=True)
class Proj:
    name: str
    d_i: int
    d_o: int
    norm: str | None  # which RMSNorm feeds it ("attn", "ffn") or None (plain input)


def qwen_layer(hidden: int, inter: int, n_q: int, n_kv: int, head_dim: int) -> tuple[Proj, ...]:
    q, kv = n_q * head_dim, n_kv * head_dim
    return (
        Proj("q", hidden, q, "attn"),
        Proj("k", hidden, kv, "attn"),
        Proj("v", hidden, kv, "attn"),
        Proj("o", q, hidden, None),
        Proj("gate", hidden, inter, "ffn"),
        Proj("up", hidden, inter, "ffn"),
        Proj("down", inter, hidden, None),
    )


QWEN7B_LAYER = qwen_layer(3584, 18944, 28, 4, 128)
QWEN32B_LAYER = qwen_layer(5120, 27648, 64, 8, 128)


@dataclass(frozen=True)
class Workload:
    name: str
    projs: tuple[Proj, ...]
    Ms: tuple[int, ...]
    r: int
    lam: float
    sigma: float
    seed: int
    outlier_frac: float = 0.0
    layers: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", (Proj("proj", 256, 256, "attn"),), (4,), 8, 2.0, 1e-2, 0,
                     notes="d_i=d_o=256, M=4, r=8"),
    "decode_proj_7b": Workload("decode_proj_7b", (Proj("proj", 3584, 3584, "attn"),),
                               (1, 8, 16, 32, 64), 32, 2.0, 1e-2, 2, outlier_frac=1e-3,
                               notes="7B-shaped 3584x3584 projection, M sweep"),
    "layer_7b": Workload("layer_7b", QWEN7B_LAYER, (8, 32, 64), 32, 2.0, 1e-2, 3,
                         notes="Qwen2.5-7B-shaped decoder-layer projection set"),
    "prefill_7b": Workload("prefill_7b", QWEN7B_LAYER, (4096,), 32, 2.0, 1e-2, 4,
                           notes="same set at M=4096 (8 responses x 512 tokens)"),
    "stack_32b": Workload("stack_32b", QWEN32B_LAYER, (1, 16, 64), 32, 2.0, 5e-3, 5,
                          layers=64, notes="Qwen2.5-32B-shaped 64-layer decode stack"),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(stream))
    return g


def weight(d_o: int, d_i: int, seed: int, outlier_frac: float = 0.0,
           device="cpu") -> torch.Tensor:
    """Backbone weight [d_o, d_i] as BF16: N(0, 0.02^2), a Bernoulli(outlier_frac)
    subset multiplied by 20."""
    w = torch.randn(d_o, d_i, generator=_gen(seed, 1, device), device=device) * 0.02
    if outlier_frac > 0:
        mask = torch.rand(d_o, d_i, generator=_gen(seed, 2, device), device=device) < outlier_frac
        w = torch.where(mask, w * 20.0, w)
    return w.to(torch.bfloat16)


def activations(M: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    return torch.randn(M, d, generator=_gen(seed, 3, device), device=device).to(torch.bfloat16)


def norm_scale(d: int, seed: int, device="cpu") -> torch.Tensor:
    return 1.0 + 0.1 * torch.randn(d, generator=_gen(seed, 4, device), device=device)


def noise(d: int, sigma: float, seed: int, device="cpu") -> torch.Tensor:
    return sigma * torch.randn(d, generator=_gen(seed, 5, device), device=device)


def lora(d_o: int, d_i: int, r: int, seed: int, device="cpu"):
    A = (0.02 * torch.randn(r, d_i, generator=_gen(seed, 6, device), device=device)).to(torch.bfloat16)
    B = (0.02 * torch.randn(d_o, r, generator=_gen(seed, 7, device), device=device)).to(torch.bfloat16)
    return A, B


def projection_case(d_o: int, d_i: int, M: int, r: int, sigma: float, seed: int,
                    outlier_frac: float = 0.0, device="cpu") -> dict:
    """Every input of one projection call, drawn from `seed`."""
    A, B = lora(d_o, d_i, r, seed, device)
    return dict(
        W=weight(d_o, d_i, seed, outlier_frac, device),
        x=activations(M, d_i, seed, device),
        w_norm=norm_scale(d_i, seed, device),
        z=noise(d_i, sigma, seed, device),
        A=A, B=B,
    )


def proj_seed(wl: Workload, layer: int, proj_index: int) -> int:
    """Seed of one projection of one layer of a workload."""
    base = 5000 + layer if wl.layers > 1 else wl.seed
    return base * 16 + proj_index


NORMS = ("attn", "ffn")


def norm_seed(wl: Workload, layer: int, norm: str) -> int:
    """Seed of the input shared by the projections that read one RMSNorm of a layer."""
    base = 5000 + layer if wl.layers > 1 else wl.seed
    return base * 16 + 8 + NORMS.index(norm)


def layer_case(wl: Workload, layer: int, M: int, device="cpu") -> dict:
    """Every input of one decoder layer's projections, wired as in the layer.

    The projections behind one RMSNorm read the same tensors: q, k and v take one
    (x, w_norm, z) -- the attention norm's input, scale and noise state -- and gate and
    up take the FFN norm's; o and down take plain BF16 inputs of their own (the attention
    output and the SwiGLU product, outside this path, replaced by seeded draws).  Each
    projection has its own weight and adapter.  Returns {name: case dict}; the shared
    entries are the same tensor objects."""
    shared = {}
    for nm in NORMS:
        p0 = next(p for p in wl.projs if p.norm == nm)
        sd = norm_seed(wl, layer, nm)
        shared[nm] = dict(x=activations(M, p0.d_i, sd, device), w_norm=norm_scale(p0.d_i, sd, device),
                          z=noise(p0.d_i, wl.sigma, sd, device))
    out = {}
    for i, p in enumerate(wl.projs):
        sd = proj_seed(wl, layer, i)
        A, B = lora(p.d_o, p.d_i, wl.r, sd, device)
        c = dict(W=weight(p.d_o, p.d_i, sd, wl.outlier_frac, device), A=A, B=B)
        if p.norm is not None:
            c.update(shared[p.norm])
        else:
            c.update(x=activations(M, p.d_i, sd, device), w_norm=None, z=None)
        out[p.name] = c
    return out
