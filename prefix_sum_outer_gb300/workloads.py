"""Seeded synthetic inputs for the causal product.

This module only draws inputs; it holds none of the causal-product
arithmetic, so both the CUDA path's tests and the oracle's tests may use
it.  Everything is drawn on the CPU from a seeded ``torch.Generator`` in a
fixed order (W first when a random-feature map is used, then x_q, x_k, v,
g), computed in float32 and rounded to the requested dtype with
round-to-nearest-even.

Feature maps (the positive features the linear-attention line of work feeds
to the causal product; triton-lang/triton issue #217 discusses the kernel
as a drop-in for Performer-style models):

* ``"elu"``:  phi(x) = elu(x) + 1 with alpha = 1 (x + 1 for x > 0, e^x
  otherwise), x ~ N(0, x_std^2) per element.
* ``"favor"``: phi(x) = exp(W x - |x|^2 / 2) / sqrt(D) with x ~ N(0, I_r)
  / r^(1/4) per token (r = 64 input features), W ~ N(0, I) of shape
  [D, r], one W shared by q, k and every (b, h); independent x for q and k.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    M: int
    dtype: str            # "f32" or "bf16"
    backward: bool
    seed: int
    feature: str = "elu"
    x_std: float = 1.0

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16}[self.dtype]

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.N


# The five synthetic workloads: sizes, dtypes, value distributions and seeds.
WORKLOADS = {
    "tiny_f32_fwd": Workload("tiny_f32_fwd", 1, 2, 64, 16, 16, "f32", False, 1),
    "mid_f32_fwd": Workload("mid_f32_fwd", 4, 8, 1024, 64, 64, "f32", False, 2),
    "bf16_b8h16_n4096_d64": Workload("bf16_b8h16_n4096_d64", 8, 16, 4096, 64, 64,
                                     "bf16", True, 3),
    "bf16_long_n32768_d128": Workload("bf16_long_n32768_d128", 2, 8, 32768, 128, 128,
                                      "bf16", True, 4, x_std=0.5),
    "bf16_favor_n8229_d256_m64": Workload("bf16_favor_n8229_d256_m64", 4, 8, 8229, 256, 64,
                                          "bf16", True, 5, feature="favor"),
}

FAVOR_INPUT_FEATURES = 64


def _elu_plus_one(x: torch.Tensor) -> torch.Tensor:
    return torch.where(x > 0, x + 1.0, torch.exp(x))


def _favor_draw(gen: torch.Generator, B: int, H: int, N: int, D: int):
    """The random part of the "favor" inputs, in draw order: W [D, r], then
    x_q and x_k [B, H, N, r] (float32)."""
    r = FAVOR_INPUT_FEATURES
    f32 = torch.float32
    W = torch.randn((D, r), generator=gen, dtype=f32)
    scale = 1.0 / (r ** 0.25)
    xq = torch.randn((B, H, N, r), generator=gen, dtype=f32) * scale
    xk = torch.randn((B, H, N, r), generator=gen, dtype=f32) * scale
    return W, xq, xk


def favor_raw_inputs(B: int, H: int, N: int, D: int, seed: int):
    """(W, x_q, x_k) behind make_inputs(..., feature="favor") with the same
    seed: the projection and the raw rows before the feature map."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    return _favor_draw(gen, B, H, N, D)


def make_inputs(B: int, H: int, N: int, D: int, M: int, dtype: torch.dtype, seed: int,
                feature: str = "elu", x_std: float = 1.0, backward: bool = True,
                v_std: float = 1.0):
    """Return CPU tensors (q, k, v, g) in ``dtype``; g is None if not backward."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    f32 = torch.float32
    if feature == "elu":
        xq = torch.randn((B, H, N, D), generator=gen, dtype=f32) * x_std
        xk = torch.randn((B, H, N, D), generator=gen, dtype=f32) * x_std
        q = _elu_plus_one(xq)
        k = _elu_plus_one(xk)
    elif feature == "favor":
        W, xq, xk = _favor_draw(gen, B, H, N, D)
        q = torch.exp(xq @ W.t() - 0.5 * (xq * xq).sum(-1, keepdim=True)) / math.sqrt(D)
        k = torch.exp(xk @ W.t() - 0.5 * (xk * xk).sum(-1, keepdim=True)) / math.sqrt(D)
    elif feature == "normal":
        q = torch.randn((B, H, N, D), generator=gen, dtype=f32) * x_std
        k = torch.randn((B, H, N, D), generator=gen, dtype=f32) * x_std
    else:
        raise ValueError(f"unknown feature map {feature!r}")
    v = torch.randn((B, H, N, M), generator=gen, dtype=f32) * v_std
    g = torch.randn((B, H, N, M), generator=gen, dtype=f32) if backward else None
    cast = lambda t: None if t is None else t.to(dtype).contiguous()
    return cast(q), cast(k), cast(v), cast(g)


def make_norm_inputs(B: int, H: int, N: int, D: int, dtype: torch.dtype, seed: int,
                     feature: str = "elu", x_std: float = 1.0):
    """Inputs of the normaliser: CPU tensors q, k [B,H,N,D] in ``dtype`` (the
    same draw as ``make_inputs`` with M = 1) and grad_z ~ N(0, 1), float32
    [B,H,N], from a second generator seeded ``seed + 7919``."""
    q, k, _, _ = make_inputs(B, H, N, D, 1, dtype, seed, feature=feature, x_std=x_std,
                             backward=False)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 7919)
    gz = torch.randn((B, H, N), generator=gen, dtype=torch.float32)
    return q, k, gz


def workload_inputs(w: Workload, N: Optional[int] = None, BH_limit: Optional[int] = None):
    """Inputs of a named workload; ``N``/``BH_limit`` shrink it for quick checks
    (the draw is then of the smaller shape, same seed and distributions)."""
    B, H = w.B, w.H
    if BH_limit is not None and B * H > BH_limit:
        B, H = 1, BH_limit
    return make_inputs(B, H, N if N is not None else w.N, w.D, w.M, w.torch_dtype, w.seed,
                       feature=w.feature, x_std=w.x_std, backward=w.backward)
