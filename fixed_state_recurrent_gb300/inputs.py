"""Seeded synthetic inputs for the linear-attention and delta-rule workloads.

This module is the only code that the CUDA path and the fp64 oracle's tests
both use.  It holds no arithmetic of the method: it draws Gaussian numbers from
a seeded torch generator, rounds them to the storage dtype, and (for the delta
workload) applies the input preparation the workload names -- unit-normalised
keys and sigmoid step sizes.

Recipe (every workload): draw fp32 N(0, 1) with ``torch.Generator`` seeded by
``seed``, in the order q, k, v (then beta), scale if the workload says so,
then round to the storage dtype with round-to-nearest-even (``Tensor.to``).
The rounded values are the inputs of both sides; the oracle receives them
widened to float64.

Shapes: tokens [B, H, N, d] contiguous (d fastest); beta [B, H, N].
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

__all__ = [
    "Workload", "WORKLOADS", "gaussian", "la_inputs", "delta_inputs",
    "decode_step_inputs",
]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, storage dtype and generator seed."""
    name: str
    B: int
    H: int
    N: int
    dk: int
    dv: int
    dtype: torch.dtype
    seed: int
    scale: float = 1.0
    steps: int = 0  # decode only: number of consecutive decode steps

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.N


# The five workloads of the hot path.  "pr1" is the small fp32 case, "prefill"
# and "long" the bf16 prefill cases, "decode" 100 steps after a 1024-token
# prefix (N is the prefix length), "delta" the delta-rule memory;
# "prefill128" is the prefill case at dk = dv = 128.
WORKLOADS = {
    "pr1": Workload("pr1", 1, 1, 256, 64, 64, torch.float32, 7),
    "prefill": Workload("prefill", 4, 8, 4096, 64, 64, torch.bfloat16, 1),
    "long": Workload("long", 1, 16, 65536, 64, 64, torch.bfloat16, 2, scale=0.5),
    "decode": Workload("decode", 256, 32, 1024, 128, 128, torch.bfloat16, 3,
                       steps=100),
    "delta": Workload("delta", 8, 16, 8192, 128, 128, torch.bfloat16, 4),
    # the prefill operator at the wider head size dk = dv = 128
    "prefill128": Workload("prefill128", 4, 8, 4096, 128, 128, torch.bfloat16, 5),
}


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(shape, gen: torch.Generator, dtype=torch.float32, scale=1.0,
             device="cpu") -> torch.Tensor:
    """fp32 N(0, 1) draw, optionally scaled in fp32, rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32,
                    device=device)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def la_inputs(B, H, N, dk, dv, dtype=torch.bfloat16, seed=0, scale=1.0,
              device="cpu"):
    """q, k, v for the linear-attention prefill, drawn in that order."""
    g = _generator(seed, device)
    q = gaussian((B, H, N, dk), g, dtype, scale, device)
    k = gaussian((B, H, N, dk), g, dtype, scale, device)
    v = gaussian((B, H, N, dv), g, dtype, scale, device)
    return q, k, v


def decode_step_inputs(B, H, dk, dv, steps, dtype=torch.bfloat16, seed=0,
                       device="cpu"):
    """q, k, v for ``steps`` decode steps: [steps, B, H, d] each.  Drawn after
    the prefix with a separate stream (seed + 1000)."""
    g = _generator(seed + 1000, device)
    q = gaussian((steps, B, H, dk), g, dtype, 1.0, device)
    k = gaussian((steps, B, H, dk), g, dtype, 1.0, device)
    v = gaussian((steps, B, H, dv), g, dtype, 1.0, device)
    return q, k, v


def delta_inputs(B, H, N, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu"):
    """k, v, beta for the delta-rule memory.

    Keys: N(0,1) in fp32, divided by their per-token L2 norm in fp32, then
    rounded to ``dtype`` (so they are unit length only up to that rounding).
    Values: N(0,1) rounded to ``dtype``.  beta: sigmoid of N(0,1), fp32."""
    g = _generator(seed, device)
    k = torch.randn((B, H, N, dk), generator=g, dtype=torch.float32,
                    device=device)
    k = k / k.norm(dim=-1, keepdim=True)
    k = k.to(dtype)
    v = gaussian((B, H, N, dv), g, dtype, 1.0, device)
    beta = torch.sigmoid(torch.randn((B, H, N), generator=g,
                                     dtype=torch.float32, device=device))
    return k, v, beta


def workload_inputs(w: Workload, device="cpu"):
    """The inputs of a named workload (prefix tokens for "decode")."""
    if w.name == "delta":
        return delta_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed, device)
    return la_inputs(w.B, w.H, w.N, w.dk, w.dv, w.dtype, w.seed, w.scale,
                     device)
