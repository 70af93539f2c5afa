"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers and lays them out; it holds none of the layer's
arithmetic. Both the CUDA path and the fp64 oracle take their inputs from here.

Draw order for one workload, all from one CPU ``torch.Generator`` seeded with the
workload's seed:

1. ``x``   [T, d]      ~ N(0, 1), rounded to bf16 (round to nearest even)
2. ``W_r`` [E, d]      ~ N(0, 1/d), fp32
3. ``b``   [E]         ~ U[-0.05, 0.05], fp32 (drawn in both router modes, used by sigmoid)
4. ``W_g`` [E, f, d]   ~ N(0, 1/d), then ``W_u`` [E, f, d] ~ N(0, 1/d), then
   ``W_d`` [E, d, f]   ~ N(0, 1/f), each rounded to bf16
5. shared expert, when present: ``Ws_g`` [f_s, d], ``Ws_u`` [f_s, d] ~ N(0, 1/d),
   ``Ws_d`` [d, f_s] ~ N(0, 1/f_s), bf16
6. ``dY``  [T, d]      ~ N(0, 1), bf16 (upstream gradient of the layer output)

Weights use the ``nn.Linear`` out x in convention: a row of ``W_g[e]`` maps d_model to one
hidden unit.

Skewed workloads (``zipf=True``) rescale rows of ``W_r`` after all of the above: a
permutation drawn last from the same generator assigns popularity ranks, rank r (1-based) of the live experts gets row scale
``ZIPF_SCALE0 * r**-ZIPF_ALPHA``, and ``ZIPF_DEAD`` experts get an all-zero row. A zero row
gives that expert a fixed logit of 0 for every token, so it is outranked by the live
experts' tails and receives no tokens. The rescaling needs no routing computation.
"""
from __future__ import annotations

import torch

from .configs import MoEConfig

ZIPF_DEAD = 12
ZIPF_SCALE0 = 2.0
ZIPF_ALPHA = 0.45


def _normal(g: torch.Generator, shape, std: float) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def zipf_row_scales(cfg: MoEConfig, g: torch.Generator) -> torch.Tensor:
    """Per-expert multipliers for the rows of W_r in skewed workloads."""
    perm = torch.randperm(cfg.E, generator=g)
    scales = torch.zeros(cfg.E, dtype=torch.float32)
    live = cfg.E - ZIPF_DEAD
    for r in range(live):
        scales[perm[r]] = ZIPF_SCALE0 * float(r + 1) ** (-ZIPF_ALPHA)
    return scales


def make_inputs(cfg: MoEConfig, with_grad_input: bool | None = None) -> dict:
    """All host tensors of one workload, drawn in the documented order."""
    g = torch.Generator().manual_seed(cfg.seed)
    T, d, E, f, fs = cfg.T, cfg.d, cfg.E, cfg.f, cfg.f_shared
    out = {}
    out["x"] = _normal(g, (T, d), 1.0).to(torch.bfloat16)
    W_r = _normal(g, (E, d), d ** -0.5)
    out["b"] = torch.rand((E,), generator=g, dtype=torch.float32) * 0.1 - 0.05
    out["W_g"] = _normal(g, (E, f, d), d ** -0.5).to(torch.bfloat16)
    out["W_u"] = _normal(g, (E, f, d), d ** -0.5).to(torch.bfloat16)
    out["W_d"] = _normal(g, (E, d, f), f ** -0.5).to(torch.bfloat16)
    if fs > 0:
        out["Ws_g"] = _normal(g, (fs, d), d ** -0.5).to(torch.bfloat16)
        out["Ws_u"] = _normal(g, (fs, d), d ** -0.5).to(torch.bfloat16)
        out["Ws_d"] = _normal(g, (d, fs), fs ** -0.5).to(torch.bfloat16)
    want_dy = cfg.backward if with_grad_input is None else with_grad_input
    if want_dy:
        out["dY"] = _normal(g, (T, d), 1.0).to(torch.bfloat16)
    if cfg.zipf:
        W_r = W_r * zipf_row_scales(cfg, g)[:, None]
    out["W_r"] = W_r.contiguous()
    return out


def make_upstream_gate_grad(T: int, k: int, seed: int) -> torch.Tensor:
    """A synthetic gradient with respect to the gates, [T, k] fp32 ~ N(0, 1).

    Used to exercise the router backward on its own at sizes where the full layer's
    gate gradient is too costly for the CPU oracle."""
    g = torch.Generator().manual_seed(seed + 7919)
    return torch.randn((T, k), generator=g, dtype=torch.float32)
