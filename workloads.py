"""Seeded synthetic inputs and the workload table.

This module is shared by the CUDA-path tests, the benchmark and the oracle
tests.  It draws random numbers and names shapes; it contains none of the
normalization arithmetic.

Recipe: one ``torch.Generator`` per workload, seeded (0 by default), values
drawn in fp32 with ``randn`` as ``mean + std * N(0, 1)`` and cast to bf16
(round to nearest even).  Draw order: x, then residual (or dy), then the
weight (or gamma), then beta.  Shapes are row-major ``[rows, hidden]``;
parameters are ``[hidden]``.  The small-batch sweep takes the first ``rows``
rows of a 128-row draw so that its cases nest.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Hidden sizes the library instantiates at compile time.
HIDDEN_SET = (1024, 2048, 4096, 5120, 8192, 12288)


def _draw(gen: torch.Generator, shape, mean: float, std: float, device) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fused_inputs(rows: int, hidden: int, seed: int = 0, residual_scale: float = 1.0,
                 device="cpu", draw_rows: int | None = None):
    """x ~ N(0,1), residual ~ residual_scale * N(0,1), weight ~ N(1, 0.1), all bf16.

    ``draw_rows`` (>= rows) draws that many rows and keeps the first ``rows``."""
    n = max(rows, draw_rows or rows)
    g = _gen(seed, device)
    x = _draw(g, (n, hidden), 0.0, 1.0, device)[:rows].contiguous()
    res = _draw(g, (n, hidden), 0.0, residual_scale, device)[:rows].contiguous()
    w = _draw(g, (hidden,), 1.0, 0.1, device)
    return x, res, w


def rms_inputs(rows: int, hidden: int, seed: int = 0, device="cpu"):
    """x ~ N(0,1), weight ~ N(1, 0.1), bf16."""
    g = _gen(seed, device)
    x = _draw(g, (rows, hidden), 0.0, 1.0, device)
    w = _draw(g, (hidden,), 1.0, 0.1, device)
    return x, w


def layernorm_fwd_inputs(rows: int, hidden: int, seed: int = 0, device="cpu",
                         x_mean: float = 0.5, x_std: float = 2.0):
    """x ~ N(0.5, 2), gamma ~ N(1, 0.1), beta ~ N(0, 0.1), bf16."""
    g = _gen(seed, device)
    x = _draw(g, (rows, hidden), x_mean, x_std, device)
    gamma = _draw(g, (hidden,), 1.0, 0.1, device)
    beta = _draw(g, (hidden,), 0.0, 0.1, device)
    return x, gamma, beta


def layernorm_bwd_inputs(rows: int, hidden: int, seed: int = 0, device="cpu"):
    """x ~ N(0,1), dy ~ N(0,1), gamma ~ N(1, 0.1), bf16.

    The saved mean/rstd are not drawn: they come from a forward pass."""
    g = _gen(seed, device)
    x = _draw(g, (rows, hidden), 0.0, 1.0, device)
    dy = _draw(g, (rows, hidden), 0.0, 1.0, device)
    gamma = _draw(g, (hidden,), 1.0, 0.1, device)
    return x, dy, gamma


def rms_bwd_inputs(rows: int, hidden: int, seed: int = 0, device="cpu"):
    """x ~ N(0,1), dy ~ N(0,1), weight ~ N(1, 0.1), bf16."""
    return layernorm_bwd_inputs(rows, hidden, seed, device)


def fused_bwd_inputs(rows: int, hidden: int, seed: int = 0, device="cpu"):
    """Fused add + RMSNorm backward: the saved residual stream s ~ N(0, 4.12)
    (the spread of x + 4 N(0,1)), dy ~ N(0,1), dres ~ N(0,1), weight ~ N(1, 0.1),
    all bf16.  Returns (s, weight, dy, dres)."""
    g = _gen(seed, device)
    s = _draw(g, (rows, hidden), 0.0, 4.12, device)
    dy = _draw(g, (rows, hidden), 0.0, 1.0, device)
    dres = _draw(g, (rows, hidden), 0.0, 1.0, device)
    w = _draw(g, (hidden,), 1.0, 0.1, device)
    return s, w, dy, dres


def outer_inputs(rows: int, hidden: int, seed: int = 0, device="cpu"):
    """Per-column normalization inputs: x ~ N(0.5, 2), dy ~ N(0, 1),
    gamma ~ N(1, 0.1), beta ~ N(0, 0.1), bf16."""
    g = _gen(seed, device)
    x = _draw(g, (rows, hidden), 0.5, 2.0, device)
    dy = _draw(g, (rows, hidden), 0.0, 1.0, device)
    gamma = _draw(g, (hidden,), 1.0, 0.1, device)
    beta = _draw(g, (hidden,), 0.0, 0.1, device)
    return x, dy, gamma, beta


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # fused_add_rmsnorm | rmsnorm_fwd | layernorm_fwd | layernorm_bwd
    rows: tuple
    hidden: tuple
    eps: float
    residual_scale: float = 1.0
    draw_rows: int | None = None
    notes: str = field(default="")


# The workloads, by what they are.
FUSED_DECODE_16 = Workload("fused add+RMSNorm decode, 16 rows x 4096", "fused_add_rmsnorm",
                           (16,), (4096,), 1e-6)
FUSED_SMALL_BATCH = Workload("fused add+RMSNorm small-batch sweep", "fused_add_rmsnorm",
                             (1, 2, 4, 8, 32, 128), (4096, 8192), 1e-6, draw_rows=128)
FUSED_PREFILL = Workload("fused add+RMSNorm LLM prefill", "fused_add_rmsnorm",
                         (4096, 16384, 65536), (2048, 4096, 5120, 8192), 1e-5,
                         residual_scale=4.0)
LAYERNORM_FWD = Workload("LayerNorm forward", "layernorm_fwd", (16384,), (1024, 4096, 12288), 1e-5)
LAYERNORM_BWD = Workload("LayerNorm backward", "layernorm_bwd", (16384,), (1024, 4096, 8192), 1e-5)

ALL = (FUSED_DECODE_16, FUSED_SMALL_BATCH, FUSED_PREFILL, LAYERNORM_FWD, LAYERNORM_BWD)
