"""Shared helpers for the GPU parity tests: tolerances and comparisons
against the fp64 oracle.

Tolerances (the stated bar for this path):
  * bf16 outputs: |gpu - bf16(ref)| <= 2e-2 + 1.6e-2 * |bf16(ref)| elementwise
    (max abs 2e-2, max rel 1.6e-2: about two bf16 ulps).
  * fp32 results (dgamma, dbeta, mean, rstd): relative 1e-3, read elementwise
    as |gpu - ref| <= 1e-3 * max(|ref|, 1e-2 * max|ref|) -- a plain relative
    bound is ill-conditioned where a column sum nearly cancels -- and
    normwise as max|gpu - ref| / max|ref| <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_ATOL = 2e-2
BF16_RTOL = 1.6e-2
F32_RTOL = 1e-3


def host_f64(t: torch.Tensor) -> np.ndarray:
    """A device or host tensor as float64 numpy (bf16 widened exactly)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return oracle.widen(t)
    return t.double().numpy()


def check_bf16(gpu: torch.Tensor, ref: np.ndarray, name: str) -> dict:
    g = host_f64(gpu).reshape(ref.shape)
    r = oracle.bf16_value(ref)
    err = np.abs(g - r)
    bound = BF16_ATOL + BF16_RTOL * np.abs(r)
    bad = ~(err <= bound)  # NaN counts as bad
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "max_rel": float((err / np.maximum(np.abs(r), 1e-30)).max()) if err.size else 0.0}
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                             f"first {idx.tolist()} gpu={g[bad][:5]} ref={r[bad][:5]} {stats}")
    return stats


def check_f32(gpu: torch.Tensor, ref: np.ndarray, name: str, rtol: float = F32_RTOL) -> dict:
    g = host_f64(gpu).reshape(ref.shape)
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = np.abs(g - ref)
    bound = rtol * np.maximum(np.abs(ref), 1e-2 * scale)
    bad = ~(err <= bound)
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "normwise": float(err.max() / scale) if scale > 0 else float(err.max() if err.size else 0)}
    if bad.any():
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside rel {rtol}; {stats}")
    assert stats["normwise"] <= rtol, (name, stats)
    return stats


def ulp_diff_bf16(a: torch.Tensor, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between a bf16 tensor and bf16 bit patterns
    (same sign assumed for nonzero values; used for the residual output)."""
    ab = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).astype(np.int64)
    bb = b_bits.astype(np.int64)

    def ordered(x):
        # map sign-magnitude bit patterns onto a monotone integer line
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(ab) - ordered(bb.reshape(ab.shape)))
