"""Shared helpers for the GPU-vs-oracle parity tests (test infrastructure).

Tolerances (the stated acceptance rule, applied per tensor):
  O:           max |gpu - oracle| <= 2e-2
  LSE:         max |gpu - oracle| <= 1e-3 on finite entries; -inf must match exactly
  dQ, dK, dV:  max |gpu - oracle| <= 5e-2 * max |oracle|   (per tensor)
Finiteness is checked first (FlashAttention_01 page, mixed-precision
acceptance: finiteness, then absolute/relative tolerance).
"""
from __future__ import annotations

import numpy as np
import torch

O_TOL = 2e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 5e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(gpu: np.ndarray, ref: np.ndarray, what="O"):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values from the GPU"
    err = float(np.abs(gpu - ref).max()) if gpu.size else 0.0
    assert err <= O_TOL, f"{what}: max abs error {err:.3e} > {O_TOL}"
    return err


def check_lse(gpu: np.ndarray, ref: np.ndarray, what="LSE"):
    assert not np.any(np.isnan(gpu)), f"{what}: NaN from the GPU"
    dead = ref == -np.inf
    assert np.array_equal(gpu == -np.inf, dead), (
        f"{what}: -inf pattern differs ({int((gpu == -np.inf).sum())} vs {int(dead.sum())})")
    live = ~dead
    err = float(np.abs(gpu[live] - ref[live]).max()) if live.any() else 0.0
    assert err <= LSE_TOL, f"{what}: max abs error {err:.3e} > {LSE_TOL}"
    return err


def check_grad(gpu: np.ndarray, ref: np.ndarray, what):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values from the GPU"
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(gpu - ref).max()) if gpu.size else 0.0
    bound = GRAD_REL_TOL * scale if scale > 0 else 1e-6
    assert err <= bound, f"{what}: max abs error {err:.3e} > {bound:.3e} (max|ref| {scale:.3e})"
    return err / scale if scale > 0 else err


def sample_rows(B, H, S, n, seed, must=()):
    """Flat row ids (b*H + h)*S + i: `must` rows plus n seeded random ones."""
    g = np.random.default_rng(seed)
    rows = set(int(r) for r in must)
    total = B * H * S
    rows.update(int(x) for x in g.integers(0, total, size=n))
    return np.array(sorted(rows), dtype=np.int64)
