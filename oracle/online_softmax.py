"""Tiled online-softmax recurrence in FP64 (NumPy), an independent restatement.

TEST INFRASTRUCTURE ONLY.  It exists to pin the untiled oracle in
``fa_oracle.c``: the pages state that the block-by-block recurrence reaches
exactly the one-shot softmax result, so the two must agree for any tile length.

The steps follow the "online softmax" rule of the "Flash Attention" history
page (section 1.2) and the derivation of the FlashAttention_01 page: keep a
running maximum m, a running denominator l and an unnormalised accumulator u;
for each key block with scores s, raise m to max(m, max s), multiply the old l
and u by exp(m_old - m_new), add exp(s - m_new) and exp(s - m_new) @ V, and
divide u by l once at the end.  Masked keys are dropped before the maximum.
An empty row keeps m = -inf, l = 0 and returns O = 0, LSE = -inf; the rescale
factor of a block whose maximum is still -inf is taken as 1 so that
-inf - (-inf) is never formed.

``merge_states`` applies the same rescale rule to whole per-chunk states; it
is the reduction that split-KV decode uses.
"""
from __future__ import annotations

import numpy as np


def tiled_row(q, K, V, tile: int, scale=None, visible=None, trace=None):
    """One query row q[d] against keys K[n,d], values V[n,d], keys taken in
    blocks of ``tile``.  Returns (m, l, u, O, LSE).  ``trace`` (a list) receives
    (m, l, u.copy()) after every block."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    n, d = K.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vis = np.ones(n, bool) if visible is None else np.asarray(visible, bool)
    m, l, u = -np.inf, 0.0, np.zeros(V.shape[1])
    for start in range(0, n, tile):
        sl = slice(start, start + tile)
        s = (K[sl] @ q) * scale
        keep = vis[sl]
        s = s[keep]
        Vb = V[sl][keep]
        if s.size:
            m_new = max(m, float(s.max()))
            a = 1.0 if m == -np.inf else float(np.exp(m - m_new))
            p = np.exp(s - m_new)
            u = a * u + p @ Vb
            l = a * l + float(p.sum())
            m = m_new
        if trace is not None:
            trace.append((m, l, u.copy()))
    if l == 0.0:
        return m, l, u, np.zeros_like(u), -np.inf
    return m, l, u, u / l, m + np.log(l)


def merge_states(states):
    """Combine per-chunk (LSE_s, O_s) pairs of one query row into (LSE, O).
    Chunks with LSE_s = -inf (no visible key) contribute nothing."""
    lses = np.array([s[0] for s in states], np.float64)
    outs = np.array([s[1] for s in states], np.float64)
    live = lses > -np.inf
    if not live.any():
        return -np.inf, np.zeros(outs.shape[1])
    mx = lses[live].max()
    w = np.where(live, np.exp(np.where(live, lses - mx, 0.0)), 0.0)
    tot = w.sum()
    return mx + np.log(tot), (w[:, None] * outs).sum(0) / tot
