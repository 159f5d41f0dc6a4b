"""Pins of the FP64 oracle against what the pages and the mathematics fix.

Each test names the passage it follows.  None of these values comes from the
CUDA path: they are the pages' printed numbers, closed forms, brute force or a
library routine (torch fp64 CPU SDPA and its autograd) the oracle does not use.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle import online_softmax as ons

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed, dtype=torch.float64, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * mult).to(dtype)


# --- worked example (FlashAttention_01 page, large-score practice section) ---

def test_worked_example_printed_values():
    g = _golden("worked_example.json")
    k = np.array(g["scores"])[:, None]
    v = np.array(g["values"])[:, None]
    m, l, u, o, lse = orc.row_state(np.array([1.0]), k, v, scale=1.0)
    tol = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    last = g["printed_steps"][-1]
    assert m == last["m"]
    assert abs(l - last["l"]) <= tol
    assert abs(u[0] - last["u"]) <= tol
    assert abs(o[0] - g["printed_output"]) <= tol
    assert math.isfinite(lse)


def test_worked_example_closed_form():
    k = np.array([[1000.0], [1001.0], [999.0]])
    v = np.array([[1.0], [3.0], [7.0]])
    m, l, u, o, lse = orc.row_state(np.array([1.0]), k, v, scale=1.0)
    e1, e2 = math.exp(-1.0), math.exp(-2.0)
    assert abs(l - (e1 + 1.0 + e2)) < 1e-14
    assert abs(u[0] - (e1 * 1 + 3 + 7 * e2)) < 1e-13
    assert abs(o[0] - (e1 + 3 + 7 * e2) / (e1 + 1 + e2)) < 1e-14
    assert abs(lse - (1001.0 + math.log(e1 + 1 + e2))) < 1e-12


def test_worked_example_step_trace():
    """One key per tile: the recurrence's states after each block are the
    printed (m, l, u) triples."""
    g = _golden("worked_example.json")
    trace = []
    ons.tiled_row([1.0], np.array(g["scores"])[:, None], np.array(g["values"])[:, None],
                  tile=1, scale=1.0, trace=trace)
    tol = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    for (m, l, u), want in zip(trace, g["printed_steps"]):
        assert m == want["m"]
        assert abs(l - want["l"]) <= tol
        assert abs(u[0] - want["u"]) <= tol


def test_worked_example_bf16_encoding_is_exact():
    """The bf16 encoding used on the GPU reproduces scores 1000, 1001, 999."""
    from io_aware_exact_tcgen05_gb300.workloads import worked_example_bf16
    q, k, v = worked_example_bf16()
    s = (k.double()[0, 0] @ q.double()[0, 0, 0])
    assert s.tolist() == [1000.0, 1001.0, 999.0]
    assert v.double()[0, 0, :, 0].tolist() == [1.0, 3.0, 7.0]
    o, lse = orc.fwd(q, k, v, causal=False, scale=1.0)
    e1, e2 = math.exp(-1.0), math.exp(-2.0)
    assert abs(o[0, 0, 0, 0] - (e1 + 3 + 7 * e2) / (e1 + 1 + e2)) < 1e-14
    assert np.all(o[0, 0, 0, 1:] == 0.0)


# --- tiled vs one-shot (FlashAttention_01 page, reviewable experiment) ---

@pytest.mark.parametrize("tile", [1, 2, 3, 8, 16, 37])
@pytest.mark.parametrize("mult", [1.0, 300.0])
def test_tiled_recurrence_matches_untiled_oracle(tile, mult):
    n, d = 100, 16  # 100 keys: every listed tile length leaves a ragged last block
    q = _rand((d,), 1, mult=mult).numpy()
    K = _rand((n, d), 2).numpy()
    V = _rand((n, d), 3).numpy()
    m1, l1, u1, o1, lse1 = ons.tiled_row(q, K, V, tile)
    m0, l0, u0, o0, lse0 = orc.row_state(q, K, V, 1.0 / math.sqrt(d))
    assert np.all(np.isfinite(o1)) and math.isfinite(lse1)
    scale_o = max(1.0, float(np.abs(o0).max()))
    assert float(np.abs(o1 - o0).max()) <= 1e-12 * scale_o
    assert abs(lse1 - lse0) <= 1e-12 * max(1.0, abs(lse0))
    assert abs(m1 - m0) <= 1e-14 * max(1.0, abs(m0))  # dot-product order differs


def test_tiled_recurrence_with_mask_and_empty_row():
    n, d = 37, 8
    q = _rand((d,), 4).numpy()
    K = _rand((n, d), 5).numpy()
    V = _rand((n, d), 6).numpy()
    vis = np.zeros(n, bool)
    vis[10:20] = True
    for tile in (1, 2, 3, 8):
        m, l, u, o, lse = ons.tiled_row(q, K, V, tile, visible=vis)
        _, _, _, o0, lse0 = orc.row_state(q, K[10:20], V[10:20], 1.0 / math.sqrt(d))
        assert np.abs(o - o0).max() < 1e-13 and abs(lse - lse0) < 1e-13
    m, l, u, o, lse = ons.tiled_row(q, K, V, 3, visible=np.zeros(n, bool))
    assert m == -np.inf and l == 0.0 and lse == -np.inf and np.all(o == 0)


# --- cross-check with the framework's native SDPA, fp64 CPU (FlashAttention_01
#     page, 5.1: build the numerical baseline with native SDPA) ---

def _mask(Sq, Sk, causal, ks, ke, B):
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Sk)[None, :]
    m = torch.ones(B, 1, Sq, Sk, dtype=torch.bool)
    for b in range(B):
        vis = (j >= ks[b]) & (j < ke[b])
        if causal:
            vis = vis & (j <= i + Sk - Sq)
        m[b, 0] = vis
    return m


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal, ks, ke
    (2, 4, 4, 33, 33, 16, True, None, None),
    (1, 4, 2, 17, 29, 8, True, None, None),
    (2, 6, 2, 31, 20, 16, False, [3, 0], [20, 11]),
    (2, 4, 1, 24, 24, 32, True, [5, 0], [24, 24]),
    (1, 2, 2, 1, 40, 8, False, [0], [13]),
]


@pytest.mark.parametrize("case", CASES)
def test_forward_matches_torch_sdpa_fp64(case):
    B, Hq, Hkv, Sq, Sk, d, causal, ks, ke = case
    ks = ks or [0] * B
    ke = ke or [Sk] * B
    q = _rand((B, Hq, Sq, d), 10)
    k = _rand((B, Hkv, Sk, d), 11)
    v = _rand((B, Hkv, Sk, d), 12)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.fwd(q, k, v, causal, scale, k_start=ks, k_end=ke)
    mask = _mask(Sq, Sk, causal, ks, ke, B)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=scale, enable_gqa=(Hq != Hkv))
    rep = Hq // Hkv
    s = torch.einsum("bhid,bhjd->bhij", q, k.repeat_interleave(rep, 1)) * scale
    s = s.masked_fill(~mask, -math.inf)
    ref_lse = torch.logsumexp(s, -1)
    live = mask.any(-1).expand(B, Hq, Sq)
    assert np.abs(o[live.numpy()] - ref[live].numpy()).max() < 1e-12
    assert np.abs(lse[live.numpy()] - ref_lse[live].numpy()).max() < 1e-12
    dead = ~live.numpy()
    assert np.all(o[dead] == 0.0) and np.all(lse[dead] == -np.inf)


@pytest.mark.parametrize("case", CASES)
def test_backward_matches_torch_autograd_fp64(case):
    B, Hq, Hkv, Sq, Sk, d, causal, ks, ke = case
    ks = ks or [0] * B
    ke = ke or [Sk] * B
    q = _rand((B, Hq, Sq, d), 20)
    k = _rand((B, Hkv, Sk, d), 21)
    v = _rand((B, Hkv, Sk, d), 22)
    do = _rand((B, Hq, Sq, d), 23)
    scale = 1.0 / math.sqrt(d)
    mask = _mask(Sq, Sk, causal, ks, ke, B)
    live = mask.any(-1).expand(B, Hq, Sq)
    # torch yields NaN rows where nothing is visible; zero their upstream grad
    do_t = do.masked_fill(~live[..., None], 0.0)
    qt, kt, vt = (x.clone().requires_grad_() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=scale, enable_gqa=(Hq != Hkv))
    ref = torch.where(live[..., None], ref, torch.zeros_like(ref))
    ref.backward(do_t)
    dq, dk, dv = orc.bwd(q, k, v, do, causal, scale, k_start=ks, k_end=ke)
    for mine, theirs in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.abs(mine - theirs.numpy()).max() < 1e-11
    assert np.all(dq[~live.numpy()] == 0.0)


# --- per-key boolean masks and packed ragged sequences (FlashAttention_01
#     page, "interface and implementation constraints": masks and ragged
#     layouts are part of the kernel contract; logical vs packed rows) ---

def _key_mask(B, Sk, seed, drop=0.3):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(B, Sk, generator=g) >= drop


def _sdpa_ref(q, k, v, mask, scale, do=None):
    """fp64 torch SDPA with a boolean [B,1,Sq,Sk] mask: (O, LSE, live rows) and,
    with do, the autograd gradients (dead rows get zero upstream grad)."""
    B, Hq, Sq, _ = q.shape
    Hkv = k.shape[1]
    live = mask.any(-1).expand(B, Hq, Sq)
    qt, kt, vt = (x.clone().requires_grad_() for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=mask, scale=scale, enable_gqa=(Hq != Hkv))
    ref = torch.where(live[..., None], ref, torch.zeros_like(ref))
    s = torch.einsum("bhid,bhjd->bhij", q, k.repeat_interleave(Hq // Hkv, 1)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), -1)
    grads = None
    if do is not None:
        ref.backward(do.masked_fill(~live[..., None], 0.0))
        grads = (qt.grad, kt.grad, vt.grad)
    return ref.detach(), lse, live, grads


MASK_CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (2, 4, 2, 29, 37, 16, True),
    (1, 2, 2, 40, 40, 8, False),
    (2, 2, 1, 17, 23, 16, True),
]


@pytest.mark.parametrize("case", MASK_CASES)
def test_key_mask_matches_torch_sdpa_fp64(case):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    q = _rand((B, Hq, Sq, d), 40)
    k = _rand((B, Hkv, Sk, d), 41)
    v = _rand((B, Hkv, Sk, d), 42)
    do = _rand((B, Hq, Sq, d), 43)
    km = _key_mask(B, Sk, 44)
    km[0, :Sk // 2] = False  # long masked run: some causal rows see nothing
    scale = 1.0 / math.sqrt(d)
    mask = _mask(Sq, Sk, causal, [0] * B, [Sk] * B, B) & km[:, None, None, :]
    ref, ref_lse, live, (gq, gk, gv) = _sdpa_ref(q, k, v, mask, scale, do)
    o, lse = orc.fwd(q, k, v, causal, scale, key_mask=km)
    L = live.numpy()
    assert L.any() and (L.all() != causal)  # causal rows 0.. see only masked keys
    assert np.abs(o[L] - ref[live].numpy()).max() < 1e-12
    assert np.abs(lse[L] - ref_lse[live].numpy()).max() < 1e-12
    assert np.all(o[~L] == 0.0) and np.all(lse[~L] == -np.inf)
    dq, dk, dv = orc.bwd(q, k, v, do, causal, scale, key_mask=km)
    for mine, theirs in ((dq, gq), (dk, gk), (dv, gv)):
        assert np.abs(mine - theirs.numpy()).max() < 1e-11
    # a masked key gets exactly zero gradient and zero probability
    dead_keys = ~km.numpy()
    for b in range(B):
        assert np.all(dk[b][:, dead_keys[b]] == 0.0) and np.all(dv[b][:, dead_keys[b]] == 0.0)
    p = orc.probs(q, k, v, causal, scale, key_mask=km)
    assert np.all(p[..., :][np.broadcast_to(dead_keys[:, None, None, :], p.shape)] == 0.0)


def test_interval_key_mask_equals_key_interval():
    B, Hq, Hkv, Sq, Sk, d = 2, 2, 1, 21, 30, 8
    q = _rand((B, Hq, Sq, d), 50)
    k = _rand((B, Hkv, Sk, d), 51)
    v = _rand((B, Hkv, Sk, d), 52)
    do = _rand((B, Hq, Sq, d), 53)
    ks, ke = [4, 0], [30, 17]
    j = torch.arange(Sk)[None, :]
    km = (j >= torch.tensor(ks)[:, None]) & (j < torch.tensor(ke)[:, None])
    for causal in (False, True):
        a = orc.fwd(q, k, v, causal, 0.3, k_start=ks, k_end=ke)
        b = orc.fwd(q, k, v, causal, 0.3, key_mask=km)
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
        ga = orc.bwd(q, k, v, do, causal, 0.3, k_start=ks, k_end=ke)
        gb = orc.bwd(q, k, v, do, causal, 0.3, key_mask=km)
        assert all(np.array_equal(x, y) for x, y in zip(ga, gb))


VARLEN_Q = [5, 0, 17, 33, 3]
VARLEN_K = [9, 4, 17, 20, 0]


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_per_sequence_torch_sdpa(causal):
    Hq, Hkv, d = 4, 2, 16
    cu_q = np.concatenate([[0], np.cumsum(VARLEN_Q)])
    cu_k = np.concatenate([[0], np.cumsum(VARLEN_K)])
    q = _rand((Hq, int(cu_q[-1]), d), 60)
    k = _rand((Hkv, int(cu_k[-1]), d), 61)
    v = _rand((Hkv, int(cu_k[-1]), d), 62)
    do = _rand((Hq, int(cu_q[-1]), d), 63)
    km = _key_mask(1, int(cu_k[-1]), 64, drop=0.2)[0]
    scale = 1.0 / math.sqrt(d)
    for use_mask in (False, True):
        kmask = km if use_mask else None
        o, lse = orc.fwd_varlen(q, k, v, cu_q, cu_k, causal, scale, key_mask=kmask)
        dq, dk, dv = orc.bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale, key_mask=kmask)
        for s in range(len(VARLEN_Q)):
            q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
            if q1 == q0:
                continue
            if k1 == k0:  # a sequence without keys: its rows are fully masked
                assert np.all(o[:, q0:q1] == 0.0) and np.all(lse[:, q0:q1] == -np.inf)
                assert np.all(dq[:, q0:q1] == 0.0)
                continue
            Sq, Sk = q1 - q0, k1 - k0
            mask = _mask(Sq, Sk, causal, [0], [Sk], 1)
            if use_mask:
                mask = mask & km[None, None, None, k0:k1]
            ref, ref_lse, live, (gq, gk, gv) = _sdpa_ref(
                q[None, :, q0:q1], k[None, :, k0:k1], v[None, :, k0:k1], mask, scale,
                do[None, :, q0:q1])
            L = live[0].numpy()
            assert np.abs(o[:, q0:q1][L] - ref[0][live[0]].numpy()).max() < 1e-12
            assert np.abs(lse[:, q0:q1][L] - ref_lse[0][live[0]].numpy()).max() < 1e-12
            assert np.all(lse[:, q0:q1][~L] == -np.inf)
            assert np.abs(dq[:, q0:q1] - gq[0].numpy()).max() < 1e-11
            assert np.abs(dk[:, k0:k1] - gk[0].numpy()).max() < 1e-11
            assert np.abs(dv[:, k0:k1] - gv[0].numpy()).max() < 1e-11


def test_varlen_equal_lengths_equals_batched():
    B, Hq, Hkv, S, d = 3, 2, 1, 12, 8
    q = _rand((B, Hq, S, d), 70)
    k = _rand((B, Hkv, S, d), 71)
    v = _rand((B, Hkv, S, d), 72)
    pack = lambda x: x.permute(1, 0, 2, 3).reshape(x.shape[1], B * S, d)  # noqa: E731
    cu = np.arange(B + 1) * S
    o, lse = orc.fwd_varlen(pack(q), pack(k), pack(v), cu, cu, True, 0.4)
    ob, lb = orc.fwd(q, k, v, True, 0.4)
    assert np.array_equal(o, ob.transpose(1, 0, 2, 3).reshape(Hq, B * S, d))
    assert np.array_equal(lse, lb.transpose(1, 0, 2).reshape(Hq, B * S))


# --- dropout with a counter-based mask (FlashAttention_01 page, "why the
#     backward can recompute" and "interface and implementation constraints":
#     the element-to-random-number mapping is part of the contract) ---

# Known-answer vectors published with the reference implementation of
# Philox4x32-10 (Random123, Salmon et al., SC 2011): counter, key -> output.
PHILOX_KAT = [
    ([0, 0, 0, 0], [0, 0], [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]),
    ([0xffffffff] * 4, [0xffffffff] * 2, [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]),
    ([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0],
     [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]),
]


@pytest.mark.parametrize("ctr,key,want", PHILOX_KAT)
def test_philox_known_answers(ctr, key, want):
    assert [int(x) for x in orc.philox4x32_10(ctr, key)] == want


def test_dropout_keep_rate_and_mapping():
    p, seed, off = 0.3, 0x0123456789ABCDEF, 7
    keep = np.array([orc.dropout_keep(p, seed, off, bh, i, j)
                     for bh in range(2) for i in range(60) for j in range(257)])
    n = keep.size
    sigma = math.sqrt(n * p * (1 - p))
    assert abs(keep.sum() - n * (1 - p)) < 5 * sigma
    # the decision is the 16-bit half j % 2 of word (j % 8) // 2 of the Philox
    # call at counter (j // 8, i, bh, offset), against floor(p * 2^16)
    for (bh, i, j) in [(0, 0, 0), (1, 5, 6), (1, 59, 255), (0, 17, 3), (1, 2, 7), (0, 44, 9)]:
        w = orc.philox4x32_10([j // 8, i, bh, off], [seed & 0xffffffff, seed >> 32])
        draw = (int(w[(j % 8) // 2]) >> (16 * (j % 2))) & 0xFFFF
        assert orc.dropout_keep(p, seed, off, bh, i, j) == (draw >= int(p * 2**16))
    # eight consecutive keys share one call; the next eight use the next counter
    w0 = orc.philox4x32_10([0, 3, 1, off], [seed & 0xffffffff, seed >> 32])
    w1 = orc.philox4x32_10([1, 3, 1, off], [seed & 0xffffffff, seed >> 32])
    halves = [(int(x) >> s) & 0xFFFF for w in (w0, w1) for x in w for s in (0, 16)]
    assert [orc.dropout_keep(p, seed, off, 1, 3, j) for j in range(16)] == \
        [h >= int(p * 2**16) for h in halves]
    # a probability below 2^-16 keeps every weight (threshold 0)
    assert all(orc.dropout_keep(1e-6, seed, off, 0, 3, j) for j in range(64))
    # p = 0 keeps everything; another seed or offset gives another mask
    assert all(orc.dropout_keep(0.0, seed, off, 0, 3, j) for j in range(64))
    a = [orc.dropout_keep(p, seed, off, 0, 3, j) for j in range(256)]
    assert a != [orc.dropout_keep(p, seed + 1, off, 0, 3, j) for j in range(256)]
    assert a != [orc.dropout_keep(p, seed, off + 1, 0, 3, j) for j in range(256)]


def test_dropout_that_drops_nothing_is_the_plain_attention():
    # p below 2^-16: every 16-bit draw is >= 0, so nothing is dropped, the
    # keep probability is 1 and the result must be the undropped attention
    B, Hq, Hkv, Sq, Sk, d = 1, 2, 1, 17, 29, 8
    q = _rand((B, Hq, Sq, d), 90)
    k = _rand((B, Hkv, Sk, d), 91)
    v = _rand((B, Hkv, Sk, d), 92)
    do = _rand((B, Hq, Sq, d), 93)
    o0, l0 = orc.fwd(q, k, v, True, 0.3)
    o1, l1 = orc.fwd(q, k, v, True, 0.3, dropout_p=2.0**-17, seed=5, offset=1)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0 = orc.bwd(q, k, v, do, True, 0.3)
    g1 = orc.bwd(q, k, v, do, True, 0.3, dropout_p=2.0**-17, seed=5, offset=1)
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


def test_dropout_keeps_the_expectation():
    # inverted dropout: averaged over many masks, the dropped output is the
    # undropped one (the kept weights carry 1 / P(keep)); with the 16-bit
    # threshold P(keep) = 1 - floor(p 2^16) / 2^16, which differs from 1 - p
    # for p = 0.3, so the mean of keep * scale must be 1, not (1-q)/(1-p)
    p, off = 0.3, 2
    Sk, d = 64, 4
    q = torch.zeros(1, 1, 1, d, dtype=torch.float64)
    k = torch.zeros(1, 1, Sk, d, dtype=torch.float64)
    v = torch.ones(1, 1, Sk, d, dtype=torch.float64)
    # scale 0: uniform weights 1/Sk, so O = mean over keys of keep * scale
    outs = [orc.fwd(q, k, v, False, 0.0, dropout_p=p, seed=s, offset=off)[0][0, 0, 0, 0]
            for s in range(400)]
    thr = math.floor(p * 65536)
    r = 65536.0 / (65536.0 - thr)
    kept = np.array(outs) / r * Sk  # kept keys per mask
    assert np.allclose(kept, np.round(kept), atol=1e-9)  # O is (kept count) * r / Sk exactly
    n = len(outs) * Sk
    keep_rate = kept.sum() / n
    sigma = math.sqrt((1 - thr / 65536) * (thr / 65536) / n)
    assert abs(keep_rate - (1 - thr / 65536)) < 5 * sigma
    assert abs(np.mean(outs) - 1.0) < 5 * sigma * r


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_matches_explicit_mask_in_torch_fp64(causal):
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 19, 23, 8
    p, seed, off = 0.25, 99, 3
    q = _rand((B, Hq, Sq, d), 80)
    k = _rand((B, Hkv, Sk, d), 81)
    v = _rand((B, Hkv, Sk, d), 82)
    do = _rand((B, Hq, Sq, d), 83)
    scale = 1.0 / math.sqrt(d)
    keep = torch.tensor([[[[orc.dropout_keep(p, seed, off, b * Hq + h, i, j) for j in range(Sk)]
                           for i in range(Sq)] for h in range(Hq)] for b in range(B)],
                        dtype=torch.float64)
    vis = _mask(Sq, Sk, causal, [0] * B, [Sk] * B, B)
    qt, kt, vt = (x.clone().requires_grad_() for x in (q, k, v))
    rep = Hq // Hkv
    s = torch.einsum("bhid,bhjd->bhij", qt, kt.repeat_interleave(rep, 1)) * scale
    s = s.masked_fill(~vis, -math.inf)
    prob = torch.softmax(s, -1)
    ref = torch.einsum("bhij,bhjd->bhid", prob * keep / (1 - p), vt.repeat_interleave(rep, 1))
    ref.backward(do)
    o, lse = orc.fwd(q, k, v, causal, scale, dropout_p=p, seed=seed, offset=off)
    assert np.abs(o - ref.detach().numpy()).max() < 1e-12
    assert np.abs(lse - torch.logsumexp(s.detach(), -1).numpy()).max() < 1e-12  # undropped
    dq, dk, dv = orc.bwd(q, k, v, do, causal, scale, dropout_p=p, seed=seed, offset=off)
    for mine, theirs in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.abs(mine - theirs.numpy()).max() < 1e-11
    # p = 0 is exactly the plain path
    a = orc.fwd(q, k, v, causal, scale, dropout_p=0.0, seed=seed, offset=off)
    b_ = orc.fwd(q, k, v, causal, scale)
    assert all(np.array_equal(x, y) for x, y in zip(a, b_))


# --- FP8 (e4m3) inputs: the decoder is the format's definition ---

def test_e4m3_decoder_known_codes_and_torch():
    codes = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x7E: 448.0, 0x80: -0.0, 0xC0: -2.0, 0xFE: -448.0}
    got = orc.decode_e4m3(np.array(list(codes), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(codes.values())))
    assert np.isnan(orc.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch without float8_e4m3fn")
    allc = torch.arange(256, dtype=torch.uint8)
    ref = allc.view(f8).to(torch.float64).numpy()
    mine = orc.decode_e4m3(allc.numpy())
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(mine), ~finite)
    assert np.array_equal(mine[finite], ref[finite])


# --- chain-rule section: central differences on the 2x3x2 masked example ---

def _loss(q, k, v):
    o, _ = orc.fwd(q, k, v, causal=True, scale=1.0 / math.sqrt(2))
    return 0.5 * float((o ** 2).sum())


def test_central_differences_2x3_masked():
    """2 queries, 3 keys, d=2; row 0 may not read key 2 (bottom-right causal
    rule, Sq=2, Sk=3); J = 0.5*sum(O^2) so dO = O."""
    q = _rand((1, 1, 2, 2), 30).numpy()
    k = _rand((1, 1, 3, 2), 31).numpy()
    v = _rand((1, 1, 3, 2), 32).numpy()
    p = orc.probs(q, k, v, causal=True, scale=1.0 / math.sqrt(2))
    assert p[0, 0, 0, 2] == 0.0 and p[0, 0, 1, 2] > 0.0
    o, _ = orc.fwd(q, k, v, causal=True, scale=1.0 / math.sqrt(2))
    dq, dk, dv = orc.bwd(q, k, v, o, causal=True, scale=1.0 / math.sqrt(2))
    h = 1e-6
    worst = 0.0
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(arr.shape):
            save = arr[idx]
            arr[idx] = save + h
            jp = _loss(q, k, v)
            arr[idx] = save - h
            jm = _loss(q, k, v)
            arr[idx] = save
            num = (jp - jm) / (2 * h)
            worst = max(worst, abs(num - grad[idx]))
    assert worst < 1e-8, worst


# --- gradient invariants (chain-rule section) ---

def test_gradient_invariants():
    B, Hq, Hkv, Sq, Sk, d = 2, 4, 2, 12, 12, 8
    ks, ke = [4, 0], [12, 9]
    q, k, v, do = (_rand(s, 40 + i) for i, s in enumerate(
        [(B, Hq, Sq, d), (B, Hkv, Sk, d), (B, Hkv, Sk, d), (B, Hq, Sq, d)]))
    scale = 1.0 / math.sqrt(d)
    p, ds = orc.probs(q, k, v, causal=True, scale=scale, dout=do, k_start=ks, k_end=ke)
    mask = _mask(Sq, Sk, True, ks, ke, B).expand(B, Hq, Sq, Sk).numpy()
    assert np.abs(ds.sum(-1)).max() < 1e-13  # rowsum dS = 0
    assert np.all(p[~mask] == 0.0) and np.all(ds[~mask] == 0.0)
    live = mask.any(-1)
    assert np.allclose(p.sum(-1)[live], 1.0, atol=1e-14)
    dq, dk, dv = orc.bwd(q, k, v, do, True, scale, k_start=ks, k_end=ke)
    assert np.abs(dk.sum(2)).max() < 1e-12  # sum_j dK_j = 0 per (b, hkv)
    # sum_j dV_j = sum over non-empty rows of dO, per KV head
    dos = do.numpy() * live[..., None]
    want = dos.reshape(B, Hkv, Hq // Hkv, Sq, d).sum((2, 3))
    assert np.abs(dv.sum(2) - want).max() < 1e-12


# --- special cases (boundary section: single visible key, empty row, repeated maxima) ---

def test_single_visible_key():
    q = _rand((1, 1, 1, 4), 50)
    k = _rand((1, 1, 6, 4), 51)
    v = _rand((1, 1, 6, 4), 52)
    o, lse = orc.fwd(q, k, v, False, 0.5, k_start=[3], k_end=[4])
    assert np.abs(o[0, 0, 0] - v[0, 0, 3].numpy()).max() == 0.0
    assert abs(lse[0, 0, 0] - 0.5 * float(q[0, 0, 0] @ k[0, 0, 3])) < 1e-15


def test_zero_query_gives_mean_and_log_count():
    q = torch.zeros(1, 1, 5, 8, dtype=torch.float64)
    k = _rand((1, 1, 5, 8), 53)
    v = _rand((1, 1, 5, 8), 54)
    o, lse = orc.fwd(q, k, v, True, 0.3)
    for i in range(5):
        assert np.abs(o[0, 0, i] - v[0, 0, : i + 1].numpy().mean(0)).max() < 1e-15
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-15


def test_fully_masked_rows_are_zero_and_finite():
    B, H, S, d = 1, 2, 10, 8
    q, k, v, do = (_rand((B, H, S, d), 60 + i) for i in range(4))
    o, lse = orc.fwd(q, k, v, True, 0.25, k_start=[4], k_end=[10])
    assert np.all(o[0, :, :4] == 0.0) and np.all(lse[0, :, :4] == -np.inf)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse[0, :, 4:]))
    dq, dk, dv = orc.bwd(q, k, v, do, True, 0.25, k_start=[4], k_end=[10])
    for g in (dq, dk, dv):
        assert np.all(np.isfinite(g))
    assert np.all(dq[0, :, :4] == 0.0)
    assert np.all(dk[0, :, :4] == 0.0) and np.all(dv[0, :, :4] == 0.0)


def test_repeated_maxima():
    K = np.array([[2.0], [2.0], [1.0], [2.0]])
    V = np.array([[1.0], [2.0], [3.0], [4.0]])
    m, l, u, o, lse = orc.row_state(np.array([1.0]), K, V, 1.0)
    e = math.exp(-1.0)
    assert m == 2.0
    assert abs(l - (3 + e)) < 1e-15
    assert abs(o[0] - (1 + 2 + 4 + 3 * e) / (3 + e)) < 1e-15
    for tile in (1, 2, 3):
        _, _, _, ot, _ = ons.tiled_row([1.0], K, V, tile, scale=1.0)
        assert abs(ot[0] - o[0]) < 1e-15


def test_large_logits_stay_finite():
    q = _rand((1, 2, 16, 8), 70, mult=800.0)
    k = _rand((1, 2, 16, 8), 71)
    v = _rand((1, 2, 16, 8), 72)
    o, lse = orc.fwd(q, k, v, True, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.abs(lse).max() > 710  # exp(lse) itself would overflow fp64


# --- decode and split-KV merge ---

def test_decode_equals_forward_with_interval_and_split_invariance():
    B, Hq, Hkv, Smax, d = 3, 4, 2, 50, 8
    q = _rand((B, Hq, 1, d), 80)
    k = _rand((B, Hkv, Smax, d), 81)
    v = _rand((B, Hkv, Smax, d), 82)
    lens = [50, 7, 23]
    o, lse = orc.decode(q, k, v, lens, 0.35)
    o2, lse2 = orc.fwd(q, k, v, False, 0.35, k_start=[0] * B, k_end=lens)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    for b in range(B):
        for h in range(Hq):
            for chunk in (1, 5, 16, 64):
                states = []
                for c0 in range(0, Smax, chunk):
                    oc, lc = orc.fwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], False, 0.35,
                                     k_start=[c0], k_end=[min(c0 + chunk, lens[b])])
                    states.append((lc[0, h, 0], oc[0, h, 0]))
                lm, om = ons.merge_states(states)
                assert abs(lm - lse[b, h, 0]) < 1e-12
                assert np.abs(om - o[b, h, 0]).max() < 1e-12


def test_bf16_inputs_widen_exactly():
    q = _rand((1, 2, 9, 16), 90).to(torch.bfloat16)
    k = _rand((1, 1, 9, 16), 91).to(torch.bfloat16)
    v = _rand((1, 1, 9, 16), 92).to(torch.bfloat16)
    a = orc.fwd(q, k, v, True, 0.25)
    b = orc.fwd(q.double(), k.double(), v.double(), True, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_dq_rows_equal_full_backward():
    B, Hq, Hkv, S, d = 2, 4, 2, 37, 16
    q = _rand((B, Hq, S, d), 100)
    k = _rand((B, Hkv, S, d), 101)
    v = _rand((B, Hkv, S, d), 102)
    do = _rand((B, Hq, S, d), 103)
    for causal in (False, True):
        dq, _, _ = orc.bwd(q, k, v, do, causal, 0.3, k_start=[3, 0], k_end=[37, 20])
        rows = [0, 5, 36, 37, 80, 143, B * Hq * S - 1]
        got = orc.bwd_dq_rows(q, k, v, do, causal, 0.3, rows, k_start=[3, 0], k_end=[37, 20])
        assert np.array_equal(got, dq.reshape(-1, d)[rows])


def test_row_subset_equals_full():
    q = _rand((2, 4, 20, 8), 95)
    k = _rand((2, 2, 20, 8), 96)
    v = _rand((2, 2, 20, 8), 97)
    o, lse = orc.fwd(q, k, v, True, 0.3, k_start=[2, 0], k_end=[20, 15])
    rows = [0, 1, 5, 79, 80, 159]
    os_, ls = orc.fwd(q, k, v, True, 0.3, k_start=[2, 0], k_end=[20, 15], rows=rows)
    assert np.array_equal(os_, o.reshape(-1, 8)[rows])
    assert np.array_equal(ls, lse.reshape(-1)[rows])
