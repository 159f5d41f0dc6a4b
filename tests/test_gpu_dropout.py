"""GPU dropout (fa_fwd_dropout / fa_bwd_dropout through the C ABI) against the
FP64 oracle's Philox4x32-10 mapping: the keep decisions must agree exactly
(they are integer comparisons of 16-bit draws on both sides), and O, LSE, dQ,
dK, dV within the usual tolerances.  Probabilities are exact in float32, so
both sides use the same integer threshold thr = floor(p * 2^16); kept weights
are scaled by 2^16 / (2^16 - thr), and 2^-17 has threshold 0 (every weight
kept, unscaled)."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _status_ok():
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)


@pytest.mark.parametrize("p", [0.25, 0.625, 2.0**-17])
def test_keep_decisions_match_the_mapping_exactly(p):
    # scale 0: every visible key has weight 1/128; V row j is the unit vector
    # e_(j - k0), so O[..., c] = keep(key k0 + c) * r / 128 reads the
    # mask off directly.  Keys 384..511 of batch row 1 exercise large key
    # indices; several heads and 200 rows vary the other counter words.
    B, H, Sq, Sk, d = 2, 3, 200, 512, 128
    k0s = [0, 384]
    q = torch.zeros(B, H, Sq, d, dtype=torch.bfloat16)
    k = torch.zeros(B, H, Sk, d, dtype=torch.bfloat16)
    v = torch.zeros(B, H, Sk, d, dtype=torch.bfloat16)
    for b, k0 in enumerate(k0s):
        v[b, :, k0:k0 + 128] = torch.eye(128, dtype=torch.bfloat16)
    ks = torch.tensor(k0s, dtype=torch.int32)
    ke = ks + 128
    seed, off = 0x1234_5678_9ABC_DEF0, 11
    o, lse = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), False, 0.0, k_start=ks.to(DEV),
                       k_end=ke.to(DEV), dropout_p=p, seed=seed, offset=off)
    torch.cuda.synchronize()
    _status_ok()
    got = to_np(o) > 0
    want = np.zeros_like(got)
    for b, k0 in enumerate(k0s):
        for h in range(H):
            for i in range(Sq):
                for c in range(128):
                    want[b, h, i, c] = orc.dropout_keep(p, seed, off, b * H + h, i, k0 + c)
    assert np.array_equal(got, want), f"{int((got != want).sum())} decisions differ"
    kept = to_np(o)[got]
    thr = math.floor(p * 65536.0)
    assert np.allclose(kept, 65536.0 / (65536.0 - thr) / 128.0, rtol=1e-2)
    assert np.allclose(to_np(lse), math.log(128.0), atol=1e-5)  # LSE of the undropped weights


CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal, p
    (2, 4, 2, 300, 300, 128, True, 0.25),
    (1, 2, 2, 257, 400, 64, False, 0.125),
    (2, 2, 1, 130, 130, 128, True, 0.5),
]


@pytest.mark.parametrize("case", CASES)
def test_dropout_fwd_bwd_against_oracle(case):
    B, Hq, Hkv, Sq, Sk, d, causal, p = case
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=51, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    seed, off = 2024, 5
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, causal, scale, dropout_p=p, seed=seed, offset=off)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal, scale, dropout_p=p, seed=seed,
                           offset=off)
    torch.cuda.synchronize()
    _status_ok()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], causal, scale, dropout_p=p, seed=seed, offset=off)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    rq, rk, rv = orc.bwd(t["q"], t["k"], t["v"], t["dout"], causal, scale, dropout_p=p,
                         seed=seed, offset=off)
    check_grad(to_np(dq), rq, "dQ")
    check_grad(to_np(dk), rk, "dK")
    check_grad(to_np(dv), rv, "dV")


def test_dropout_with_key_mask_and_zero_probability():
    B, H, S, d = 1, 2, 200, 128
    t = workloads.random_qkv(B, H, H, S, S, d, seed=53, with_dout=True)
    g = torch.Generator().manual_seed(54)
    km = torch.rand(B, S, generator=g) >= 0.3
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, True, 0.1, key_mask=km.to(DEV), dropout_p=0.375, seed=7)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, True, 0.1, key_mask=km.to(DEV),
                           dropout_p=0.375, seed=7)
    torch.cuda.synchronize()
    _status_ok()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, 0.1, key_mask=km, dropout_p=0.375, seed=7)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    rq, rk, rv = orc.bwd(t["q"], t["k"], t["v"], t["dout"], True, 0.1, key_mask=km,
                         dropout_p=0.375, seed=7)
    check_grad(to_np(dq), rq, "dQ")
    check_grad(to_np(dk), rk, "dK")
    check_grad(to_np(dv), rv, "dV")
    # dropout_p = 0 through the dropout entry point is exactly the plain forward
    lib = fa.load_library()
    o0 = torch.empty_like(q)
    l0 = torch.empty(B, H, S, dtype=torch.float32, device=DEV)
    import ctypes
    st = lib.fa_fwd_dropout(fa._ptr(q), fa._ptr(k), fa._ptr(v), fa._ptr(o0), fa._ptr(l0), B, H, H,
                            S, S, d, 1, ctypes.c_float(0.1), None, None, None,
                            ctypes.c_float(0.0), 7, 0, fa._stream(None))
    assert st == 0
    o1, l1 = fa.fa_fwd(q, k, v, True, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
