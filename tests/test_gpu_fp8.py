"""GPU FP8 (e4m3) forward (fa_fwd_fp8 through the C ABI) against the FP64
oracle run on the exactly dequantised inputs.

Tolerance, derived from the arithmetic: the dequantised inputs are exact and
fp32 accumulation of e4m3 products is exact to ~2^-24, so the error comes from
rounding the softmax weights to e4m3 for the PV product.  A rounded weight
has relative error <= 2^-4 (normal range) or absolute error <= 2^-10
(subnormals and flush); the kernel's weights are relative to a running max,
so the row's weight sum l >= 1, and O is normalised by the sum of the rounded
weights.  Hence, per row i and output column c,
  |O_gpu - O| <= (2^-4 / (1 - 2^-4)) * sum_j P_ij |v_jc - O_ic|
               + (2^-10 / (1 - 2^-4)) * sum_j |v_jc - O_ic|
plus the bf16 rounding of the output (bf16 keeps 8 significant bits: at
most 2^-8 |O|); a 1e-4 floor absorbs fp32 accumulation.  The LSE comes from
the exact fp32 weight sum: 1e-3 as always."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_lse, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
F8 = getattr(torch, "float8_e4m3fn", None)


def _quant(x):
    """e4m3 bytes of x / descale with descale = max|x| / 448 (per tensor)."""
    xf = x.float()
    ds = float(xf.abs().max()) / 448.0
    return (xf / ds).to(F8), ds


def _case(B, Hq, Hkv, Sq, Sk, causal, seed, ks=None, ke=None, qmul=1.0, heads=None):
    """heads: query heads whose every row is held to the element-wise bound
    (default all; the LSE of every head is checked either way)."""
    if F8 is None:
        pytest.skip("torch without float8_e4m3fn")
    d = 128
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=seed)
    q8, qd = _quant(t["q"].float() * qmul)
    k8, kd = _quant(t["k"])
    v8, vd = _quant(t["v"])
    vt8 = v8.transpose(-1, -2).contiguous()
    scale = 1.0 / math.sqrt(d)
    kst = None if ks is None else torch.tensor(ks, dtype=torch.int32)
    ken = None if ke is None else torch.tensor(ke, dtype=torch.int32)
    o, lse = fa.fa_fwd_fp8(q8.to(DEV), k8.to(DEV), vt8.to(DEV), causal, scale, qd, kd, vd,
                           k_start=None if kst is None else kst.to(DEV),
                           k_end=None if ken is None else ken.to(DEV))
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    ro, rl = orc.fwd_fp8(q8, k8, vt8, causal, scale, qd, kd, vd, k_start=kst, k_end=ken)
    check_lse(to_np(lse), rl)
    rep = Hq // Hkv
    heads = list(range(Hq)) if heads is None else list(heads)
    # the bound needs P and V of the dequantised problem (for the checked heads)
    qx = (orc.decode_e4m3(q8) * qd)[:, heads]
    kx = (orc.decode_e4m3(k8) * kd)[:, [h // rep for h in heads]]
    vx = (np.swapaxes(orc.decode_e4m3(vt8), -1, -2) * vd)[:, [h // rep for h in heads]]
    P = orc.probs(qx, kx, vx, causal, scale, k_start=kst, k_end=ken)  # [B,len(heads),Sq,Sk]
    ro = ro[:, heads]
    A = np.zeros_like(ro)     # sum_j P_ij |v_jc - O_ic|
    Bsum = np.zeros_like(ro)  # sum over visible j of |v_jc - O_ic|
    for b in range(B):
        for h in range(len(heads)):
            vh = vx[b, h]
            for i0 in range(0, Sq, 64):
                dv_ = np.abs(vh[None, :, :] - ro[b, h, i0:i0 + 64, None, :])  # [rows, Sk, d]
                Pb = P[b, h, i0:i0 + 64]
                A[b, h, i0:i0 + 64] = np.einsum("ij,ijc->ic", Pb, dv_)
                Bsum[b, h, i0:i0 + 64] = np.einsum("ij,ijc->ic", (Pb > 0).astype(np.float64), dv_)
    bound = (2.0 ** -4 * A + 2.0 ** -10 * Bsum) / (1 - 2.0 ** -4) + 2.0 ** -8 * np.abs(ro) + 1e-4
    got_all = to_np(o)
    assert np.all(np.isfinite(got_all))
    got = got_all[:, heads]
    err = np.abs(got - ro)
    worst = float((err / bound).max())
    assert worst <= 1.0, f"O error exceeds the e4m3 weight-rounding bound by {worst:.3f}x"
    return float(err.max()), float(np.sqrt((err ** 2).mean()))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_within_rounding_bound(causal):
    _case(1, 4, 2, 384, 384, causal, seed=81)


def test_fp8_forward_large_logits_max_growth():
    # Q x 8: raw logits reach about +-100, so a row's max keeps growing across
    # key tiles, past the 2^8 rescale threshold (O and l rescaled) and below
    # it (weights up to 256 against the stale max)
    _case(1, 2, 2, 512, 1024, True, seed=84, qmul=8.0)
    _case(1, 2, 1, 300, 304, False, seed=85, qmul=8.0)


def test_fp8_forward_rectangular_interval_and_slots():
    _case(2, 3, 3, 200, 512, False, seed=82, ks=[0, 100], ke=[512, 333])
    _case(1, 2, 2, 130, 300 // 16 * 16, True, seed=83)


def test_fp8_forward_persistent_many_units():
    # 64 heads x 5 units of two 128-row tiles = 320 units over the CTAs (one
    # per SM): every CTA walks two or three units, carrying its barrier phases,
    # Q reloads and O hand-over across them.  Heads 24-63 have their light
    # units in the second and third walk; all rows of four of them are held
    # to the bound, and every head's LSE is checked.
    _case(1, 64, 64, 1280, 1280, True, seed=86, qmul=8.0, heads=[0, 31, 47, 63])


def test_fp8_forward_bench_workload_sampled_rows():
    # The causal 8k workload the bench times (B=2 H=16 S=8192, Q x 8, batch
    # row 0 keys 0..63 padded, so its first 64 query rows see no key),
    # quantised per tensor: sampled rows, including the empty ones, are held
    # to the element-wise bound and the LSE tolerance.
    w = workloads.make("prefill_8k_masked")
    t = w.tensors
    q8, qd = _quant(t["q"])
    k8, kd = _quant(t["k"])
    v8, vd = _quant(t["v"])
    vt8 = v8.transpose(-1, -2).contiguous()
    kst, ken = t["k_start"], t["k_end"]
    o, lse = fa.fa_fwd_fp8(q8.to(DEV), k8.to(DEV), vt8.to(DEV), True, w.scale, qd, kd, vd,
                           k_start=kst.to(DEV), k_end=ken.to(DEV))
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    B, Hq, S, d = t["q"].shape
    Hkv = t["k"].shape[1]
    must = [0, 63, 64, 65, 127, 128, 4095, S - 1, S + 5, 15 * S + 8000, (Hq + 3) * S + 64]
    rows = np.array(sorted(set(must) | set(
        int(x) for x in np.random.default_rng(87).integers(0, B * Hq * S, size=40))), np.int64)
    qx = orc.decode_e4m3(q8) * qd
    kx = orc.decode_e4m3(k8) * kd
    vx = np.swapaxes(orc.decode_e4m3(vt8), -1, -2) * vd
    ro, rl = orc.fwd(qx, kx, vx, True, w.scale, k_start=kst, k_end=ken, rows=rows)
    got_o = to_np(o).reshape(-1, d)[rows]
    check_lse(to_np(lse).reshape(-1)[rows], rl)
    assert np.all(np.isfinite(got_o))
    rep = Hq // Hkv
    for n, r in enumerate(rows):
        b, h, i = int(r) // (Hq * S), (int(r) // S) % Hq, int(r) % S
        klo, khi = int(kst[b]), min(int(ken[b]), i + 1)  # causal, Sq == Sk
        bound = 2.0 ** -8 * np.abs(ro[n]) + 1e-4
        if khi > klo:
            kk = kx[b, h // rep, klo:khi]
            vv = vx[b, h // rep, klo:khi]
            s = kk @ qx[b, h, i] * w.scale
            pr = np.exp(s - s.max())
            pr /= pr.sum()
            dv_ = np.abs(vv - ro[n][None, :])
            bound = bound + (2.0 ** -4 * (pr @ dv_) + 2.0 ** -10 * dv_.sum(axis=0)) / (1 - 2.0 ** -4)
        worst = float((np.abs(got_o[n] - ro[n]) / bound).max())
        assert worst <= 1.0, f"row {int(r)}: O error exceeds the e4m3 bound by {worst:.3f}x"
