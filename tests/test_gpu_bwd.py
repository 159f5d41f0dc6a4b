"""GPU backward (fa_bwd through the C ABI, fed by fa_fwd's O and LSE) against
the FP64 oracle's gradients, element by element."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_grad, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(B, Hq, Hkv, Sq, Sk, d, causal, ks=None, ke=None, seed=0, q_mult=1.0):
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=seed, q_mult=q_mult, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    kst = torch.tensor(ks, dtype=torch.int32) if ks is not None else None
    ken = torch.tensor(ke, dtype=torch.int32) if ke is not None else None
    kd = None if kst is None else kst.to(DEV)
    ked = None if ken is None else ken.to(DEV)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, causal, scale, k_start=kd, k_end=ked)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal, scale, k_start=kd, k_end=ked)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    rq, rk, rv = orc.bwd(t["q"], t["k"], t["v"], t["dout"], causal, scale, k_start=kst,
                         k_end=ken)
    check_grad(to_np(dq), rq, "dQ")
    check_grad(to_np(dk), rk, "dK")
    check_grad(to_np(dv), rv, "dV")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 37, 128, 255, 300])
def test_bwd_shapes(d, causal, S):
    _run(1, 2, 2, S, S, d, causal, seed=S + d)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 2), (3, 1), (6, 6)])
def test_bwd_gqa(Hq, Hkv):
    _run(2, Hq, Hkv, 200, 200, 128, True, seed=Hq * 7 + Hkv)


@pytest.mark.parametrize("Sq,Sk", [(100, 333), (333, 100), (1, 300)])
def test_bwd_rectangular(Sq, Sk):
    _run(1, 2, 1, Sq, Sk, 128, True, seed=Sq * 3 + Sk)


def test_bwd_key_interval_masked_rows():
    _run(3, 4, 2, 300, 300, 128, True, ks=[64, 5, 50], ke=[300, 130, 50], seed=21)


def test_bwd_large_logits():
    _run(1, 2, 2, 513, 513, 128, True, seed=22, q_mult=8.0)


def test_bwd_many_tiles():
    _run(1, 2, 2, 1100, 1100, 128, True, seed=23)
