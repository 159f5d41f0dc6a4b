"""The persistent forward and backward kernels walk several work units per CTA
(one CTA per SM), carrying barrier phases across units and skipping units
without work.  These cases have many more units than SMs, with empty and
partial key intervals mixed in, and are checked against the FP64 oracle in
full."""
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


def _intervals(B, Sk, seed):
    """Per-batch key intervals: every fifth batch row empty, others random."""
    g = np.random.default_rng(seed)
    ks, ke = [], []
    for b in range(B):
        if b % 5 == 3:
            a = int(g.integers(0, Sk))
            ks.append(a)
            ke.append(a)  # empty interval: every row of the batch row sees nothing
        else:
            a = int(g.integers(0, Sk // 3))
            e = int(g.integers(a + 1, Sk + 1))
            ks.append(a)
            ke.append(e)
    return torch.tensor(ks, dtype=torch.int32), torch.tensor(ke, dtype=torch.int32)


@pytest.mark.parametrize("B,Hq,Hkv,S,d,causal", [
    (40, 8, 4, 260, 64, True),    # grouped heads: two heads per unit
    (48, 3, 1, 200, 64, False),   # odd group: two row blocks per unit
    (24, 4, 4, 300, 128, True),
])
def test_many_units_per_cta_fwd_bwd(B, Hq, Hkv, S, d, causal):
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=91, with_dout=True)
    ks, ke = _intervals(B, S, 92)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, causal, scale, k_start=ks.to(DEV), k_end=ke.to(DEV))
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal, scale, k_start=ks.to(DEV),
                           k_end=ke.to(DEV))
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], causal, scale, k_start=ks, k_end=ke)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    rq, rk, rv = orc.bwd(t["q"], t["k"], t["v"], t["dout"], causal, scale, k_start=ks, k_end=ke)
    # per batch row, so rows with small gradients are held to their own scale
    for b in range(B):
        check_grad(to_np(dq[b]), rq[b], f"dQ[{b}]")
        check_grad(to_np(dk[b]), rk[b], f"dK[{b}]")
        check_grad(to_np(dv[b]), rv[b], f"dV[{b}]")
        if int(ke[b]) <= int(ks[b]):
            assert np.all(to_np(dq[b]) == 0.0) and np.all(to_np(dk[b]) == 0.0)
