"""The backward walks its units key-tile-major inside groups of (batch, KV
head) pairs once all pairs' dQ accumulators and Q/dO tiles exceed twice L2.
These shapes are large enough in pair count (320+ MB) to be split into
several groups with a partial last one, yet short enough in sequence length
for the FP64 oracle: batch rows are independent in the backward, so the
first, a middle and the last batch row (the partial group) are checked in
full."""
import math

import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("B,Hq,Hkv,S", [
    (41, 16, 16, 512),  # 656 pairs: five groups of 128 and one of 16
    (20, 32, 8, 512),   # grouped heads: 160 pairs, groups of 112 and 48
])
def test_grouped_backward_rows(B, Hq, Hkv, S):
    d = 128
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=131, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, True, scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, True, scale)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    for b in (0, B // 2, B - 1):
        sl = slice(b, b + 1)
        sub = {n: t[n][sl] for n in ("q", "k", "v", "dout")}
        ro, rl = orc.fwd(sub["q"], sub["k"], sub["v"], True, scale)
        check_o(to_np(o[sl]), ro)
        check_lse(to_np(lse[sl]), rl)
        rq, rk, rv = orc.bwd(sub["q"], sub["k"], sub["v"], sub["dout"], True, scale)
        check_grad(to_np(dq[sl]), rq, f"dQ[{b}]")
        check_grad(to_np(dk[sl]), rk, f"dK[{b}]")
        check_grad(to_np(dv[sl]), rv, f"dV[{b}]")


def test_grouped_backward_packed_sequences():
    # 41 packed sequences x 16 KV heads = 656 pairs sized by the longest (512)
    # sequence: five groups of 128 pairs and one of 16.  Lengths are ragged,
    # so many units of a group are partial or empty.
    nseq, H, d = 41, 16, 128
    g = torch.Generator().manual_seed(141)
    lens = torch.randint(64, 513, (nseq,), generator=g)
    lens[0] = 512
    cu = torch.zeros(nseq + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    total = int(cu[-1])
    t = workloads.random_qkv(1, H, H, total, total, d, seed=142, with_dout=True)
    q, k, v, do = (t[n][0] for n in ("q", "k", "v", "dout"))  # [H, total, d]
    scale = 1.0 / math.sqrt(d)
    cud = cu.to(DEV)
    L = int(lens.max())
    o, lse = fa.fa_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cud, cud, L, L, True, scale)
    dq, dk, dv = fa.fa_bwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), o, do.to(DEV), lse, cud, cud,
                                  L, L, True, scale)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    for s in (0, nseq // 2, nseq - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        sub = {n: x[:, a:b][None].contiguous() for n, x in (("q", q), ("k", k), ("v", v),
                                                           ("dout", do))}
        ro, rl = orc.fwd(sub["q"], sub["k"], sub["v"], True, scale)
        check_o(to_np(o[:, a:b])[None], ro)
        check_lse(to_np(lse[:, a:b])[None], rl)
        rq, rk, rv = orc.bwd(sub["q"], sub["k"], sub["v"], sub["dout"], True, scale)
        check_grad(to_np(dq[:, a:b])[None], rq, f"dQ[seq {s}]")
        check_grad(to_np(dk[:, a:b])[None], rk, f"dK[seq {s}]")
        check_grad(to_np(dv[:, a:b])[None], rv, f"dV[seq {s}]")
