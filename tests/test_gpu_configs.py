"""Parity at the full sizes of the five workloads the measurements use, in the
launch configuration bench.py times (same generators, same calls).

The oracle cannot recompute a full S=8192 problem in a test, so each check
samples: forward rows (always including batch row 0's fully masked rows and
the first rows that see keys again), whole heads for the backward (the oracle
recomputes every statistic of that head itself), and every (batch, head) row
of the decode."""

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_grad, check_lse, check_o, sample_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _fwd_rows(w, o, lse, rows):
    t = w.tensors
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], w.causal, w.scale, k_start=t.get("k_start"),
                     k_end=t.get("k_end"), rows=rows)
    go = to_np(o).reshape(-1, w.d)[rows]
    gl = to_np(lse).reshape(-1)[rows]
    check_o(go, ro)
    check_lse(gl, rl)


def _run_fwd(w):
    t = w.tensors
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    ks = t.get("k_start")
    ke = t.get("k_end")
    o, lse = fa.fa_fwd(q, k, v, w.causal, w.scale,
                       k_start=None if ks is None else ks.to(DEV),
                       k_end=None if ke is None else ke.to(DEV))
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    return q, k, v, o, lse


def _head_grads(w, b, h):
    """Oracle dQ, dK, dV of query head h (and its KV head) of batch row b."""
    t = w.tensors
    hk = h // (w.Hq // w.Hkv)
    sl = lambda x, hh: x[b:b + 1, hh:hh + 1]  # noqa: E731
    ks = t.get("k_start")
    ke = t.get("k_end")
    return orc.bwd(sl(t["q"], h), sl(t["k"], hk), sl(t["v"], hk), sl(t["dout"], h), w.causal,
                   w.scale, k_start=None if ks is None else ks[b:b + 1],
                   k_end=None if ke is None else ke[b:b + 1])


def test_small_noncausal_full():
    w = workloads.make("small_noncausal")
    _, _, _, o, lse = _run_fwd(w)
    ro, rl = orc.fwd(w.tensors["q"], w.tensors["k"], w.tensors["v"], False, w.scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)


@pytest.mark.parametrize("name", ["prefill_2k", "prefill_8k_masked"])
def test_prefill_fwd_bwd(name):
    w = workloads.make(name)
    q, k, v, o, lse = _run_fwd(w)
    must = list(range(0, 70)) + list(range(w.Sq - 3, w.Sq))  # batch row 0, head 0
    must += [(w.B * w.Hq - 1) * w.Sq + i for i in (0, 1, 127, 128, w.Sq - 1)]
    _fwd_rows(w, o, lse, sample_rows(w.B, w.Hq, w.Sq, 600, seed=1, must=must))
    t = w.tensors
    ks = t.get("k_start")
    ke = t.get("k_end")
    do = t["dout"].to(DEV)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale,
                           k_start=None if ks is None else ks.to(DEV),
                           k_end=None if ke is None else ke.to(DEV))
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    for b, h in ((0, 0), (w.B - 1, w.Hq - 1)):
        rq, rk, rv = _head_grads(w, b, h)
        hk = h // (w.Hq // w.Hkv)
        check_grad(to_np(dq[b:b + 1, h:h + 1]), rq, f"dQ[b={b},h={h}]")
        check_grad(to_np(dk[b:b + 1, hk:hk + 1]), rk, f"dK[b={b},hk={hk}]")
        check_grad(to_np(dv[b:b + 1, hk:hk + 1]), rv, f"dV[b={b},hk={hk}]")
        if ks is not None and int(ks[b]) > 0:
            # rows that see no key get exactly zero gradient
            n = min(int(ks[b]), w.Sq)
            assert np.all(to_np(dq[b, h, :n]) == 0.0)


def test_gqa_fwd():
    w = workloads.make("gqa_4k")
    _, _, _, o, lse = _run_fwd(w)
    must = [(b * w.Hq + h) * w.Sq + i for b in (0, w.B - 1) for h in range(w.Hq)
            for i in (0, w.Sq - 1)]
    _fwd_rows(w, o, lse, sample_rows(w.B, w.Hq, w.Sq, 500, seed=2, must=must))


def test_decode_ragged_all_rows():
    w = workloads.make("decode_ragged")
    t = w.tensors
    q, kc, vc, sl = (t[n].to(DEV) for n in ("q", "k", "v", "seqlens_k"))
    o, lse = fa.fa_decode(q, kc, vc, sl, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status()[0] == 0
    ro, rl = orc.decode(t["q"], t["k"], t["v"], t["seqlens_k"], w.scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl[:, :, 0])
