"""Stray-write checks: every output and workspace the kernels write is carved
out of a larger device buffer whose bytes all start as a sentinel, and after
the call every byte outside the region the contract says is written must
still hold the sentinel.  This stands in for a memory checker (which is not
available on these GPUs): an index or bound mistake that writes past a row,
a head or a tensor shows up here even when the results inside are right.

Shapes are odd on purpose (37, 129, 300 rows; ragged packed sequences; rows
that belong to no sequence), so that every kernel runs partial tiles."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENT = 0xA7     # sentinel byte
GUARD = 8192    # bytes of sentinel on each side of a carved tensor


class Carved:
    """A tensor of `shape`/`dtype` inside a sentinel-filled byte buffer."""

    def __init__(self, shape, dtype):
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * esize
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), SENT, dtype=torch.uint8, device=DEV)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def check_guards(self, what):
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.nbytes:]
        bad_lo = int((lo != SENT).sum())
        bad_hi = int((hi != SENT).sum())
        assert bad_lo == 0 and bad_hi == 0, (
            f"{what}: {bad_lo} bytes written before and {bad_hi} after the tensor")

    def untouched_rows(self, row_mask):
        """True per row (first axis after flattening all but the last) whose bytes
        still all hold the sentinel."""
        rows = self.buf[GUARD:GUARD + self.nbytes].view(row_mask.size, -1)
        return (rows == SENT).all(dim=1).cpu().numpy()


def _status_ok():
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)


FWD_BWD_CASES = [
    # B, Hq, Hkv, S, d, causal
    (1, 2, 2, 37, 64, True),
    (2, 4, 2, 129, 128, True),
    (1, 3, 1, 300, 128, False),
    (2, 2, 1, 300, 64, True),
]


@pytest.mark.parametrize("case", FWD_BWD_CASES)
def test_fwd_bwd_write_only_their_outputs(case):
    B, Hq, Hkv, S, d, causal = case
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=S + d, with_dout=True)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    o = Carved((B, Hq, S, d), torch.bfloat16)
    lse = Carved((B, Hq, S), torch.float32)
    fa.fa_fwd(q, k, v, causal, scale, o=o.t, lse=lse.t)
    torch.cuda.synchronize()
    _status_ok()
    o.check_guards("fwd O")
    lse.check_guards("fwd LSE")
    assert not np.any(o.untouched_rows(np.zeros(B * Hq * S))), "fwd left rows of O unwritten"
    dq = Carved((B, Hq, S, d), torch.bfloat16)
    dk = Carved((B, Hkv, S, d), torch.bfloat16)
    dv = Carved((B, Hkv, S, d), torch.bfloat16)
    ws = Carved((fa.fa_bwd_workspace_size(B, Hq, S, d),), torch.uint8)
    fa.fa_bwd(q, k, v, o.t, do, lse.t, causal, scale, dq=dq.t, dk=dk.t, dv=dv.t, workspace=ws.t)
    torch.cuda.synchronize()
    _status_ok()
    for c, n in ((dq, "dQ"), (dk, "dK"), (dv, "dV"), (ws, "workspace")):
        c.check_guards(f"bwd {n}")
    for c, n, rows in ((dq, "dQ", B * Hq * S), (dk, "dK", B * Hkv * S), (dv, "dV", B * Hkv * S)):
        assert not np.any(c.untouched_rows(np.zeros(rows))), f"bwd left rows of {n} unwritten"


def test_dropout_and_masked_write_only_their_outputs():
    B, Hq, Hkv, S, d = 2, 4, 2, 129, 128
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=7, with_dout=True)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    scale = 1.0 / math.sqrt(d)
    km = (torch.rand(B, S, generator=torch.Generator().manual_seed(7)) >= 0.3).to(DEV)
    for kw in (dict(key_mask=km), dict(dropout_p=0.25, seed=11, offset=3)):
        o = Carved((B, Hq, S, d), torch.bfloat16)
        lse = Carved((B, Hq, S), torch.float32)
        fa.fa_fwd(q, k, v, True, scale, o=o.t, lse=lse.t, **kw)
        dq = Carved((B, Hq, S, d), torch.bfloat16)
        dk = Carved((B, Hkv, S, d), torch.bfloat16)
        dv = Carved((B, Hkv, S, d), torch.bfloat16)
        ws = Carved((fa.fa_bwd_workspace_size(B, Hq, S, d),), torch.uint8)
        fa.fa_bwd(q, k, v, o.t, do, lse.t, True, scale, dq=dq.t, dk=dk.t, dv=dv.t,
                  workspace=ws.t, **kw)
        torch.cuda.synchronize()
        _status_ok()
        for c, n in ((o, "O"), (lse, "LSE"), (dq, "dQ"), (dk, "dK"), (dv, "dV"), (ws, "ws")):
            c.check_guards(f"{sorted(kw)[0]} {n}")


def test_varlen_writes_only_rows_of_its_sequences():
    # three sequences packed with 40 spare rows/keys after the last one that
    # belong to no sequence: the contract leaves those rows unwritten
    Hq, Hkv, d = 4, 2, 128
    lens_q = [37, 300, 129]
    lens_k = [37, 300, 200]
    spare = 40
    total_q, total_k = sum(lens_q) + spare, sum(lens_k) + spare
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(Hq, total_q, d, generator=g)).to(torch.bfloat16).to(DEV)
    k = (torch.randn(Hkv, total_k, d, generator=g)).to(torch.bfloat16).to(DEV)
    v = (torch.randn(Hkv, total_k, d, generator=g)).to(torch.bfloat16).to(DEV)
    do = (torch.randn(Hq, total_q, d, generator=g)).to(torch.bfloat16).to(DEV)
    scale = 1.0 / math.sqrt(d)
    o = Carved((Hq, total_q, d), torch.bfloat16)
    lse = Carved((Hq, total_q), torch.float32)
    fa.fa_fwd_varlen(q, k, v, cu_q.to(DEV), cu_k.to(DEV), max(lens_q), max(lens_k), True, scale,
                     o=o.t, lse=lse.t)
    dq = Carved((Hq, total_q, d), torch.bfloat16)
    dk = Carved((Hkv, total_k, d), torch.bfloat16)
    dv = Carved((Hkv, total_k, d), torch.bfloat16)
    ws = Carved((fa.fa_bwd_workspace_size(1, Hq, total_q, d),), torch.uint8)
    fa.fa_bwd_varlen(q, k, v, o.t, do, lse.t, cu_q.to(DEV), cu_k.to(DEV), max(lens_q),
                     max(lens_k), True, scale, dq=dq.t, dk=dk.t, dv=dv.t, workspace=ws.t)
    torch.cuda.synchronize()
    _status_ok()
    for c, n in ((o, "O"), (lse, "LSE"), (dq, "dQ"), (dk, "dK"), (dv, "dV"), (ws, "ws")):
        c.check_guards(f"varlen {n}")
    in_q = np.zeros(total_q, dtype=bool)
    in_q[: sum(lens_q)] = True
    in_k = np.zeros(total_k, dtype=bool)
    in_k[: sum(lens_k)] = True
    for c, n, mask in ((o, "O", in_q), (dk, "dK", in_k), (dv, "dV", in_k)):
        heads = c.t.shape[0]
        rows = np.tile(mask, heads)
        untouched = c.untouched_rows(rows)
        assert np.all(untouched[~rows]), f"varlen {n}: a row of no sequence was written"
        assert not np.any(untouched[rows]), f"varlen {n}: a row of a sequence was not written"


def test_decode_writes_only_its_outputs():
    B, Hq, Hkv, Smax, d = 3, 8, 2, 1500, 128
    t = workloads.random_qkv(B, Hq, Hkv, 1, Smax, d, seed=2)
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    sl = torch.tensor([1500, 1, 0], dtype=torch.int32, device=DEV)
    scale = 1.0 / math.sqrt(d)
    for noalloc in (False, True):
        o = Carved((B, Hq, 1, d), torch.bfloat16)
        lse = Carved((B, Hq), torch.float32)
        if noalloc:
            fa.fa_decode_noalloc(q, k, v, sl, scale, o=o.t, lse=lse.t)
            carved = ((o, "O"), (lse, "LSE"))
        else:
            ws = Carved((fa.fa_decode_workspace_size(B, Hq, Smax, d),), torch.uint8)
            fa.fa_decode(q, k, v, sl, scale, o=o.t, lse=lse.t, workspace=ws.t)
            carved = ((o, "O"), (lse, "LSE"), (ws, "workspace"))
        torch.cuda.synchronize()
        _status_ok()
        for c, n in carved:
            c.check_guards(f"decode{' noalloc' if noalloc else ''} {n}")
        assert not np.any(o.untouched_rows(np.zeros(B * Hq)))


def test_fp8_forward_writes_only_its_outputs():
    F8 = getattr(torch, "float8_e4m3fn", None)
    if F8 is None:
        pytest.skip("torch without float8_e4m3fn")
    B, Hq, Hkv, Sq, Sk, d = 1, 4, 2, 129, 144, 128
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=8)
    q8 = t["q"].float().to(F8).to(DEV)
    k8 = t["k"].float().to(F8).to(DEV)
    vt8 = t["v"].float().to(F8).transpose(-1, -2).contiguous().to(DEV)
    o = Carved((B, Hq, Sq, d), torch.bfloat16)
    lse = Carved((B, Hq, Sq), torch.float32)
    fa.fa_fwd_fp8(q8, k8, vt8, True, 1.0 / math.sqrt(d), 1.0, 1.0, 1.0, o=o.t, lse=lse.t)
    torch.cuda.synchronize()
    _status_ok()
    o.check_guards("fp8 O")
    lse.check_guards("fp8 LSE")
    assert not np.any(o.untouched_rows(np.zeros(B * Hq * Sq)))
