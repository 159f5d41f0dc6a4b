"""Long sequences and full sizes: the forward and backward at S = 65536 and
131072 against the FP64 oracle on sampled rows, the bench's key-mask and
dropout rows on its full workload (sampled rows), and dK/dV
through identities that hold at any size:
  sum over keys of dV_j = sum over query rows (that see a key) of dO_i,
    because each row of P sums to 1;
  sum over keys of dK_j = scale * sum_i q_i * (sum_j dS_ij) = 0,
    because each row of dS sums to 0 (up to D_i taken from the bf16 O)."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_grad, check_lse, check_o, sample_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _must(S):
    return [0, 1, 127, 128, 129, S // 2, S - 129, S - 128, S - 1]


def test_forward_131072_sampled_rows():
    B, Hq, Hkv, S, d = 1, 2, 1, 131072, 128
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=111)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd(t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), True, scale)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    rows = sample_rows(B, Hq, S, 64, seed=112, must=_must(S) + [S + r for r in _must(S)])
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, scale, rows=rows)
    check_o(to_np(o).reshape(-1, d)[rows], ro)
    check_lse(to_np(lse).reshape(-1)[rows], rl)


def test_backward_65536_sampled_rows_and_identities():
    B, Hq, Hkv, S, d = 1, 2, 1, 65536, 128
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=113, with_dout=True)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    o, lse = fa.fa_fwd(q, k, v, True, scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, True, scale)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    rows = sample_rows(B, Hq, S, 24, seed=114, must=_must(S) + [S + 1, 2 * S - 1])
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, scale, rows=rows)
    check_o(to_np(o).reshape(-1, d)[rows], ro)
    check_lse(to_np(lse).reshape(-1)[rows], rl)
    rq = orc.bwd_dq_rows(t["q"], t["k"], t["v"], t["dout"], True, scale, rows)
    check_grad(to_np(dq).reshape(-1, d)[rows], rq, "dQ rows")
    # identities over all keys of the KV head (both query heads read it)
    dv_sum = to_np(dv)[0, 0].sum(axis=0)
    do_sum = to_np(do)[0].sum(axis=(0, 1))  # every causal row sees key 0
    dv_abs = np.abs(to_np(dv)[0, 0]).sum(axis=0)
    assert np.all(np.abs(dv_sum - do_sum) <= 1e-2 * dv_abs + 1e-2), \
        float(np.abs(dv_sum - do_sum).max())
    dk_sum = to_np(dk)[0, 0].sum(axis=0)
    dk_abs = np.abs(to_np(dk)[0, 0]).sum(axis=0)
    assert np.all(np.abs(dk_sum) <= 2e-2 * dk_abs), float((np.abs(dk_sum) / dk_abs).max())


@pytest.mark.parametrize("row_kind", ["key_mask", "dropout"])
def test_bench_widened_rows_full_size_sampled(row_kind):
    # The bench's widened rows on its own workload (B=2 H=16 S=8192, Q x 8,
    # batch row 0 keys 0..63 padded): a seeded mask hiding 10% of the keys, or
    # dropout p = 0.1; sampled rows (including rows that see no key) against
    # the oracle.
    w = workloads.make("prefill_8k_masked")
    t = w.tensors
    B, Hq, S, d = t["q"].shape
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    kst, ken = t["k_start"], t["k_end"]
    kw = {}
    okw = {}
    if row_kind == "key_mask":
        km = torch.rand(B, S, generator=torch.Generator().manual_seed(1)) >= 0.1
        kw = dict(key_mask=km.to(DEV))
        okw = dict(key_mask=km.numpy())
    else:
        kw = dict(dropout_p=0.1, seed=1, offset=0)
        okw = dict(dropout_p=0.1, seed=1, offset=0)
    o, lse = fa.fa_fwd(q, k, v, True, w.scale, k_start=kst.to(DEV), k_end=ken.to(DEV), **kw)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    rows = sample_rows(B, Hq, S, 48, seed=115,
                       must=[0, 63, 64, 65, 128, S - 1, 5 * S + 4000, (Hq + 7) * S + 8191])
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, w.scale, k_start=kst, k_end=ken, rows=rows,
                     **okw)
    check_o(to_np(o).reshape(-1, d)[rows], ro)
    check_lse(to_np(lse).reshape(-1)[rows], rl)


def test_bench_varlen_full_size_sampled():
    # The bench's packed lengths (the same seeded draw): 16 causal sequences of
    # 1024..8192 tokens, H = 16, d = 128, seeded values; sampled packed rows
    # against the oracle run on the row's own sequence.
    g = torch.Generator().manual_seed(1)
    torch.rand(2, 8192, generator=g)  # the bench draws its key mask first
    lens = torch.randint(1024, 8193, (16,), generator=g)
    cu = torch.zeros(17, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    total, H, d = int(cu[-1]), 16, 128
    scale = 1.0 / math.sqrt(d)
    gq = torch.Generator().manual_seed(2)
    vq, vk, vv = (torch.randn(H, total, d, generator=gq).bfloat16() for _ in range(3))
    cud = cu.to(DEV)
    L = int(lens.max())
    o, lse = fa.fa_fwd_varlen(vq.to(DEV), vk.to(DEV), vv.to(DEV), cud, cud, L, L, True, scale)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    rng = np.random.default_rng(116)
    picks = [(0, 0), (H - 1, total - 1), (3, int(cu[5])), (7, int(cu[9]) - 1)]
    picks += [(int(h), int(r)) for h, r in zip(rng.integers(0, H, 40), rng.integers(0, total, 40))]
    got_o, ref_o, got_l, ref_l = [], [], [], []
    for h, r in picks:
        s = int(np.searchsorted(cu.numpy(), r, side="right")) - 1
        a, b = int(cu[s]), int(cu[s + 1])
        sl = lambda x: x[h:h + 1, a:b][None]  # noqa: E731  [1, 1, len, d]
        ro, rl = orc.fwd(sl(vq), sl(vk), sl(vv), True, scale, rows=np.array([r - a]))
        got_o.append(to_np(o[h, r])[None])
        ref_o.append(ro)
        got_l.append(np.array([float(lse[h, r])]))
        ref_l.append(rl)
    check_o(np.concatenate(got_o), np.concatenate(ref_o))
    check_lse(np.concatenate(got_l), np.concatenate(ref_l))
