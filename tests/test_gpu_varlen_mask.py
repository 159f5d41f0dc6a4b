"""GPU parity for per-key boolean masks and packed ragged (varlen) sequences
(fa_fwd_masked / fa_bwd_masked / fa_fwd_varlen / fa_bwd_varlen through the C
ABI) against the FP64 oracle, element by element.

The cases span several 128-key tiles with ragged tails, tiles whose keys are
all hidden, rows that see no key, sequences without queries or without keys,
sequences with fewer queries than keys, GQA and both query-slot layouts."""
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


def _key_mask(rows, Sk, seed, drop):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(rows, Sk, generator=g) >= drop


def test_pack_key_mask_bits():
    m = _key_mask(3, 300, 1, 0.5)
    m[1] = False
    bits = fa.fa_pack_key_mask(m.to(DEV))
    torch.cuda.synchronize()
    words = bits.cpu().numpy().view(np.uint32)
    assert words.shape == (3, fa.fa_key_mask_words(300))
    for r in range(3):
        for j in range(words.shape[1] * 32):
            bit = (int(words[r, j // 32]) >> (j % 32)) & 1
            assert bit == (int(m[r, j]) if j < 300 else 0), (r, j)


MASK_CASES = [
    # B, Hq, Hkv, Sq, Sk, d, causal
    (2, 4, 2, 300, 300, 128, True),
    (2, 2, 2, 257, 400, 64, False),
    (1, 3, 1, 130, 130, 128, True),
    (2, 4, 4, 200, 520, 128, False),
]


@pytest.mark.parametrize("case", MASK_CASES)
def test_key_mask_fwd_bwd(case):
    B, Hq, Hkv, Sq, Sk, d, causal = case
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=31, with_dout=True)
    km = _key_mask(B, Sk, 32, 0.3)
    km[0, 128:256] = False       # a whole 128-key tile hidden
    km[-1, : min(Sk, 150)] = False  # causal rows near the start see nothing
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    kmd = km.to(DEV)
    o, lse = fa.fa_fwd(q, k, v, causal, scale, key_mask=kmd)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, causal, scale, key_mask=kmd)
    torch.cuda.synchronize()
    _status_ok()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], causal, scale, key_mask=km)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    rq, rk, rv = orc.bwd(t["q"], t["k"], t["v"], t["dout"], causal, scale, key_mask=km)
    check_grad(to_np(dq), rq, "dQ")
    check_grad(to_np(dk), rk, "dK")
    check_grad(to_np(dv), rv, "dV")
    # hidden keys get exactly zero gradient
    hidden = ~km.numpy()
    for b in range(B):
        assert np.all(to_np(dk[b])[:, hidden[b]] == 0.0)
        assert np.all(to_np(dv[b])[:, hidden[b]] == 0.0)


def test_key_mask_with_interval_and_prebuilt_bits():
    B, Hq, Hkv, S, d = 2, 2, 1, 260, 128
    t = workloads.random_qkv(B, Hq, Hkv, S, S, d, seed=33, with_dout=True)
    km = _key_mask(B, S, 34, 0.2)
    ks, ke = torch.tensor([10, 0], dtype=torch.int32), torch.tensor([260, 199], dtype=torch.int32)
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    bits = fa.fa_pack_key_mask(km.to(DEV))
    o, lse = fa.fa_fwd(q, k, v, True, 0.09, k_start=ks.to(DEV), k_end=ke.to(DEV), key_mask=bits)
    torch.cuda.synchronize()
    _status_ok()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, 0.09, k_start=ks, k_end=ke, key_mask=km)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)


def _packed(lengths_q, lengths_k, Hq, Hkv, d, seed):
    cu_q = np.concatenate([[0], np.cumsum(lengths_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lengths_k)]).astype(np.int32)
    t = workloads.random_qkv(1, Hq, Hkv, int(cu_q[-1]), int(cu_k[-1]), d, seed=seed,
                             with_dout=True)
    return cu_q, cu_k, {n: x[0].contiguous() for n, x in t.items()}


VARLEN_CASES = [
    # lengths_q, lengths_k, Hq, Hkv, d
    ([1, 130, 0, 257, 64, 300], [5, 130, 7, 257, 0, 400], 4, 2, 128),
    ([200, 129, 3], [200, 129, 3], 2, 2, 64),
    ([384, 1, 77], [384, 513, 77], 3, 1, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", VARLEN_CASES)
@pytest.mark.parametrize("masked", [False, True])
def test_varlen_fwd_bwd(case, causal, masked):
    lq, lk, Hq, Hkv, d = case
    cu_q, cu_k, t = _packed(lq, lk, Hq, Hkv, d, seed=41)
    total_k = int(cu_k[-1])
    km = _key_mask(1, total_k, 42, 0.25)[0] if masked else None
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "dout"))
    cq, ck = torch.from_numpy(cu_q).to(DEV), torch.from_numpy(cu_k).to(DEV)
    kmd = None if km is None else km.to(DEV)
    o, lse = fa.fa_fwd_varlen(q, k, v, cq, ck, max(lq), max(lk), causal, scale, key_mask=kmd)
    dq, dk, dv = fa.fa_bwd_varlen(q, k, v, o, do, lse, cq, ck, max(lq), max(lk), causal, scale,
                                  key_mask=kmd)
    torch.cuda.synchronize()
    _status_ok()
    ro, rl = orc.fwd_varlen(t["q"], t["k"], t["v"], cu_q, cu_k, causal, scale, key_mask=km)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    rq, rk, rv = orc.bwd_varlen(t["q"], t["k"], t["v"], t["dout"], cu_q, cu_k, causal, scale,
                                key_mask=km)
    # per sequence, so a small sequence is held to its own gradient scale
    for s in range(len(lq)):
        q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        if q1 > q0:
            check_grad(to_np(dq[:, q0:q1]), rq[:, q0:q1], f"dQ seq {s}")
        if k1 > k0:
            check_grad(to_np(dk[:, k0:k1]), rk[:, k0:k1], f"dK seq {s}")
            check_grad(to_np(dv[:, k0:k1]), rv[:, k0:k1], f"dV seq {s}")
        if q1 > q0 and k1 == k0:
            assert np.all(to_np(dq[:, q0:q1]) == 0.0)
        if k1 > k0 and q1 == q0:
            assert np.all(to_np(dk[:, k0:k1]) == 0.0) and np.all(to_np(dv[:, k0:k1]) == 0.0)


def test_varlen_equal_lengths_match_batched_kernel():
    B, H, S, d = 3, 2, 256, 128  # sequences start on 128-key tile boundaries
    t = workloads.random_qkv(B, H, H, S, S, d, seed=45)
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    ob, lb = fa.fa_fwd(q, k, v, True, 0.1)
    pack = lambda x: x.permute(1, 0, 2, 3).reshape(H, B * S, d).contiguous()  # noqa: E731
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV) * S
    ov, lv = fa.fa_fwd_varlen(pack(q), pack(k), pack(v), cu, cu, S, S, True, 0.1)
    torch.cuda.synchronize()
    _status_ok()
    # the same tiles in the same order: bit-identical
    assert torch.equal(ov, pack(ob))
    assert torch.equal(lv, lb.permute(1, 0, 2).reshape(H, B * S))
