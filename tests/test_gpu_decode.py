"""GPU decode (fa_decode through the C ABI) against the FP64 oracle."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(B, Hq, Hkv, Smax, d, lens, seed=0, q_mult=1.0, scale=None):
    t = workloads.random_qkv(B, Hq, Hkv, 1, Smax, d, seed=seed, q_mult=q_mult)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    sl = torch.tensor(lens, dtype=torch.int32)
    o, lse = fa.fa_decode(t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), sl.to(DEV), scale)
    torch.cuda.synchronize()
    ro, rl = orc.decode(t["q"], t["k"], t["v"], sl, scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl[:, :, 0])
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (32, 8), (6, 2), (16, 1), (3, 1)])
def test_decode_groups(d, Hq, Hkv):
    _run(3, Hq, Hkv, 1500, d, [1500, 1, 777], seed=Hq + Hkv + d)


@pytest.mark.parametrize("Smax", [1, 63, 64, 65, 511, 513, 4096])
def test_decode_lengths(Smax):
    lens = [Smax, max(1, Smax // 2), max(1, Smax - 1), 1]
    _run(4, 8, 2, Smax, 128, lens, seed=Smax)


def test_decode_empty_and_clamped_lengths():
    # 0 -> O = 0, LSE = -inf; > Smax and < 0 are clamped
    t = workloads.random_qkv(3, 4, 2, 1, 300, 128, seed=5)
    sl = torch.tensor([0, 1000, -5], dtype=torch.int32)
    o, lse = fa.fa_decode(t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), sl.to(DEV),
                          1 / math.sqrt(128))
    ro, rl = orc.decode(t["q"], t["k"], t["v"], torch.tensor([0, 300, 0]), 1 / math.sqrt(128))
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl[:, :, 0])


def test_decode_large_logits():
    _run(2, 8, 2, 3000, 128, [3000, 2999], seed=9, q_mult=8.0)


def test_decode_zero_scale_gives_uniform_weights():
    # the first finite max of a split is taken even when every score is 0
    _run(3, 8, 2, 5000, 128, [5000, 1, 4097], seed=71, scale=0.0)
