"""GPU forward (fa_fwd through the C ABI) against the FP64 oracle, element by
element, on seeded inputs that span several tiles and ragged tails."""
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


def _run(B, Hq, Hkv, Sq, Sk, d, causal, ks=None, ke=None, seed=0, q_mult=1.0, scale=None):
    t = workloads.random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=seed, q_mult=q_mult)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    kst = torch.tensor(ks, dtype=torch.int32) if ks is not None else None
    ken = torch.tensor(ke, dtype=torch.int32) if ke is not None else None
    o, lse = fa.fa_fwd(t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), causal, scale,
                       k_start=None if kst is None else kst.to(DEV),
                       k_end=None if ken is None else ken.to(DEV))
    torch.cuda.synchronize()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], causal, scale, k_start=kst, k_end=ken)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
    return o, lse


def test_small_noncausal_config_full():
    w = workloads.make("small_noncausal")
    q, k, v = (w.tensors[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.fa_fwd(q, k, v, False, w.scale)
    ro, rl = orc.fwd(w.tensors["q"], w.tensors["k"], w.tensors["v"], False, w.scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)


def test_worked_example_on_gpu():
    """Scores 1000, 1001, 999 with values 1, 3, 7 (FlashAttention_01 page, worked
    example): O = 2.870665 (bf16: 2.875), LSE = 1001.407606, no overflow."""
    q, k, v = workloads.worked_example_bf16()
    o, lse = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), False, 1.0)
    o = to_np(o)
    lse = to_np(lse)
    want = (math.exp(-1) + 3 + 7 * math.exp(-2)) / (math.exp(-1) + 1 + math.exp(-2))
    assert abs(o[0, 0, 0, 0] - want) <= 2e-2
    assert np.all(o[0, 0, 0, 1:] == 0.0)
    assert abs(lse[0, 0, 0] - (1001.0 + math.log(math.exp(-1) + 1 + math.exp(-2)))) <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 37, 127, 129, 255, 300])
def test_shapes_single_head(d, causal, S):
    _run(1, 2, 2, S, S, d, causal, seed=S)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (6, 2), (3, 1), (5, 5)])
def test_gqa_groups(Hq, Hkv):
    _run(2, Hq, Hkv, 200, 200, 128, True, seed=Hq * 10 + Hkv)


@pytest.mark.parametrize("Sq,Sk", [(100, 333), (333, 100), (1, 700), (64, 64), (256, 1024)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular(Sq, Sk, causal):
    _run(1, 2, 1, Sq, Sk, 128, causal, seed=Sq + Sk)


def test_key_interval_and_fully_masked_rows():
    # batch row 0: keys [64, 300); under causal, rows 0..63 see nothing
    # batch row 1: keys [5, 130); batch row 2: empty interval
    _run(3, 4, 2, 300, 300, 128, True, ks=[64, 5, 50], ke=[300, 130, 50], seed=7)
    _run(3, 4, 4, 130, 130, 64, False, ks=[0, 129, 3], ke=[1, 130, 4], seed=8)


def test_large_logits_no_overflow():
    # Q * 8 so raw logits reach ~+-100 (naive exp would overflow fp32 sums)
    _run(1, 2, 2, 513, 513, 128, True, seed=11, q_mult=8.0)
    _run(1, 2, 2, 257, 257, 64, False, seed=12, q_mult=30.0)


def _run_tensors(q, k, v, causal, scale):
    o, lse = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal, scale)
    torch.cuda.synchronize()
    ro, rl = orc.fwd(q, k, v, causal, scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,d", [(2, 2, 128), (4, 2, 64)])
def test_score_jumps_after_first_tile(causal, Hq, Hkv, d):
    # Later key blocks are scaled by powers of two (exact in bf16) so the
    # scores of a row jump by hundreds of log2 units well after its first
    # tile: the weights relative to the running max overflow and the kernel
    # must redo those tiles from the exact tile max.  The jumps land in both
    # halves of a tile (keys 200 and 330) and in a ragged last tile; rows
    # with a zero query see flat scores and never jump.
    t = workloads.random_qkv(1, Hq, Hkv, 613, 613, d, seed=21, q_mult=4.0)
    q, k, v = t["q"].float(), t["k"].float(), t["v"]
    k[:, :, 200:330] *= 8.0
    k[:, :, 330:600] *= 32.0
    k[:, :, 600:] *= 64.0
    q[:, :, 1::5] = 0.0
    _run_tensors(q.bfloat16(), k.bfloat16(), v, causal, 1.0 / math.sqrt(d))


def test_many_tiles_random_scale():
    _run(2, 2, 2, 1100, 1100, 128, True, seed=13, scale=0.05)


def test_zero_scale_gives_uniform_weights():
    # scale 0: O is the mean of the visible V rows and LSE = ln(#visible),
    # including the first tile of every row (no finite max from a score
    # change) and rows whose first tiles are fully masked
    B, H, S, d = 2, 2, 300, 128
    ks = [0, 200]
    _run(B, H, H, S, S, d, True, ks=ks, ke=[S, S], seed=61, scale=0.0)
    _run(B, H, H, S, S, 64, False, seed=62, scale=0.0)
