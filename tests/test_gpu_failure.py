"""Failure detection without a GPU fault.  The library's self-test kernel
(fa_selftest_wait_timeout) waits, with the pipeline-wait helpers of the
attention kernels, on barriers that nothing arrives on: the first wait must
run out after its 1 s limit, record FA_ERR_TIMEOUT at its wait site in the
device status word and raise the abort flag; the second must give up on the
flag without a second record.  The kernel returns normally, so the context
stays usable: the status word clears and the next attention call is correct."""
import math

import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import workloads
from oracle import oracle as orc
from tests.parity import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
SELFTEST_SITE = 0x7E


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    st, word = fa.fa_device_status(clear=True)
    assert st == 0, hex(word)
    flags = fa.fa_selftest_wait_timeout()
    assert flags == [1, 1], flags
    st, word = fa.fa_device_status(clear=True)
    assert st == fa.FA_ERR_TIMEOUT
    assert word == (SELFTEST_SITE << 16) | 1, hex(word)
    st, word = fa.fa_device_status()
    assert st == 0 and word == 0, hex(word)
    # the next call runs normally and is correct
    t = workloads.random_qkv(1, 2, 2, 200, 200, 128, seed=3)
    scale = 1.0 / math.sqrt(128)
    o, lse = fa.fa_fwd(t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), True, scale)
    torch.cuda.synchronize()
    ro, rl = orc.fwd(t["q"], t["k"], t["v"], True, scale)
    check_o(to_np(o), ro)
    check_lse(to_np(lse), rl)
    st, word = fa.fa_device_status()
    assert st == 0, hex(word)
