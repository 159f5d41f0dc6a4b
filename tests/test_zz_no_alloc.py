"""fa_decode_noalloc: the decode entry point for callers that cannot allocate
device scratch (their interface has no workspace slot, or allocating is not
allowed or too costly where they run).  It must give the same results as
fa_decode with a caller workspace, call after call, and must refuse problems
larger than its built-in scratch before doing any device work.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import build as fabuild
from io_aware_exact_tcgen05_gb300 import workloads
from tests.parity import LSE_TOL, O_TOL, to_np


def test_noalloc_rejects_oversized_problem_before_device_work():
    fabuild.build()
    lib = fa.load_library()
    need = fa.fa_decode_workspace_size(64, 64, 1 << 20, 128)
    assert need > fa.DECODE_NOALLOC_MAX_SCRATCH_BYTES
    P = ctypes.c_void_p
    st = lib.fa_decode_noalloc(P(16), P(16), P(16), P(16), None, P(16), 64, 64, 8, 1 << 20, 128,
                               ctypes.c_float(0.1), None)
    assert st == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error_detail()


@pytest.mark.gpu
def test_noalloc_matches_fa_decode_on_consecutive_calls():
    fabuild.build()
    dev = "cuda"
    d = 128
    scale = 1.0 / math.sqrt(d)
    cases = [
        # two different problems back to back: the second call must not see
        # anything the first one left in the shared scratch
        (workloads.random_qkv(4, 32, 8, 1, 4096, d, seed=31), [4096, 1, 2049, 3000]),
        (workloads.random_qkv(3, 8, 2, 1, 1500, d, seed=32), [700, 1500, 64]),
    ]
    for t, lens in cases:
        q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        o_ref, lse_ref = fa.fa_decode(q, k, v, sl, scale)
        o_na, lse_na = fa.fa_decode_noalloc(q, k, v, sl, scale)
        torch.cuda.synchronize()
        assert fa.fa_device_status()[0] == 0
        a, b = to_np(o_na), to_np(o_ref)
        assert np.all(np.isfinite(a))
        assert float(np.abs(a - b).max()) <= O_TOL
        la, lb = to_np(lse_na), to_np(lse_ref)
        assert np.array_equal(la == -np.inf, lb == -np.inf)
        live = lb > -np.inf
        assert float(np.abs(la[live] - lb[live]).max()) <= LSE_TOL
