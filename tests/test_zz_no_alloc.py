"""fa_decode_noalloc: the decode entry point for callers that cannot allocate
device scratch (their interface has no workspace slot, or allocating is not
allowed or too costly where they run).  It must give the same results as
fa_decode with a caller workspace, call after call, agree with the FP64
oracle, and refuse problems larger than its built-in scratch before doing any
device work.

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
from oracle import oracle as orc
from tests.parity import LSE_TOL, O_TOL, check_lse, check_o, sample_rows, to_np

# A problem whose decode workspace sits just under the built-in scratch: with
# Sk_max = 1024 the split plan uses 8 splits of 128 keys, so the workspace is
# B*Hq*8 rows of d fp32 partial outputs plus their fp32 LSEs, and the LSEs
# occupy the last bytes of the array.  One more batch row goes over the limit.
NEAR = dict(B=254, Hq=64, Hkv=1, Sk_max=1024, d=128)


def _noalloc(lib, B, Hq, Hkv, Sk_max, d):
    P = ctypes.c_void_p
    return lib.fa_decode_noalloc(P(16), P(16), P(16), P(16), None, P(16), B, Hq, Hkv, Sk_max, d,
                                 ctypes.c_float(0.1), None)


def test_noalloc_rejects_oversized_problem_before_device_work():
    fabuild.build()
    lib = fa.load_library()
    need = fa.fa_decode_workspace_size(64, 64, 1 << 20, 128)
    assert need > fa.DECODE_NOALLOC_MAX_SCRATCH_BYTES
    assert _noalloc(lib, 64, 64, 8, 1 << 20, 128) == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error_detail()


def test_noalloc_limit_boundary_on_the_host():
    fabuild.build()
    lib = fa.load_library()
    limit = fa.DECODE_NOALLOC_MAX_SCRATCH_BYTES
    n = NEAR
    need = fa.fa_decode_workspace_size(n["B"], n["Hq"], n["Sk_max"], n["d"])
    assert need <= limit and limit - need <= 8192, (need, limit)
    over = fa.fa_decode_workspace_size(n["B"] + 1, n["Hq"], n["Sk_max"], n["d"])
    assert over > limit
    assert _noalloc(lib, n["B"] + 1, n["Hq"], n["Hkv"], n["Sk_max"], n["d"]) == fa.FA_ERR_WORKSPACE
    assert str(over).encode() in lib.fa_last_error_detail()


def _compare(q, k, v, sl, scale, t, lens, rows=None):
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
    # and against the FP64 oracle (all rows, or the sampled ones)
    sl_cpu = torch.tensor(lens, dtype=torch.int32)
    B, Hq, _, d = q.shape
    ro, rl = orc.decode(t["q"], t["k"], t["v"], sl_cpu, scale, rows=rows)
    if rows is None:
        check_o(a, ro)
        check_lse(la, rl[:, :, 0])
    else:
        check_o(a.reshape(B * Hq, d)[rows], ro)
        check_lse(la.reshape(B * Hq)[rows], rl)


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
        _compare(q, k, v, sl, scale, t, lens)


@pytest.mark.gpu
def test_noalloc_just_under_the_scratch_limit():
    # the largest workspace this test can size just below the limit: every
    # split slot up to the end of the array is written and read
    fabuild.build()
    n = NEAR
    d = n["d"]
    t = workloads.random_qkv(n["B"], n["Hq"], n["Hkv"], 1, n["Sk_max"], d, seed=33)
    g = np.random.default_rng(33)
    lens = [int(x) for x in g.integers(1, n["Sk_max"] + 1, size=n["B"])]
    lens[-1] = n["Sk_max"]  # the last row fills all 8 splits at the end of the array
    lens[0] = 0             # and an empty row: O = 0, LSE = -inf
    q, k, v = (t[x].to("cuda") for x in ("q", "k", "v"))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    rows = sample_rows(n["B"], n["Hq"], 1, 48, seed=33,
                       must=(0, n["Hq"] - 1, (n["B"] - 1) * n["Hq"], n["B"] * n["Hq"] - 1))
    scale = 1.0 / math.sqrt(d)
    for _ in range(2):  # two calls in a row on the same shared scratch
        _compare(q, k, v, sl, scale, t, lens, rows=rows)
