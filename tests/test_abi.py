"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/fa.h declares, validates arguments
before touching the device, and sizes its workspaces."""
import ctypes
import os
import re

import pytest

import io_aware_exact_tcgen05_gb300 as fa
from io_aware_exact_tcgen05_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_symbols_are_exported(lib):
    names = _declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_decode"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version(lib):
    assert "sm_103a" in fa.version()


P = ctypes.c_void_p


def _fwd(lib, q=16, k=16, v=16, o=16, lse=None, B=1, Hq=2, Hkv=2, Sq=8, Sk=8, d=128, scale=0.1):
    return lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, Sq, Sk, d, 0,
                      ctypes.c_float(scale), None, None, None)


def test_fwd_validation_before_any_device_call(lib):
    assert _fwd(lib, B=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, Sq=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, Hq=3, Hkv=2) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, o=18) == fa.FA_ERR_INVALID_ARG  # misaligned
    assert lib.fa_last_error_detail() == b"o is not 16-byte aligned"
    assert _fwd(lib, lse=8) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_last_error_detail() == b"lse is not 16-byte aligned"
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert b"scale" in lib.fa_last_error_detail()
    assert _fwd(lib, scale=-0.5) == fa.FA_ERR_INVALID_ARG
    assert b"must be finite and >= 0" in lib.fa_last_error_detail()
    assert _fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert b"head dimension 96" in lib.fa_last_error_detail()


def test_status_strings(lib):
    for s in range(6):
        assert lib.fa_status_string(s)


def test_workspace_sizes(lib):
    n = fa.fa_bwd_workspace_size(2, 16, 8192, 128)
    rows = 2 * 16 * 8192
    assert n >= rows * 128 * 4 + rows * 4
    assert n <= rows * 128 * 4 + rows * 4 + 512
    m = fa.fa_decode_workspace_size(32, 32, 32768, 128)
    assert m >= 32 * 32 * (32768 // 4096) * 129 * 4  # 4096-key splits for long caches
    assert m <= 32 * 32 * (32768 // 128) * 129 * 4 + 512
    assert fa.fa_decode_workspace_size(0, 1, 1, 128) == 0


def test_decode_workspace_too_small(lib):
    st = lib.fa_decode(P(16), P(16), P(16), P(16), None, P(16), 2, 4, 2, 100, 128,
                       ctypes.c_float(0.1), P(256), 1, None)
    assert st == fa.FA_ERR_WORKSPACE
    st = lib.fa_decode(P(16), P(16), P(16), P(16), None, None, 2, 4, 2, 100, 128,
                       ctypes.c_float(0.1), P(256), 1 << 20, None)
    assert st == fa.FA_ERR_INVALID_ARG


def test_bwd_workspace_too_small(lib):
    st = lib.fa_bwd(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                    1, 2, 2, 8, 8, 128, 1, ctypes.c_float(0.1), None, None, P(256), 16, None)
    assert st == fa.FA_ERR_WORKSPACE


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_library.__wrapped__(str(tmp_path / "nope.so")) if hasattr(
            fa.load_library, "__wrapped__") else _load_missing(tmp_path)


def _load_missing(tmp_path):
    saved = fa._lib
    fa._lib = None
    try:
        fa.load_library(str(tmp_path / "nope.so"))
    finally:
        fa._lib = saved


def _fwd_varlen(lib, cu_q=16, cu_k=16, nseq=2, max_q=8, max_k=8, total_q=16, total_k=16, Hq=2,
                Hkv=2, d=128, bits=None):
    return lib.fa_fwd_varlen(P(16), P(16), P(16), P(16), None, P(cu_q), P(cu_k), nseq, max_q,
                             max_k, total_q, total_k, Hq, Hkv, d, 1, ctypes.c_float(0.1),
                             P(bits), None)


def test_varlen_and_mask_validation_before_any_device_call(lib):
    assert _fwd_varlen(lib, cu_q=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, cu_k=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, cu_q=18) == fa.FA_ERR_INVALID_ARG  # not 4-byte aligned
    assert _fwd_varlen(lib, nseq=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, max_q=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, max_q=17) == fa.FA_ERR_INVALID_ARG  # longer than the packed total
    assert _fwd_varlen(lib, max_k=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, total_k=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_varlen(lib, d=80) == fa.FA_ERR_UNSUPPORTED
    assert _fwd_varlen(lib, bits=20) == fa.FA_ERR_INVALID_ARG  # bits not 16-byte aligned
    st = lib.fa_fwd_masked(P(16), P(16), P(16), P(16), None, 1, 2, 2, 8, 8, 128, 0,
                           ctypes.c_float(0.1), None, None, P(24), None)
    assert st == fa.FA_ERR_INVALID_ARG
    st = lib.fa_bwd_varlen(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                           None, P(16), 2, 8, 8, 16, 16, 2, 2, 128, 1, ctypes.c_float(0.1), None,
                           P(256), 1 << 20, None)
    assert st == fa.FA_ERR_INVALID_ARG
    st = lib.fa_bwd_masked(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                           1, 2, 2, 8, 8, 128, 1, ctypes.c_float(0.1), None, None, P(16),
                           P(256), 16, None)
    assert st == fa.FA_ERR_WORKSPACE
    assert lib.fa_pack_key_mask(P(16), P(16), 0, 8, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_pack_key_mask(None, P(16), 1, 8, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_pack_key_mask(P(16), P(20), 1, 8, None) == fa.FA_ERR_INVALID_ARG


def test_key_mask_words(lib):
    # 4 words (one 128-key tile) per started tile, so every tile's bits are one
    # aligned 16-byte load
    assert fa.fa_key_mask_words(1) == 4
    assert fa.fa_key_mask_words(128) == 4
    assert fa.fa_key_mask_words(129) == 8
    assert fa.fa_key_mask_words(8192) == 256
    assert fa.fa_key_mask_words(0) == 0


def test_dropout_validation_before_any_device_call(lib):
    def fwd(p):
        return lib.fa_fwd_dropout(P(16), P(16), P(16), P(16), None, 1, 2, 2, 8, 8, 128, 0,
                                  ctypes.c_float(0.1), None, None, None, ctypes.c_float(p), 1, 0,
                                  None)
    assert fwd(-0.1) == fa.FA_ERR_INVALID_ARG
    assert fwd(1.0) == fa.FA_ERR_INVALID_ARG
    assert fwd(float("nan")) == fa.FA_ERR_INVALID_ARG
    st = lib.fa_bwd_dropout(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                            1, 2, 2, 8, 8, 128, 1, ctypes.c_float(0.1), None, None, None,
                            ctypes.c_float(1.5), 1, 0, P(256), 1 << 20, None)
    assert st == fa.FA_ERR_INVALID_ARG


def test_fp8_validation_before_any_device_call(lib):
    def fwd8(d=128, Sk=128, qd=1.0):
        return lib.fa_fwd_fp8(P(16), P(16), P(16), P(16), None, 1, 2, 2, 8, Sk, d, 0,
                              ctypes.c_float(0.1), ctypes.c_float(qd), ctypes.c_float(1.0),
                              ctypes.c_float(1.0), None, None, None)
    assert fwd8(d=64) == fa.FA_ERR_UNSUPPORTED
    assert fwd8(Sk=100) == fa.FA_ERR_INVALID_ARG  # V^T rows must be whole 16-byte units
    assert fwd8(qd=0.0) == fa.FA_ERR_INVALID_ARG
    assert fwd8(qd=float("inf")) == fa.FA_ERR_INVALID_ARG
