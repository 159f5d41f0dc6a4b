"""GB300-native exact tiled attention: thin Python binding over libfa.so.

Every function here only marshals arguments (device pointers, sizes, the
current CUDA stream) into the C ABI declared in ``include/fa.h``; all of the
attention arithmetic runs in the library's sm_103a kernels.  PyTorch is used
only to allocate device memory and to provide streams.  There is no CPU or
PyTorch fallback: if ``libfa.so`` is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5

EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_decode", "fa_decode_workspace_size",
            "fa_decode_noalloc", "fa_fwd_masked", "fa_bwd_masked", "fa_fwd_varlen",
            "fa_bwd_varlen", "fa_fwd_dropout", "fa_bwd_dropout", "fa_key_mask_words",
            "fa_pack_key_mask", "fa_fwd_fp8", "fa_device_status", "fa_selftest_wait_timeout",
            "fa_profile_next_launch", "fa_status_string", "fa_last_error_detail", "fa_version")

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status}: {detail}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libfa.so (build it first with ``io_aware_exact_tcgen05_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfa.so not found at {path}: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P]
    lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, Z, P]
    lib.fa_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P, Z, P]
    lib.fa_decode_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
    lib.fa_fwd_masked.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P]
    lib.fa_bwd_masked.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P, Z,
                                  P]
    lib.fa_fwd_varlen.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P]
    lib.fa_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P,
                                  P, Z, P]
    U64, U32 = ctypes.c_ulonglong, ctypes.c_uint
    lib.fa_fwd_dropout.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, F, U64, U32, P]
    lib.fa_bwd_dropout.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, F,
                                   U64, U32, P, Z, P]
    lib.fa_fwd_dropout.restype = I
    lib.fa_bwd_dropout.restype = I
    lib.fa_fwd_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, F, F, P, P, P]
    lib.fa_fwd_fp8.restype = I
    lib.fa_key_mask_words.argtypes = [I]
    lib.fa_key_mask_words.restype = Z
    lib.fa_pack_key_mask.argtypes = [P, P, I, I, P]
    for f in (lib.fa_fwd_masked, lib.fa_bwd_masked, lib.fa_fwd_varlen, lib.fa_bwd_varlen,
              lib.fa_pack_key_mask):
        f.restype = I
    lib.fa_decode_noalloc.restype = I
    lib.fa_bwd_workspace_size.argtypes = [I, I, I, I]
    lib.fa_bwd_workspace_size.restype = Z
    lib.fa_decode_workspace_size.argtypes = [I, I, I, I]
    lib.fa_decode_workspace_size.restype = Z
    lib.fa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
    for f in (lib.fa_fwd, lib.fa_bwd, lib.fa_decode, lib.fa_device_status):
        f.restype = I
    lib.fa_selftest_wait_timeout.argtypes = [P, P]
    lib.fa_selftest_wait_timeout.restype = I
    lib.fa_profile_next_launch.argtypes = [P, P]
    lib.fa_profile_next_launch.restype = I
    lib.fa_status_string.argtypes = [I]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_error_detail.restype = ctypes.c_char_p
    lib.fa_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != FA_OK:
        detail = _lib.fa_last_error_detail().decode()
        raise FAError(status, where, detail or _lib.fa_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def fa_key_mask_words(Sk: int) -> int:
    return int(load_library().fa_key_mask_words(Sk))


def fa_pack_key_mask(mask, stream=None):
    """Visibility bit words [rows, fa_key_mask_words(Sk)] (int32 storage of the
    uint32 words) from a bool/uint8 CUDA mask [rows, Sk], via fa_pack_key_mask."""
    lib = load_library()
    if not isinstance(mask, torch.Tensor) or not mask.is_cuda:
        raise TypeError("mask must be a CUDA tensor")
    if mask.dtype not in (torch.bool, torch.uint8) or not mask.is_contiguous() or mask.dim() != 2:
        raise ValueError("mask must be a contiguous 2-D bool or uint8 tensor")
    rows, Sk = mask.shape
    bits = torch.empty(rows, fa_key_mask_words(Sk), dtype=torch.int32, device=mask.device)
    _check(lib.fa_pack_key_mask(_ptr(mask), _ptr(bits), rows, Sk, _stream(stream)),
           "fa_pack_key_mask")
    return bits


def _mask_bits(key_mask, rows, Sk, stream):
    """Bit words for a key mask given as bools [rows, Sk] (packed on the
    device) or as bit words already; None when there is no mask."""
    if key_mask is None:
        return None
    if key_mask.dtype in (torch.bool, torch.uint8):
        if tuple(key_mask.shape) != (rows, Sk):
            raise ValueError(f"key_mask must be [{rows}, {Sk}], got {tuple(key_mask.shape)}")
        return fa_pack_key_mask(key_mask.contiguous(), stream)
    _need(key_mask, "key_mask bits", torch.int32, 2)
    if tuple(key_mask.shape) != (rows, fa_key_mask_words(Sk)):
        raise ValueError("key_mask bit words have the wrong shape")
    return key_mask


def fa_fwd(q, k, v, causal: bool, scale: float, k_start=None, k_end=None, o=None, lse=None,
           stream=None, key_mask=None, dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """O, LSE = attention(q, k, v) via the library's fa_fwd (see include/fa.h).
    q [B,Hq,Sq,d], k/v [B,Hkv,Sk,d] bf16 CUDA tensors; k_start/k_end optional
    int32 [B] CUDA tensors; key_mask optional [B, Sk] bool CUDA tensor (or its
    fa_pack_key_mask words), giving fa_fwd_masked.  dropout_p > 0 (taken as
    float32) gives fa_fwd_dropout with the given seed and offset.
    Returns (o, lse)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Hq, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    for t, n in ((k_start, "k_start"), (k_end, "k_end")):
        if t is not None:
            _need(t, n, torch.int32, 1)
    bits = _mask_bits(key_mask, B, Sk, stream)
    if dropout_p > 0.0:
        st = lib.fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq,
                                Sk, d, int(bool(causal)), float(scale), _ptr(k_start),
                                _ptr(k_end), _ptr(bits), float(dropout_p), int(seed),
                                int(offset), _stream(stream))
        _check(st, "fa_fwd_dropout")
    elif bits is None:
        st = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, d,
                        int(bool(causal)), float(scale), _ptr(k_start), _ptr(k_end),
                        _stream(stream))
        _check(st, "fa_fwd")
    else:
        st = lib.fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk,
                               d, int(bool(causal)), float(scale), _ptr(k_start), _ptr(k_end),
                               _ptr(bits), _stream(stream))
        _check(st, "fa_fwd_masked")
    return o, lse


def _need8(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    f8 = getattr(torch, "float8_e4m3fn", None)
    if t.dtype not in tuple(x for x in (f8, torch.uint8) if x is not None):
        raise TypeError(f"{name} must hold e4m3 bytes (float8_e4m3fn or uint8), got {t.dtype}")
    if not t.is_contiguous() or t.dim() != 4:
        raise ValueError(f"{name} must be a contiguous 4-D tensor")


def fa_fwd_fp8(q8, k8, vt8, causal: bool, scale: float, q_descale: float, k_descale: float,
               v_descale: float, k_start=None, k_end=None, o=None, lse=None, stream=None):
    """FP8 forward via fa_fwd_fp8: q8 [B,Hq,Sq,128], k8 [B,Hkv,Sk,128] and
    vt8 [B,Hkv,128,Sk] (V transposed) e4m3 CUDA tensors with per-tensor
    descale factors.  Returns (o bf16 [B,Hq,Sq,128], lse [B,Hq,Sq])."""
    lib = load_library()
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        _need8(t, n)
    B, Hq, Sq, d = q8.shape
    _, Hkv, Sk, _ = k8.shape
    if tuple(vt8.shape) != (B, Hkv, d, Sk):
        raise ValueError(f"vt8 must be [B, Hkv, d, Sk] = {(B, Hkv, d, Sk)}")
    o = torch.empty(B, Hq, Sq, d, dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q8.device) if lse is None else lse
    st = lib.fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, d,
                        int(bool(causal)), float(scale), float(q_descale), float(k_descale),
                        float(v_descale), _ptr(k_start), _ptr(k_end), _stream(stream))
    _check(st, "fa_fwd_fp8")
    return o, lse


def fa_bwd_workspace_size(B, Hq, Sq, d) -> int:
    return int(load_library().fa_bwd_workspace_size(B, Hq, Sq, d))


def fa_bwd(q, k, v, o, dout, lse, causal: bool, scale: float, k_start=None, k_end=None,
           dq=None, dk=None, dv=None, workspace=None, stream=None, key_mask=None,
           dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """dQ, dK, dV by recomputation via the library's fa_bwd (fa_bwd_masked
    when key_mask is given, fa_bwd_dropout when dropout_p > 0; mask and
    dropout arguments must be the forward's).  Returns (dq, dk, dv)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, Hq, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = fa_bwd_workspace_size(B, Hq, Sq, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    bits = _mask_bits(key_mask, B, Sk, stream)
    if dropout_p > 0.0:
        st = lib.fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d,
                                int(bool(causal)), float(scale), _ptr(k_start), _ptr(k_end),
                                _ptr(bits), float(dropout_p), int(seed), int(offset),
                                _ptr(workspace), workspace.numel(), _stream(stream))
        _check(st, "fa_bwd_dropout")
    elif bits is None:
        st = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d, int(bool(causal)),
                        float(scale), _ptr(k_start), _ptr(k_end), _ptr(workspace),
                        workspace.numel(), _stream(stream))
        _check(st, "fa_bwd")
    else:
        st = lib.fa_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Sk, d,
                               int(bool(causal)), float(scale), _ptr(k_start), _ptr(k_end),
                               _ptr(bits), _ptr(workspace), workspace.numel(), _stream(stream))
        _check(st, "fa_bwd_masked")
    return dq, dk, dv


def _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k):
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, n, torch.int32, 1)
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold nseq + 1 >= 2 offsets")
    Hq, total_q, d = q.shape
    Hkv, total_k, _ = k.shape
    return cu_seqlens_q.numel() - 1, Hq, Hkv, total_q, total_k, d


def fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  causal: bool, scale: float, key_mask=None, o=None, lse=None, stream=None):
    """Packed ragged forward via fa_fwd_varlen: q [Hq,total_q,d], k/v
    [Hkv,total_k,d] bf16; cu_seqlens_* int32 [nseq+1] CUDA offsets; key_mask
    optional [total_k] bools over the packed keys.  Returns (o, lse [Hq,total_q])."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 3)
    nseq, Hq, Hkv, total_q, total_k, d = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k,
                                                      max_seqlen_q, max_seqlen_k)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(Hq, total_q, dtype=torch.float32, device=q.device) if lse is None else lse
    bits = _mask_bits(None if key_mask is None else key_mask.reshape(1, -1), 1, total_k, stream)
    st = lib.fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                           _ptr(cu_seqlens_k), nseq, int(max_seqlen_q), int(max_seqlen_k),
                           total_q, total_k, Hq, Hkv, d, int(bool(causal)), float(scale),
                           _ptr(bits), _stream(stream))
    _check(st, "fa_fwd_varlen")
    return o, lse


def fa_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool, scale: float, key_mask=None, dq=None,
                  dk=None, dv=None, workspace=None, stream=None):
    """Packed ragged backward via fa_bwd_varlen (layout of fa_fwd_varlen).
    Returns (dq [Hq,total_q,d], dk, dv [Hkv,total_k,d])."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, n, torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    nseq, Hq, Hkv, total_q, total_k, d = _varlen_args(q, k, cu_seqlens_q, cu_seqlens_k,
                                                      max_seqlen_q, max_seqlen_k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(1, Hq, total_q, d), dtype=torch.uint8,
                                device=q.device)
    bits = _mask_bits(None if key_mask is None else key_mask.reshape(1, -1), 1, total_k, stream)
    st = lib.fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), nseq,
                           int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, Hq, Hkv, d,
                           int(bool(causal)), float(scale), _ptr(bits), _ptr(workspace),
                           workspace.numel(), _stream(stream))
    _check(st, "fa_bwd_varlen")
    return dq, dk, dv


def fa_decode_workspace_size(B, Hq, Sk_max, d) -> int:
    return int(load_library().fa_decode_workspace_size(B, Hq, Sk_max, d))


def fa_decode(q, k_cache, v_cache, seqlens_k, scale: float, o=None, lse=None, workspace=None,
              stream=None):
    """Single-query decode over a padded cache via the library's fa_decode.
    q [B,Hq,1,d], k_cache/v_cache [B,Hkv,Sk_max,d], seqlens_k int32 [B] (CUDA).
    Returns (o [B,Hq,1,d], lse [B,Hq])."""
    lib = load_library()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
    _need(seqlens_k, "seqlens_k", torch.int32, 1)
    B, Hq, _, d = q.shape
    _, Hkv, Sk_max, _ = k_cache.shape
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = fa_decode_workspace_size(B, Hq, Sk_max, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    st = lib.fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                       _ptr(seqlens_k), B, Hq, Hkv, Sk_max, d, float(scale), _ptr(workspace),
                       workspace.numel(), _stream(stream))
    _check(st, "fa_decode")
    return o, lse


DECODE_NOALLOC_MAX_SCRATCH_BYTES = 64 << 20


def fa_decode_noalloc(q, k_cache, v_cache, seqlens_k, scale: float, o=None, lse=None,
                      stream=None):
    """fa_decode without a caller workspace: the library uses its built-in
    64 MiB scratch array instead (see include/fa.h).  For callers that cannot
    allocate device scratch; outputs may still be passed in.  Calls that can
    overlap on the GPU share that scratch and race."""
    lib = load_library()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, 4)
    _need(seqlens_k, "seqlens_k", torch.int32, 1)
    B, Hq, _, d = q.shape
    _, Hkv, Sk_max, _ = k_cache.shape
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device) if lse is None else lse
    st = lib.fa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                               _ptr(seqlens_k), B, Hq, Hkv, Sk_max, d, float(scale),
                               _stream(stream))
    _check(st, "fa_decode_noalloc")
    return o, lse


def fa_device_status(clear: bool = True):
    """(status, raw word) of the device status words; synchronises the device."""
    lib = load_library()
    w = ctypes.c_uint(0)
    st = lib.fa_device_status(ctypes.byref(w), int(bool(clear)))
    return st, w.value


def fa_selftest_wait_timeout(stream=None):
    """Run the bounded-wait self-test (about 1 s): returns the two flags the
    kernel sets (1 = that wait reported failure).  fa_device_status() then
    reports the recorded timeout."""
    lib = load_library()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    _check(lib.fa_selftest_wait_timeout(_ptr(res), _stream(stream)), "fa_selftest_wait_timeout")
    return [int(x) for x in res[:2].cpu()]


def fa_profile_next_launch(start=None, stop=None):
    """Arm the one-shot hook: the next fa_* call on this thread records the two
    torch.cuda.Event objects around its main kernel (None, None disarms)."""
    lib = load_library()
    a = None if start is None else ctypes.c_void_p(start.cuda_event)
    b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check(lib.fa_profile_next_launch(a, b), "fa_profile_next_launch")


def version() -> str:
    return load_library().fa_version().decode()
