"""Seeded synthetic inputs shaped like the pages' attention workloads.

This module holds no attention arithmetic: it only draws random tensors, so
the tests can hand the very same inputs to the CUDA path and to the oracle.

Recipe (used for every workload): a CPU ``torch.Generator`` seeded with 0
draws, in this order, Q, K, V and then dO (when the workload has a backward),
each as i.i.d. N(0, 1) in fp32, in the [B, H, S, d] layout, and each is then
rounded to bf16 (round to nearest even).  Workload-specific extras:

* ``prefill_8k_masked``: Q is multiplied by 8 before rounding, so raw
  logits reach about +-100 and a naive exp would overflow; batch row 0 gets
  the key interval [64, Sk), i.e. keys 0..63 are padding, which under the
  causal rule leaves query rows 0..63 of that batch row with no visible key.
* ``decode_ragged``: per-sequence key lengths are drawn first, uniform integers in
  [1024, 32768], from the same seeded generator; the KV cache is padded to
  32768 positions and the padding is left at zero.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    kind: str  # "fwd", "fwd+bwd" or "decode"
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    scale: float
    q_mult: float = 1.0
    masked_prefix: int = 0  # keys [0, masked_prefix) are padding in batch row 0
    tensors: dict = field(default_factory=dict)

    def flops_fwd(self) -> float:
        """4*B*Hq*Sq*Sk*d, halved under the causal rule."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


def _randn(gen, shape, mult=1.0):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(torch.bfloat16)


SPECS = {
    "small_noncausal": dict(kind="fwd", B=1, Hq=2, Hkv=2, Sq=256, Sk=256, d=64, causal=False),
    "prefill_2k": dict(kind="fwd+bwd", B=4, Hq=16, Hkv=16, Sq=2048, Sk=2048, d=128,
                       causal=True),
    "gqa_4k": dict(kind="fwd", B=8, Hq=32, Hkv=8, Sq=4096, Sk=4096, d=128, causal=True),
    "prefill_8k_masked": dict(kind="fwd+bwd", B=2, Hq=16, Hkv=16, Sq=8192, Sk=8192, d=128,
                              causal=True, q_mult=8.0, masked_prefix=64),
    "decode_ragged": dict(kind="decode", B=32, Hq=32, Hkv=8, Sq=1, Sk=32768, d=128,
                          causal=False),
}

# Human-readable descriptions used in reports.
DESCRIPTIONS = {
    "small_noncausal": "fwd, non-causal, B=1 H=2 S=256 d=64",
    "prefill_2k": "fwd+bwd, causal, B=4 H=16 S=2048 d=128",
    "gqa_4k": "GQA fwd, causal, B=8 Hq=32 Hkv=8 S=4096 d=128",
    "prefill_8k_masked": "fwd+bwd, causal, B=2 H=16 S=8192 d=128, Q*8, "
                         "batch row 0 keys 0..63 padded",
    "decode_ragged": "decode Sq=1, B=32 Hq=32 Hkv=8 d=128, Sk in [1024, 32768], cache 32768",
}


def make(name: str, seed: int = 0, with_dout=None, **overrides) -> Workload:
    """Build workload ``name`` with seeded CPU tensors.  ``overrides`` may shrink
    any size (B, Hq, Hkv, Sq, Sk) for small parity cases; the recipe is kept."""
    spec = dict(SPECS[name])
    spec.update(overrides)
    kind = spec.pop("kind")
    q_mult = spec.pop("q_mult", 1.0)
    masked_prefix = spec.pop("masked_prefix", 0)
    w = Workload(name=name, kind=kind, scale=1.0 / math.sqrt(spec["d"]), q_mult=q_mult,
                 masked_prefix=masked_prefix, **spec)
    gen = torch.Generator().manual_seed(seed)
    if kind == "decode":
        seqlens = torch.randint(1024, 32769, (w.B,), generator=gen, dtype=torch.int64)
        seqlens = seqlens.clamp(max=w.Sk).to(torch.int32)
        w.tensors["q"] = _randn(gen, (w.B, w.Hq, 1, w.d))
        kc = torch.zeros(w.B, w.Hkv, w.Sk, w.d, dtype=torch.bfloat16)
        vc = torch.zeros(w.B, w.Hkv, w.Sk, w.d, dtype=torch.bfloat16)
        for b in range(w.B):
            n = int(seqlens[b])
            kc[b, :, :n] = _randn(gen, (w.Hkv, n, w.d))
        for b in range(w.B):
            n = int(seqlens[b])
            vc[b, :, :n] = _randn(gen, (w.Hkv, n, w.d))
        w.tensors.update(k=kc, v=vc, seqlens_k=seqlens)
        return w
    w.tensors["q"] = _randn(gen, (w.B, w.Hq, w.Sq, w.d), q_mult)
    w.tensors["k"] = _randn(gen, (w.B, w.Hkv, w.Sk, w.d))
    w.tensors["v"] = _randn(gen, (w.B, w.Hkv, w.Sk, w.d))
    if with_dout if with_dout is not None else kind == "fwd+bwd":
        w.tensors["dout"] = _randn(gen, (w.B, w.Hq, w.Sq, w.d))
    if masked_prefix:
        ks = torch.zeros(w.B, dtype=torch.int32)
        ks[0] = masked_prefix
        w.tensors["k_start"] = ks
        w.tensors["k_end"] = torch.full((w.B,), w.Sk, dtype=torch.int32)
    return w


def worked_example_bf16():
    """The pages' single-query example (scores 1000, 1001, 999; values 1, 3, 7)
    encoded exactly in bf16 with d=64 and scale 1: 1001 and 999 are not bf16
    values, so each score is split over two exact products, 992 + 8, 992 + 9,
    992 + 7, with q = [1, 1, 0, ...]."""
    d = 64
    q = torch.zeros(1, 1, 1, d)
    q[0, 0, 0, 0] = 1.0
    q[0, 0, 0, 1] = 1.0
    k = torch.zeros(1, 1, 3, d)
    k[0, 0, :, 0] = 992.0
    k[0, 0, :, 1] = torch.tensor([8.0, 9.0, 7.0])
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, :, 0] = torch.tensor([1.0, 3.0, 7.0])
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def random_qkv(B, Hq, Hkv, Sq, Sk, d, seed=0, q_mult=1.0, with_dout=False):
    """Seeded bf16 Q, K, V (and dO) of arbitrary shape, same recipe as ``make``."""
    gen = torch.Generator().manual_seed(seed)
    out = {
        "q": _randn(gen, (B, Hq, Sq, d), q_mult),
        "k": _randn(gen, (B, Hkv, Sk, d)),
        "v": _randn(gen, (B, Hkv, Sk, d)),
    }
    if with_dout:
        out["dout"] = _randn(gen, (B, Hq, Sq, d))
    return out
