"""Seeded synthetic inputs for Simple GLA workloads.

This module only draws random numbers and builds shapes; it holds none of the
method's arithmetic.  It is shared by the tests, the benchmark and the smoke
check, and it is the one thing the CUDA path and the fp64 reference have in
common.

Workloads (shapes from the Laplace 3B page "线性注意力模型如何实现固定推理状态",
section "i14 与 Laplace 3B 架构": H = 16 heads, dk = 96, dv = 192, chunk 128 in
section "挑战 1"; 1,280 concurrent decode sequences in section "Trainium2 上的推理优化"):

  tiny_f32   B=1, H=2, T=256, dk=dv=64, chunk 64, fp32, h0 = 0
  layer_bf16 B=8, T=2048, H=16, dk=96, dv=192, chunk 128, bf16, h0 = 0
  long_bf16  B=1, T=32768, same shapes, h0 ~ N(0, 0.02^2)
  decode     N=1280 sequences x H=16, one token each, state ~ N(0, 0.02^2)
  ragged     64 sequences, lengths uniform in [1, 8192], packed, h0 per sequence

Draws: q, k ~ N(0,1)/sqrt(dk), v ~ N(0,1); the state / h0 ~ N(0, 0.02^2).
Decays are fixed per head, never learned: 1 - lambda_h is geometric across the
heads, i.e. log(1 - lambda_h) is evenly spaced from log(1/32) to log(1/512)
(tiny_f32, two heads) or log(1/4096) (sixteen heads).  The kernels take the
natural log of lambda_h as ``log_decay`` (fp32), computed here in fp64 as
log1p(-(1 - lambda_h)) and rounded once.

Generator: a ``torch.Generator`` on the target device seeded with ``seed``
(default 0); draw order q, k, v, then h0 / state.  Ragged lengths come from a
separate CPU generator seeded with ``seed`` (``randint(1, 8193)``) so the
lengths are the same on every device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" or "decode"
    dtype: str                # "f32" or "bf16": dtype of q, k, v and out
    H: int
    dk: int
    dv: int
    B: int = 1                # prefill: batch; decode: N sequences
    T: int = 1                # prefill: tokens per sequence (dense)
    chunk: int = 128
    h0_std: float = 0.0       # 0 => h0 = None (zeros)
    decay_lo: float = 1.0 / 32.0   # 1 - lambda for the first head
    decay_hi: float = 1.0 / 4096.0  # 1 - lambda for the last head
    ragged_n: int = 0         # > 0 => packed batch of this many sequences
    ragged_max: int = 0       # lengths uniform in [1, ragged_max]
    note: str = ""

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "prefill", "f32", H=2, dk=64, dv=64, B=1, T=256, chunk=64,
                         decay_lo=1 / 32, decay_hi=1 / 512,
                         note="tiny fp32 forward, B1 H2 T256 dk=dv=64 chunk64"),
    "layer_bf16": Workload("layer_bf16", "prefill", "bf16", H=16, dk=96, dv=192, B=8, T=2048, chunk=128,
                           note="Laplace-3B-shaped layer, B8 T2048 H16 dk96 dv192 chunk128 bf16"),
    "long_bf16": Workload("long_bf16", "prefill", "bf16", H=16, dk=96, dv=192, B=1, T=32768, chunk=128,
                          h0_std=0.02, note="long-context prefill, B1 T32768 H16 dk96 dv192, h0 != 0"),
    "decode": Workload("decode", "decode", "bf16", H=16, dk=96, dv=192, B=1280, h0_std=0.02,
                       note="recurrent decode step, N1280 x H16, fp32 state 96x192"),
    "ragged": Workload("ragged", "prefill", "bf16", H=16, dk=96, dv=192, chunk=128, h0_std=0.02,
                       ragged_n=64, ragged_max=8192,
                       note="ragged packed batch, 64 sequences with lengths U[1,8192]"),
}


def log_decays(H: int, lo: float = 1 / 32, hi: float = 1 / 4096) -> torch.Tensor:
    """Per-head natural-log decays: 1 - lambda_h geometric from ``lo`` to ``hi`` (fp32)."""
    if H == 1:
        one_minus = [lo]
    else:
        a, b = math.log(lo), math.log(hi)
        one_minus = [math.exp(a + (b - a) * h / (H - 1)) for h in range(H)]
    return torch.tensor([math.log1p(-x) for x in one_minus], dtype=torch.float64).float()


def ragged_lengths(n: int, max_len: int, seed: int = 0) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(1, max_len + 1, (n,), generator=g, dtype=torch.int64)


def cu_from_lengths(lengths) -> torch.Tensor:
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def _gen(device, seed):
    return torch.Generator(device=device).manual_seed(seed)


def _randn(shape, g, device, scale=1.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def make_prefill(w: Workload, device="cpu", seed: int = 0, lengths=None, T: Optional[int] = None,
                 B: Optional[int] = None):
    """Inputs for a prefill workload.

    Returns a dict with q, k, v (``w.dtype``), log_decay [H] fp32, h0 (fp32 or None),
    cu_seqlens (int32 CPU tensor or None), and the chunk length.  ``T``/``B`` override
    the dense sizes; ``lengths`` overrides the ragged lengths."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    if w.ragged_n > 0 or lengths is not None:
        if lengths is None:
            lengths = ragged_lengths(w.ragged_n, w.ragged_max, seed)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        cu = cu_from_lengths(lengths)
        total = int(cu[-1])
        lead, nseq = (1, total), int(lengths.numel())
    else:
        Bv = w.B if B is None else B
        Tv = w.T if T is None else T
        cu = None
        lead, nseq = (Bv, Tv), Bv
    q = _randn(lead + (w.H, w.dk), g, dev, 1.0 / math.sqrt(w.dk)).to(w.torch_dtype)
    k = _randn(lead + (w.H, w.dk), g, dev, 1.0 / math.sqrt(w.dk)).to(w.torch_dtype)
    v = _randn(lead + (w.H, w.dv), g, dev).to(w.torch_dtype)
    h0 = None
    if w.h0_std > 0:
        h0 = _randn((nseq, w.H, w.dk, w.dv), g, dev, w.h0_std)
    ld = log_decays(w.H, w.decay_lo, w.decay_hi).to(dev)
    return {"q": q, "k": k, "v": v, "log_decay": ld, "h0": h0, "cu_seqlens": cu, "chunk": w.chunk}


def make_backward(w: Workload, device="cpu", seed: int = 0, lengths=None, T: Optional[int] = None,
                  B: Optional[int] = None, dhT_std: float = 0.02):
    """Inputs for the backward of a prefill workload: make_prefill's tensors for ``seed``, plus
    dout ~ N(0, 1) with the shape of the output (``w.dtype``) and dhT ~ N(0, dhT_std^2) fp32
    (None when dhT_std is 0), drawn in that order from a generator seeded with seed + 1000003."""
    d = make_prefill(w, device=device, seed=seed, lengths=lengths, T=T, B=B)
    dev = torch.device(device)
    g = _gen(dev, seed + 1000003)
    nseq = d["q"].shape[0] if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    d["dout"] = _randn(tuple(d["q"].shape[:3]) + (w.dv,), g, dev).to(w.torch_dtype)
    d["dhT"] = _randn((nseq, w.H, w.dk, w.dv), g, dev, dhT_std) if dhT_std > 0 else None
    return d


def make_gate(shape, device="cpu", seed: int = 0, scale: float = 2.0, dtype=torch.bfloat16):
    """Output-gate pre-activations g shaped like the output (``shape``): N(0, scale^2), seeded.  A
    spread of 2 puts the gate factors well into both of its tails."""
    dev = torch.device(device)
    g = _gen(dev, seed + 7919)
    return _randn(tuple(shape), g, dev, scale).to(dtype)


def make_decode(w: Workload, device="cpu", seed: int = 0, N: Optional[int] = None):
    """Inputs for one decode step: q, k [N,H,dk], v [N,H,dv] (``w.dtype``), state fp32."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    n = w.B if N is None else N
    q = _randn((n, w.H, w.dk), g, dev, 1.0 / math.sqrt(w.dk)).to(w.torch_dtype)
    k = _randn((n, w.H, w.dk), g, dev, 1.0 / math.sqrt(w.dk)).to(w.torch_dtype)
    v = _randn((n, w.H, w.dv), g, dev).to(w.torch_dtype)
    state = _randn((n, w.H, w.dk, w.dv), g, dev, w.h0_std if w.h0_std > 0 else 0.02)
    ld = log_decays(w.H, w.decay_lo, w.decay_hi).to(dev)
    return {"q": q, "k": k, "v": v, "log_decay": ld, "state": state}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of ``w`` with some sizes replaced (smaller parity cases)."""
    return replace(w, **kw)
