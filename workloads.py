"""Seeded synthetic inputs for decode attention over a paged KV cache.

This module is shared by the tests, the benchmark and the smoke check.  It holds
input generators only -- none of the method's arithmetic (no metadata, scores,
selection, attention or quantisation) -- so that the CUDA path and the CPU
oracle can be fed identical inputs without sharing any code that computes.

Every tensor is drawn from ``torch.Generator(device).manual_seed(seed)`` -- on
the CPU for the small parity cases, on the GPU (torch's Philox generator) for
the full-size workloads, where a CPU draw of 2^31 normals would take minutes --
and rounded to its storage dtype with round-to-nearest-even.  The workloads
stand in for the pages' LongBench / 32K-prompt serving runs (TinyServe) and
the 1M-token Llama-3-8B runs (HeadInfer) with synthetic data of the same
shapes; no dataset item is used.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int           # batch (sequences)
    Hq: int          # query heads
    Hkv: int         # key/value heads
    d: int           # head dim
    N: int           # context tokens
    S: int = 16      # page size (tokens)
    top_k: int = 0   # pages kept per q-head (0: exact attention only)
    dtype: str = "bf16"   # storage dtype of q, K, V ("bf16" | "fp16")
    kind: str = "normal"  # value recipe, see make_inputs
    q4: bool = False      # K/V stored in the 4-bit group-of-64 format

    @property
    def P(self) -> int:
        return (self.N + self.S - 1) // self.S

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, in order.  Sizes follow the decode shapes the pages run:
# TinyServe's 125M-1.3B models at up to 32K context with a 2048-token budget of
# 16-token pages, Llama-3-8B GQA (32 q / 8 kv heads, d=128) as in HeadInfer,
# and an OPT-30B-shaped cache in FlexGen's 4-bit group-of-64 format.
WORKLOADS = [
    Workload("tiny-mha-b1-h16-d64-n1k", B=1, Hq=16, Hkv=16, d=64, N=1024, top_k=16),
    Workload("mha-1.3b-b8-h32-d64-n8k", B=8, Hq=32, Hkv=32, d=64, N=8192, top_k=128,
             kind="offset"),
    Workload("llama3-8b-gqa-b16-n32k", B=16, Hq=32, Hkv=8, d=128, N=32768, top_k=128,
             kind="hot"),
    Workload("llama3-8b-gqa-b1-n1m-headwise", B=1, Hq=32, Hkv=8, d=128, N=1048576),
    Workload("opt-30b-q4-b64-h56-n2k", B=64, Hq=56, Hkv=56, d=128, N=2048, top_k=32,
             dtype="fp16", q4=True),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def _randn(gen: torch.Generator, shape, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """Standard normals in fp32, drawn in fixed-size chunks (bounded memory)."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float32, device=gen.device)
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32, device=gen.device)
    return out.view(*shape)


def make_inputs(w: Workload, seed: int, device="cpu"):
    """Return (q [B,Hq,d], K [B,Hkv,N,d], V [B,Hkv,N,d]) in w's dtype on `device`.

    kinds:
      normal  q, K, V ~ N(0, 1).
      offset  K, V = N(0, 1) + a per-(batch, head, channel) offset ~ N(0, 0.5^2),
              drawn separately for K and V; q ~ N(0, 1).
      coarse  q, V ~ N(0, 1); K = N(0, 1) rounded to integers (many pages share
              their channel min / max, so bound scores tie exactly).
      hot     q, V ~ N(0, 1); K ~ N(0, 1), and in every (batch, kv-head)
              round(0.02 * P) pages drawn without replacement get every key
              shifted by 2 * qhat, qhat = the unit-length mean of that group's
              query heads (pages that the group's queries should find).
    """
    gen = torch.Generator(device=device).manual_seed(int(seed))
    dt = w.torch_dtype
    q = _randn(gen, (w.B, w.Hq, w.d))
    K = _randn(gen, (w.B, w.Hkv, w.N, w.d)).to(dt) if w.kind == "normal" else \
        _randn(gen, (w.B, w.Hkv, w.N, w.d))
    V = _randn(gen, (w.B, w.Hkv, w.N, w.d)).to(dt) if w.kind == "normal" else \
        _randn(gen, (w.B, w.Hkv, w.N, w.d))
    if w.kind == "offset":
        K += 0.5 * _randn(gen, (w.B, w.Hkv, 1, w.d))
        V += 0.5 * _randn(gen, (w.B, w.Hkv, 1, w.d))
    elif w.kind == "hot":
        n_hot = int(round(0.02 * w.P))
        qg = q.view(w.B, w.Hkv, w.G, w.d).mean(dim=2)
        qhat = qg / qg.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        # page-level mask of the hot pages, then one broadcast add per token
        hot = torch.zeros(w.B, w.Hkv, w.P, dtype=torch.float32, device=K.device)
        for b in range(w.B):
            for h in range(w.Hkv):
                pages = torch.randperm(w.P, generator=gen, device=gen.device)[:n_hot]
                hot[b, h, pages] = 1.0
        tok_hot = hot.repeat_interleave(w.S, dim=2)[:, :, :w.N]
        K += 2.0 * tok_hot.unsqueeze(-1) * qhat.unsqueeze(2)
    elif w.kind == "coarse":
        K = torch.round(K)
    elif w.kind != "normal":
        raise ValueError(w.kind)
    return q.to(dt), K.to(dt), V.to(dt)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a 16-bit float CPU tensor as numpy uint16 (a view)."""
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(t.dtype)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """Inverse of bits(): a uint16 array as a bf16 / fp16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)
