"""Seeded synthetic workloads shaped like the cuDNN Linear Attention page's GDN example.

This module only draws random inputs and fixes shapes: it contains none of the
method's arithmetic, so both the CUDA path and the CPU oracle can consume the
same tensors.  Every tensor is produced on the CPU from a seeded
``torch.Generator`` (seed = 1000 + config number unless given), so a run is
reproducible bit for bit.

Distributions (the page's worked example, section "Example"):
  q, k, v ~ N(0, 1) rounded to bf16; g = -softplus(N(0, 1)) fp32 (natural-log
  decay); beta = sigmoid(N(0, 1)) fp32; initial_state ~ 0.1 * N(0, 1) fp32 where
  a config asks for one.

The ``slow_decay`` variant (g' = 1e-4 g, beta' = 0.1 beta) keeps the state alive
across many chunks, so that the inter-chunk path, the initial state and the
transitions are actually exercised; with the page's distributions one 64-token
chunk already decays by about exp(-51).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

CHUNK = 64


@dataclasses.dataclass
class Workload:
    name: str
    cu_seqlens: torch.Tensor          # [N+1] int32 (CPU)
    q: torch.Tensor                   # [T, HK, K] bf16
    k: torch.Tensor                   # [T, HK, K] bf16
    v: torch.Tensor                   # [T, HV, V] bf16
    g: torch.Tensor                   # [T, HO] fp32
    beta: torch.Tensor                # [T, HO] fp32
    initial_state: Optional[torch.Tensor] = None   # [N, HO, K, V] fp32
    output_final_state: bool = True
    checkpoint_every_n: int = 0
    checkpoint_dtype: torch.dtype = torch.bfloat16
    use_qk_l2norm: bool = True
    spans: Optional[torch.Tensor] = None          # summary configs: span cu_seqlens

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def HK(self) -> int:
        return int(self.q.shape[1])

    @property
    def HV(self) -> int:
        return int(self.v.shape[1])

    @property
    def K(self) -> int:
        return int(self.q.shape[2])

    @property
    def V(self) -> int:
        return int(self.v.shape[2])

    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.numpy().astype(np.int64))


def _cu(lengths) -> torch.Tensor:
    cu = np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))])
    return torch.tensor(cu, dtype=torch.int32)


def draw(name, lengths, HK, HV, K, V, *, seed, initial_state=False, slow_decay=False,
         **kw) -> Workload:
    """Draw one workload with the page's distributions for the given shapes."""
    gen = torch.Generator().manual_seed(int(seed))
    cu = _cu(lengths)
    T = int(cu[-1])
    HO = HV
    q = torch.randn(T, HK, K, generator=gen).to(torch.bfloat16)
    k = torch.randn(T, HK, K, generator=gen).to(torch.bfloat16)
    v = torch.randn(T, HV, V, generator=gen).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn(T, HO, generator=gen))
    beta = torch.sigmoid(torch.randn(T, HO, generator=gen))
    if slow_decay:
        g = g * 1e-4
        beta = beta * 0.1
    s0 = None
    N = len(lengths)
    if initial_state:
        s0 = 0.1 * torch.randn(N, HO, K, V, generator=gen)
    return Workload(name=name, cu_seqlens=cu, q=q, k=k, v=v, g=g.float().contiguous(),
                    beta=beta.float().contiguous(), initial_state=s0, **kw)


def skewed_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """Lengths drawn log-uniformly in [lo, hi] and rounded (deterministic per seed)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(lo), math.log(hi), size=n)
    return [int(round(math.exp(x))) for x in u]


def config(num: int, *, slow_decay: bool = False, seed: Optional[int] = None) -> Workload:
    """The five GDN workloads (1: tiny, 2: varlen, 3: dense batch, 4: skewed GVA, 5: summary)."""
    s = 1000 + num if seed is None else seed
    if num == 1:
        return draw("tiny T=256 N=2 H=2 K=V=64", [100, 156], 2, 2, 64, 64, seed=s,
                    slow_decay=slow_decay)
    if num == 2:
        return draw("varlen T=4096 N=3 H=16 K=V=128", [1000, 1500, 1596], 16, 16, 128, 128,
                    seed=s, slow_decay=slow_decay)
    if num == 3:
        return draw("dense batch T=65536 N=8x8192 H=32 K=V=128", [8192] * 8, 32, 32, 128, 128,
                    seed=s, initial_state=True, slow_decay=slow_decay,
                    checkpoint_every_n=1024, checkpoint_dtype=torch.float32)
    if num == 4:
        return draw("skewed varlen GVA N=64 HK=16 HV=32 K=V=128",
                    skewed_lengths(64, 16, 16384, s), 16, 32, 128, 128, seed=s,
                    slow_decay=slow_decay)
    if num == 5:
        w = draw("summary T=131072 N=1 H=16 K=V=128, 8 spans of 16384", [131072], 16, 16,
                 128, 128, seed=s, slow_decay=slow_decay)
        w.spans = _cu([16384] * 8)
        return w
    raise ValueError(f"no workload {num}")


def scaled(w: Workload, name: str, lengths, seed: int) -> Workload:
    """A smaller workload with the same head layout and options as ``w``."""
    return draw(name, lengths, w.HK, w.HV, w.K, w.V, seed=seed,
                initial_state=w.initial_state is not None,
                output_final_state=w.output_final_state,
                checkpoint_every_n=w.checkpoint_every_n,
                checkpoint_dtype=w.checkpoint_dtype)
