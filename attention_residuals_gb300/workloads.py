"""Seeded synthetic inputs for the AttnRes read operator.

This module only draws random numbers and lays them out; it holds none of the
operator's arithmetic.  Both the CUDA path (through the tests and the
benchmark) and the FP64 oracle (through the tests) consume what it returns.

The five workloads follow the shapes the pages benchmark and describe:
  * "[Perf] Parallelize AttnRes long-sequence reduction", Test plan table:
    (L, T, D) = (8, 8192, 2048), (10, 32768, 4096), (64, 8192, 8192), bf16;
  * "Fast Attention Residuals", Quickstart: values [8, 2, 1024] and a
    [1024] query; sections "Full and Block schedules" (block sums plus an
    unaveraged partial block) and "Sliced LR-AttnRes" (R < D).

Every tensor comes from a ``torch.Generator`` seeded with ``seed``; on the
CPU the draws are bit-reproducible across machines.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

EPS_DEFAULT = 2.0 ** -23


@dataclass
class Workload:
    name: str
    S: int
    N: int
    D: int
    R: int
    key_offset: int
    eps: float
    scale: float
    out_norm: bool
    values: torch.Tensor            # packed [S, N, D] bf16
    q: torch.Tensor                 # [R] bf16
    w_o: Optional[torch.Tensor]     # [D] bf16 or None
    dy: torch.Tensor                # [N, D] bf16
    notes: dict = field(default_factory=dict)


CONFIGS = {
    1: dict(name="tiny S8 N2 D1024", S=8, N=2, D=1024, R=1024, out_norm=False,
            src_scale=None, q_std=None, blocks=False, zero_frac=0.0),
    2: dict(name="short S8 N8192 D2048", S=8, N=8192, D=2048, R=2048, out_norm=False,
            src_scale=(0.5, 2.0), q_std="rank", blocks=False, zero_frac=0.0),
    3: dict(name="long S10 N32768 D4096 out-norm", S=10, N=32768, D=4096, R=4096,
            out_norm=True, src_scale=(0.5, 2.0), q_std="rank", blocks=False, zero_frac=0.0),
    4: dict(name="sliced block S9 N16384 D4096 R1024", S=9, N=16384, D=4096, R=1024,
            out_norm=False, src_scale=None, q_std="rank", blocks=True, zero_frac=0.02),
    5: dict(name="deep S64 N8192 D8192 out-norm", S=64, N=8192, D=8192, R=8192,
            out_norm=True, src_scale=(0.25, 4.0), q_std="rank", blocks=False, zero_frac=0.0),
}


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def make_workload(cfg: int, *, N: Optional[int] = None, key_offset: Optional[int] = None,
                  seed: Optional[int] = None, device: str = "cpu") -> Workload:
    """Build workload ``cfg`` (1..5).  ``N`` overrides the token count (same
    distributions, fewer tokens); ``key_offset`` defaults to 0 (the first R
    channels).  Values are drawn source by source so the peak temporary is
    one fp32 [N, D] slab."""
    c = CONFIGS[cfg]
    S, D, R = c["S"], c["D"], c["R"]
    N = c["N"] if N is None else int(N)
    ko = 0 if key_offset is None else int(key_offset)
    seed = cfg if seed is None else int(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    values = torch.empty((S, N, D), dtype=torch.bfloat16, device=device)
    notes = {}
    if c["src_scale"] is not None:
        lo, hi = c["src_scale"]
        scales = lo + (hi - lo) * torch.rand((S,), generator=gen, device=device)
        notes["source_scales"] = scales.cpu().tolist()
    else:
        scales = None
    for s in range(S):
        if c["blocks"] and s < S - 1:
            # a completed block sum: three bf16 N(0,1) tensors added in fp32
            acc = torch.zeros((N, D), dtype=torch.float32, device=device)
            for _ in range(3):
                acc += _randn((N, D), gen, device).to(torch.bfloat16).float()
            values[s] = acc.to(torch.bfloat16)
        else:
            x = _randn((N, D), gen, device)
            if scales is not None:
                x *= scales[s]
            values[s] = x.to(torch.bfloat16)
    if c["zero_frac"] > 0.0 and N > 0:
        p = c["zero_frac"]
        # independent (source, token) rows zeroed with probability p ...
        mask = torch.rand((S, N), generator=gen, device=device) < p
        # ... plus a few tokens with every source zeroed (uniform routing, zero read)
        n_all = max(1, math.ceil(p * N / S))
        perm = torch.randperm(N, generator=gen, device=device)[:n_all]
        mask[:, perm] = True
        values[mask] = 0
        notes["zero_rows"] = int(mask.sum().item())
        notes["all_zero_tokens"] = sorted(perm.cpu().tolist())
    qn = _randn((R,), gen, device)
    if c["q_std"] == "rank":
        qn *= R ** -0.5
    q = qn.to(torch.bfloat16)
    w_o = None
    if c["out_norm"]:
        w_o = (1.0 + 0.1 * _randn((D,), gen, device)).to(torch.bfloat16)
    dy = _randn((N, D), gen, device).to(torch.bfloat16)
    return Workload(name=c["name"], S=S, N=N, D=D, R=R, key_offset=ko, eps=EPS_DEFAULT,
                    scale=1.0, out_norm=c["out_norm"], values=values, q=q, w_o=w_o, dy=dy,
                    notes=notes)


def make_random(S: int, N: int, D: int, R: Optional[int] = None, *, key_offset: int = 0,
                out_norm: bool = False, seed: int = 0, device: str = "cpu",
                value_std: float = 1.0, q_std: Optional[float] = None,
                scale: float = 1.0, eps: float = EPS_DEFAULT) -> Workload:
    """A free-form workload for edge cases: N(0, value_std) sources, N(0, q_std)
    query (default R^-1/2), w_o = 1 + 0.1 N(0,1) when out_norm."""
    R = D if R is None else int(R)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    values = (_randn((S, N, D), gen, device) * value_std).to(torch.bfloat16)
    qs = R ** -0.5 if q_std is None else q_std
    q = (_randn((R,), gen, device) * qs).to(torch.bfloat16)
    w_o = (1.0 + 0.1 * _randn((D,), gen, device)).to(torch.bfloat16) if out_norm else None
    dy = _randn((N, D), gen, device).to(torch.bfloat16)
    return Workload(name=f"random S{S} N{N} D{D} R{R}", S=S, N=N, D=D, R=R,
                    key_offset=int(key_offset), eps=eps, scale=scale, out_norm=out_norm,
                    values=values, q=q, w_o=w_o, dy=dy)


# ---------------------------------------------------------------------------
# Multi-query reads ("Fast Attention Residuals", section "Multi-query
# AttnRes": queries [M, R], 1 <= M <= 16, the page's example reads a packed
# [8, 2, 1024] value tensor with two rank-64 queries; its QK/V fixture routes
# two roles with two queries).
# ---------------------------------------------------------------------------
@dataclass
class MultiWorkload:
    name: str
    S: int
    N: int
    D: int
    R: int
    M: int
    key_offset: int
    eps: float
    scale: float
    values: torch.Tensor            # packed [S, N, D] bf16
    queries: torch.Tensor           # [M, R] bf16
    dy: torch.Tensor                # [M, N, D] bf16 (query-major)


MULTI_CONFIGS = {
    # the page's multi-query example: values [8, 2, 1024], queries [2, 64]
    "example": dict(S=8, N=2, D=1024, R=64, M=2, src_scale=None),
    # two queries over the long-sequence shapes at quarter rank, key in the
    # final R channels
    "long": dict(S=10, N=32768, D=4096, R=1024, M=2, src_scale=(0.5, 2.0)),
    # the most queries the page allows (M <= 16) over full-rank keys of
    # 1024-channel rows: the general backward and the tensor-core kernels
    "sixteen": dict(S=10, N=32768, D=1024, R=1024, M=16, src_scale=(0.5, 2.0)),
}


def make_multi(S: int, N: int, D: int, R: int, M: int, *, key_offset: Optional[int] = None,
               seed: int = 0, src_scale=None, device: str = "cpu", scale: float = 1.0,
               eps: float = EPS_DEFAULT, name: Optional[str] = None) -> MultiWorkload:
    """Sources N(0,1) (times one U[lo, hi] scalar per source when src_scale
    is given), queries N(0,1) * R^-1/2, dy N(0,1); key_offset defaults to
    the page's final R channels (D - R)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    values = torch.empty((S, N, D), dtype=torch.bfloat16, device=device)
    scales = None
    if src_scale is not None:
        lo, hi = src_scale
        scales = lo + (hi - lo) * torch.rand((S,), generator=gen, device=device)
    for s in range(S):
        x = _randn((N, D), gen, device)
        if scales is not None:
            x *= scales[s]
        values[s] = x.to(torch.bfloat16)
    queries = (_randn((M, R), gen, device) * R ** -0.5).to(torch.bfloat16)
    dy = _randn((M, N, D), gen, device).to(torch.bfloat16)
    ko = D - R if key_offset is None else int(key_offset)
    return MultiWorkload(name=name or f"multi S{S} N{N} D{D} R{R} M{M}", S=S, N=N, D=D, R=R, M=M,
                         key_offset=ko, eps=eps, scale=scale, values=values, queries=queries, dy=dy)


def make_multi_workload(key: str, *, N: Optional[int] = None, seed: Optional[int] = None,
                        device: str = "cpu") -> MultiWorkload:
    c = MULTI_CONFIGS[key]
    n = c["N"] if N is None else int(N)
    return make_multi(c["S"], n, c["D"], c["R"], c["M"], seed=100 + len(key) if seed is None else seed,
                      src_scale=c["src_scale"], device=device,
                      name=f"multi-query {key} S{c['S']} N{n} D{c['D']} R{c['R']} M{c['M']}")


# ---------------------------------------------------------------------------
# Selected-query reads ("Fast Attention Residuals", section "Multi-query
# AttnRes": an [E, R] query bank and integer [..., K] ids per token)
# ---------------------------------------------------------------------------
@dataclass
class SelectedWorkload:
    name: str
    S: int
    N: int
    D: int
    R: int
    E: int
    K: int
    key_offset: int
    eps: float
    scale: float
    values: torch.Tensor            # packed [S, N, D] bf16
    bank: torch.Tensor              # [E, R] bf16
    ids: torch.Tensor               # [N, K] int64 in [0, E)
    dy: torch.Tensor                # [N, K, D] bf16


def make_selected(S: int, N: int, D: int, R: int, E: int, K: int, *, key_offset: Optional[int] = None,
                  seed: int = 0, src_scale=None, device: str = "cpu", scale: float = 1.0,
                  eps: float = EPS_DEFAULT, unused_rows: int = 0) -> SelectedWorkload:
    """Sources N(0,1) (times one U[lo, hi] scalar per source when src_scale is
    given), bank rows N(0,1) * R^-1/2, ids uniform over the first
    E - unused_rows bank rows (the rest are never selected), dy N(0,1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    values = torch.empty((S, N, D), dtype=torch.bfloat16, device=device)
    scales = None
    if src_scale is not None:
        lo, hi = src_scale
        scales = lo + (hi - lo) * torch.rand((S,), generator=gen, device=device)
    for s in range(S):
        x = _randn((N, D), gen, device)
        if scales is not None:
            x *= scales[s]
        values[s] = x.to(torch.bfloat16)
    bank = (_randn((E, R), gen, device) * R ** -0.5).to(torch.bfloat16)
    ids = torch.randint(0, max(1, E - unused_rows), (N, K), generator=gen, device=device, dtype=torch.int64)
    dy = _randn((N, K, D), gen, device).to(torch.bfloat16)
    ko = D - R if key_offset is None else int(key_offset)
    return SelectedWorkload(name=f"selected S{S} N{N} D{D} R{R} E{E} K{K}", S=S, N=N, D=D, R=R, E=E, K=K,
                            key_offset=ko, eps=eps, scale=scale, values=values, bank=bank, ids=ids, dy=dy)
