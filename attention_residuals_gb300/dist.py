"""Multi-process helpers (plumbing around torch.distributed).

The read operator is independent per token; only dq and dw_o are sums over
tokens.  Under data parallelism each rank runs the operator on its own
tokens and the gradients of q and w_o are summed across ranks (the same
all-reduce a training framework applies to every parameter gradient), so
the operator itself needs no collective.  These helpers hold that logic and
the benchmark's timing rule (the slowest rank sets the step time).
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import torch


def shard_tokens(n_tokens: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, stop) token range of `rank` out of `world`; sizes
    differ by at most one."""
    if world < 1 or not (0 <= rank < world) or n_tokens < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(n_tokens, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def allreduce_param_grads_(grads: Iterable[Optional[torch.Tensor]], group=None) -> None:
    """Sum dq / dw_o (any tensors) across ranks in place; None entries are
    skipped.  bf16 gradients are summed in FP32 and rounded once."""
    import torch.distributed as dist
    for g in grads:
        if g is None:
            continue
        if g.dtype == torch.bfloat16:
            acc = g.float()
            dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
            g.copy_(acc.to(torch.bfloat16))
        else:
            dist.all_reduce(g, op=dist.ReduceOp.SUM, group=group)


def max_over_ranks(values, device=None, group=None):
    """Element-wise maximum of a list of floats over all ranks (one
    collective, outside any timed region)."""
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return [float(x) for x in t.tolist()]


def weak_scaling_throughput(bytes_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job GB/s when every rank moves `bytes_per_rank` per step and the
    slowest rank's step takes `max_ms`."""
    if max_ms <= 0:
        raise ValueError("step time must be positive")
    return world * bytes_per_rank / (max_ms * 1e-3) / 1e9
