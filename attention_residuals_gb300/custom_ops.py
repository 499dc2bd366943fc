"""torch.library registration of the read operator.

`attnres_gb300::read_fwd` and `attnres_gb300::read_bwd` wrap the C ABI
calls as custom operators with shape-only ("fake") implementations and an
autograd formula, so `torch.compile(..., fullgraph=True)` traces through
`attnres()` without graph breaks and CUDA-graph capture replays the same
kernels ("Fast Attention Residuals", Quickstart: the read is compiled with
fullgraph=True and replayed in CUDA graphs).  The operators compute nothing
themselves: every step runs in the CUDA library.

Values travel as a list plus a `packed` flag: either one packed
[S, ..., D] tensor (packed=True) or S separate [..., D] tensors; the
gradient comes back in the same form (a packed input gets one packed
gradient, with no stacking copy).  The flag is explicit because a list of
one [T, D] source and one packed [S, D] tensor (one token) have the same
shape.  The backward operators also return the FP32 sums of the reduced
gradients (dq, dw_o, the bank gradient) next to their bf16 roundings;
autograd uses the bf16 copies.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Tuple

import torch
from torch import Tensor

from . import _lib
from . import ops as _ops

_NS = "attnres_gb300"


def _shape_info(values: List[Tensor], packed: bool) -> Tuple[int, int, int, tuple]:
    if packed:
        if len(values) != 1 or values[0].dim() < 2:
            raise ValueError("packed values are one [S, ..., D] tensor")
        v = values[0]
        return v.shape[0], v.shape[-1], 1, tuple(v.shape[1:-1])
    return len(values), values[0].shape[-1], 0, tuple(values[0].shape[:-1])


def _pack_args(values):
    """(list of tensors, packed flag) for a user's values argument."""
    if isinstance(values, Tensor):
        return [values], True
    return list(values), False


def _bwd_resident(S: int, D: int, R: int, key_offset: int, out_norm: bool) -> bool:
    """Whether the backward keeps a token's rows resident (shape-only plan
    query: an empty token range needs no pointers)."""
    p = _lib.AttnresParams()
    p.S, p.D, p.R, p.key_offset, p.N = S, D, R, key_offset, 0
    p.eps, p.scale, p.out_norm, p.split_n_threshold, p.src_ld = 2.0 ** -23, 1.0, int(out_norm), 0, D
    out = (ctypes.c_int64 * 10)()
    rc = _lib.load().attnres_plan_info(ctypes.byref(p), out)
    return rc == 0 and bool(out[5])


def _as_values(values: List[Tensor], packed: int):
    return values[0] if packed else list(values)


@torch.library.custom_op(f"{_NS}::read_fwd", mutates_args=(), device_types="cuda")
def read_fwd(values: List[Tensor], q: Tensor, w_o: Optional[Tensor], eps: float, scale: float,
             key_offset: int, packed: bool) -> Tuple[Tensor, Tensor, Tensor, Tensor, Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    save = w_o is not None and not _bwd_resident(S, D, q.numel(), key_offset, True)
    r = _ops.attnres_fwd(_as_values(values, packed), q, w_o=w_o, eps=eps, scale=scale,
                         key_offset=key_offset, save_o_pre=save)
    dev = q.device
    empty = torch.empty((0,), dtype=torch.float32, device=dev)
    o_rstd = r["o_rstd"] if r["o_rstd"] is not None else empty
    o_pre = r["o_pre"] if r["o_pre"] is not None else empty.clone()
    return r["y"], r["alpha"], r["rstd"], r["logit"], o_rstd, o_pre


@read_fwd.register_fake
def _(values, q, w_o, eps, scale, key_offset, packed):
    S, D, packed, lead = _shape_info(values, packed)
    N = 1
    for d in lead:
        N *= d
    f32 = dict(dtype=torch.float32, device=q.device)
    y = torch.empty((*lead, D), dtype=torch.bfloat16, device=q.device)
    stats = [torch.empty((N, S), **f32) for _ in range(3)]
    if w_o is not None:
        o_rstd = torch.empty((N,), **f32)
        save = not _bwd_resident(S, D, q.numel(), key_offset, True)
        o_pre = torch.empty((N, D) if save else (0,), **f32)
    else:
        o_rstd = torch.empty((0,), **f32)
        o_pre = torch.empty((0,), **f32)
    return y, stats[0], stats[1], stats[2], o_rstd, o_pre


@torch.library.custom_op(f"{_NS}::read_bwd", mutates_args=(), device_types="cuda")
def read_bwd(values: List[Tensor], q: Tensor, w_o: Optional[Tensor], dy: Tensor, alpha: Tensor,
             rstd: Tensor, logit: Tensor, o_rstd: Tensor, o_pre: Tensor, eps: float, scale: float,
             key_offset: int, packed: bool) -> Tuple[List[Tensor], Tensor, Tensor, Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    saved = {"alpha": alpha, "rstd": rstd, "logit": logit,
             "o_rstd": o_rstd if o_rstd.numel() else None,
             "o_pre": o_pre if o_pre.numel() else None}
    g = _ops.attnres_bwd(_as_values(values, packed), q, dy.contiguous(), saved, w_o=w_o, eps=eps,
                         scale=scale, key_offset=key_offset)
    dv = [g["dvalues"]] if packed else list(g["dvalues"])
    dw = g["dw_o"] if g["dw_o"] is not None else torch.empty((0,), dtype=torch.bfloat16, device=q.device)
    dw32 = g["dw_o_f32"] if g["dw_o_f32"] is not None else torch.empty((0,), dtype=torch.float32,
                                                                        device=q.device)
    return dv, g["dq"].view_as(q), dw, g["dq_f32"].view(q.shape), dw32


@read_bwd.register_fake
def _(values, q, w_o, dy, alpha, rstd, logit, o_rstd, o_pre, eps, scale, key_offset, packed):
    dv = [torch.empty_like(v) for v in values]
    dw = torch.empty_like(w_o) if w_o is not None else torch.empty((0,), dtype=torch.bfloat16,
                                                                   device=q.device)
    f32 = dict(dtype=torch.float32, device=q.device)
    dw32 = torch.empty(w_o.shape if w_o is not None else (0,), **f32)
    return dv, torch.empty_like(q), dw, torch.empty(q.shape, **f32), dw32


def _setup_context(ctx, inputs, output):
    values, q, w_o, eps, scale, key_offset, packed = inputs
    y, alpha, rstd, logit, o_rstd, o_pre = output
    ctx.cfg = (eps, scale, key_offset, packed)
    ctx.has_w = w_o is not None
    ctx.nvalues = len(values)
    ctx.save_for_backward(q, w_o if w_o is not None else q.new_empty((0,)), alpha, rstd, logit,
                          o_rstd, o_pre, *values)


def _backward(ctx, dy, d_alpha, d_rstd, d_logit, d_orstd, d_opre):
    q, w_o, alpha, rstd, logit, o_rstd, o_pre, *values = ctx.saved_tensors
    eps, scale, key_offset, packed = ctx.cfg
    dv, dq, dw, _, _ = read_bwd(list(values), q, w_o if ctx.has_w else None, dy.to(torch.bfloat16),
                                alpha, rstd, logit, o_rstd, o_pre, eps, scale, key_offset, packed)
    return list(dv), dq, (dw if ctx.has_w else None), None, None, None, None


read_fwd.register_autograd(_backward, setup_context=_setup_context)


def attnres_op(values, query: Tensor, *, eps: float = _ops.EPS_DEFAULT, scale: float = 1.0,
               out_norm_weight: Optional[Tensor] = None, key_offset: Optional[int] = None) -> Tensor:
    """The read through the registered operator (compile- and graph-safe)."""
    vals, packed = _pack_args(values)
    D = vals[0].shape[-1]
    ko = D - query.numel() if key_offset is None else int(key_offset)
    y = read_fwd(vals, query, out_norm_weight, float(eps), float(scale), ko, packed)[0]
    return y


# --------------------------------------------------------------------------
# Multi-query read ("Fast Attention Residuals", section "Multi-query AttnRes")
# --------------------------------------------------------------------------
def _multi_out_shape(lead, M: int, D: int, token_major: bool):
    return (*lead, M, D) if token_major else (M, *lead, D)


@torch.library.custom_op(f"{_NS}::read_multi_fwd", mutates_args=(), device_types="cuda")
def read_multi_fwd(values: List[Tensor], queries: Tensor, eps: float, scale: float, key_offset: int,
                   token_major: bool, packed: bool) -> Tuple[Tensor, Tensor, Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    r = _ops.attnres_multi_fwd(_as_values(values, packed), queries, eps=eps, scale=scale,
                               key_offset=key_offset, token_major=token_major)
    return r["y"], r["alpha"], r["rstd"], r["logit"]


@read_multi_fwd.register_fake
def _(values, queries, eps, scale, key_offset, token_major, packed):
    S, D, packed, lead = _shape_info(values, packed)
    M = queries.shape[0]
    N = 1
    for d in lead:
        N *= d
    f32 = dict(dtype=torch.float32, device=queries.device)
    y = torch.empty(_multi_out_shape(lead, M, D, token_major), dtype=torch.bfloat16,
                    device=queries.device)
    return y, torch.empty((N, M, S), **f32), torch.empty((N, S), **f32), torch.empty((N, M, S), **f32)


@torch.library.custom_op(f"{_NS}::read_multi_bwd", mutates_args=(), device_types="cuda")
def read_multi_bwd(values: List[Tensor], queries: Tensor, dy: Tensor, alpha: Tensor, rstd: Tensor,
                   logit: Tensor, eps: float, scale: float, key_offset: int,
                   token_major: bool, packed: bool) -> Tuple[List[Tensor], Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    saved = {"alpha": alpha, "rstd": rstd, "logit": logit, "token_major": token_major}
    g = _ops.attnres_multi_bwd(_as_values(values, packed), queries, dy.contiguous(), saved, eps=eps,
                               scale=scale, key_offset=key_offset, token_major=token_major)
    dv = [g["dvalues"]] if packed else list(g["dvalues"])
    return dv, g["dq"], g["dq_f32"]


@read_multi_bwd.register_fake
def _(values, queries, dy, alpha, rstd, logit, eps, scale, key_offset, token_major, packed):
    return ([torch.empty_like(v) for v in values], torch.empty_like(queries),
            torch.empty(queries.shape, dtype=torch.float32, device=queries.device))


def _multi_setup_context(ctx, inputs, output):
    values, queries, eps, scale, key_offset, token_major, packed = inputs
    y, alpha, rstd, logit = output
    ctx.cfg = (eps, scale, key_offset, token_major, packed)
    ctx.save_for_backward(queries, alpha, rstd, logit, *values)


def _multi_backward(ctx, dy, d_alpha, d_rstd, d_logit):
    queries, alpha, rstd, logit, *values = ctx.saved_tensors
    eps, scale, key_offset, token_major, packed = ctx.cfg
    dv, dq, _ = read_multi_bwd(list(values), queries, dy.to(torch.bfloat16), alpha, rstd, logit, eps,
                               scale, key_offset, token_major, packed)
    return list(dv), dq, None, None, None, None, None


read_multi_fwd.register_autograd(_multi_backward, setup_context=_multi_setup_context)


def attnres_multi_op(values, queries: Tensor, *, eps: float = _ops.EPS_DEFAULT, scale: float = 1.0,
                     key_offset: Optional[int] = None, output_layout: str = "query_major") -> Tensor:
    """The multi-query read through the registered operator."""
    if output_layout not in ("query_major", "token_major"):
        raise ValueError("output_layout must be 'query_major' or 'token_major'")
    vals, packed = _pack_args(values)
    D = vals[0].shape[-1]
    ko = D - queries.shape[-1] if key_offset is None else int(key_offset)
    return read_multi_fwd(vals, queries, float(eps), float(scale), ko,
                          output_layout == "token_major", packed)[0]


# --------------------------------------------------------------------------
# Selected-query read ("Fast Attention Residuals", section "Multi-query
# AttnRes": attnres_selected)
# --------------------------------------------------------------------------
@torch.library.custom_op(f"{_NS}::read_selected_fwd", mutates_args=(), device_types="cuda")
def read_selected_fwd(values: List[Tensor], bank: Tensor, ids: Tensor, eps: float, scale: float,
                      key_offset: int, packed: bool) -> Tuple[Tensor, Tensor, Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    r = _ops.attnres_selected_fwd(_as_values(values, packed), bank, ids, eps=eps, scale=scale,
                                  key_offset=key_offset)
    return r["y"], r["alpha"], r["rstd"], r["logit"]


@read_selected_fwd.register_fake
def _(values, bank, ids, eps, scale, key_offset, packed):
    S, D, packed, lead = _shape_info(values, packed)
    K = ids.shape[-1]
    N = 1
    for d in lead:
        N *= d
    f32 = dict(dtype=torch.float32, device=bank.device)
    y = torch.empty((*lead, K, D), dtype=torch.bfloat16, device=bank.device)
    return y, torch.empty((N, K, S), **f32), torch.empty((N, S), **f32), torch.empty((N, K, S), **f32)


@torch.library.custom_op(f"{_NS}::read_selected_bwd", mutates_args=(), device_types="cuda")
def read_selected_bwd(values: List[Tensor], bank: Tensor, ids: Tensor, dy: Tensor, alpha: Tensor,
                      rstd: Tensor, logit: Tensor, eps: float, scale: float,
                      key_offset: int, packed: bool) -> Tuple[List[Tensor], Tensor, Tensor]:
    S, D, packed, lead = _shape_info(values, packed)
    saved = {"alpha": alpha, "rstd": rstd, "logit": logit}
    g = _ops.attnres_selected_bwd(_as_values(values, packed), bank, ids, dy.contiguous(), saved, eps=eps,
                                  scale=scale, key_offset=key_offset)
    dv = [g["dvalues"]] if packed else list(g["dvalues"])
    return dv, g["dbank"], g["dbank_f32"]


@read_selected_bwd.register_fake
def _(values, bank, ids, dy, alpha, rstd, logit, eps, scale, key_offset, packed):
    return ([torch.empty_like(v) for v in values], torch.empty_like(bank),
            torch.empty(bank.shape, dtype=torch.float32, device=bank.device))


def _sel_setup_context(ctx, inputs, output):
    values, bank, ids, eps, scale, key_offset, packed = inputs
    y, alpha, rstd, logit = output
    ctx.cfg = (eps, scale, key_offset, packed)
    ctx.save_for_backward(bank, ids, alpha, rstd, logit, *values)


def _sel_backward(ctx, dy, d_alpha, d_rstd, d_logit):
    bank, ids, alpha, rstd, logit, *values = ctx.saved_tensors
    eps, scale, key_offset, packed = ctx.cfg
    dv, db, _ = read_selected_bwd(list(values), bank, ids, dy.to(torch.bfloat16), alpha, rstd, logit, eps,
                                  scale, key_offset, packed)
    return list(dv), db, None, None, None, None, None


read_selected_fwd.register_autograd(_sel_backward, setup_context=_sel_setup_context)


def attnres_selected_op(values, query_bank: Tensor, ids: Tensor, *, eps: float = _ops.EPS_DEFAULT,
                        scale: float = 1.0, key_offset: Optional[int] = None) -> Tensor:
    """The selected-query read through the registered operator."""
    vals, packed = _pack_args(values)
    D = vals[0].shape[-1]
    ko = D - query_bank.shape[-1] if key_offset is None else int(key_offset)
    return read_selected_fwd(vals, query_bank, ids, float(eps), float(scale), ko, packed)[0]


# --------------------------------------------------------------------------
# Fused block-partial read ("Fast Attention Residuals", section "Full and
# Block schedules")
# --------------------------------------------------------------------------
@torch.library.custom_op(f"{_NS}::read_block_fwd", mutates_args=(), device_types="cuda")
def read_block_fwd(values: List[Tensor], delta: Tensor, q: Tensor, w_o: Optional[Tensor], eps: float,
                   scale: float, key_offset: int) -> Tuple[Tensor, Tensor, Tensor, Tensor, Tensor, Tensor,
                                                           Tensor]:
    r = _ops.attnres_partial_fwd(list(values[:-1]), values[-1], delta, q, w_o=w_o, eps=eps, scale=scale,
                                 key_offset=key_offset)
    empty = torch.empty((0,), dtype=torch.float32, device=q.device)
    o_rstd = r["o_rstd"] if r["o_rstd"] is not None else empty
    o_pre = r["o_pre"] if r["o_pre"] is not None else empty.clone()
    return r["y"], r["partial_new"], r["alpha"], r["rstd"], r["logit"], o_rstd, o_pre


@read_block_fwd.register_fake
def _(values, delta, q, w_o, eps, scale, key_offset):
    S, D = len(values), values[0].shape[-1]
    lead = tuple(values[0].shape[:-1])
    N = 1
    for d in lead:
        N *= d
    f32 = dict(dtype=torch.float32, device=q.device)
    y = torch.empty((*lead, D), dtype=torch.bfloat16, device=q.device)
    pn = torch.empty((*lead, D), dtype=torch.bfloat16, device=q.device)
    stats = [torch.empty((N, S), **f32) for _ in range(3)]
    if w_o is not None:
        o_rstd = torch.empty((N,), **f32)
        save = not _bwd_resident(S, D, q.numel(), key_offset, True)
        o_pre = torch.empty((N, D) if save else (0,), **f32)
    else:
        o_rstd = torch.empty((0,), **f32)
        o_pre = torch.empty((0,), **f32)
    return y, pn, stats[0], stats[1], stats[2], o_rstd, o_pre


@torch.library.custom_op(f"{_NS}::read_block_bwd", mutates_args=(), device_types="cuda")
def read_block_bwd(completed: List[Tensor], partial_new: Tensor, q: Tensor, w_o: Optional[Tensor], dy: Tensor,
                   g_partial: Optional[Tensor], alpha: Tensor, rstd: Tensor, logit: Tensor, o_rstd: Tensor,
                   o_pre: Tensor, eps: float, scale: float,
                   key_offset: int) -> Tuple[List[Tensor], Tensor, Tensor, Tensor, Tensor, Tensor]:
    saved = {"alpha": alpha, "rstd": rstd, "logit": logit,
             "o_rstd": o_rstd if o_rstd.numel() else None, "o_pre": o_pre if o_pre.numel() else None}
    g = _ops.attnres_partial_bwd(list(completed), partial_new, q, dy, saved, g_partial=g_partial, w_o=w_o,
                                 eps=eps, scale=scale, key_offset=key_offset)
    dw = g["dw_o"] if g["dw_o"] is not None else torch.empty((0,), dtype=torch.bfloat16, device=q.device)
    dw32 = g["dw_o_f32"] if g["dw_o_f32"] is not None else torch.empty((0,), dtype=torch.float32,
                                                                        device=q.device)
    return g["d_completed"], g["d_partial"], g["dq"].view_as(q), dw, g["dq_f32"].view(q.shape), dw32


@read_block_bwd.register_fake
def _(completed, partial_new, q, w_o, dy, g_partial, alpha, rstd, logit, o_rstd, o_pre, eps, scale, key_offset):
    dw = torch.empty_like(w_o) if w_o is not None else torch.empty((0,), dtype=torch.bfloat16, device=q.device)
    f32 = dict(dtype=torch.float32, device=q.device)
    dw32 = torch.empty(w_o.shape if w_o is not None else (0,), **f32)
    return ([torch.empty_like(c) for c in completed], torch.empty_like(partial_new), torch.empty_like(q), dw,
            torch.empty(q.shape, **f32), dw32)


def _block_setup_context(ctx, inputs, output):
    values, delta, q, w_o, eps, scale, key_offset = inputs
    y, partial_new, alpha, rstd, logit, o_rstd, o_pre = output
    ctx.cfg = (eps, scale, key_offset)
    ctx.has_w = w_o is not None
    ctx.ncomp = len(values) - 1
    ctx.save_for_backward(q, w_o if w_o is not None else q.new_empty((0,)), partial_new, alpha, rstd, logit,
                          o_rstd, o_pre, *values[:-1])


def _block_backward(ctx, dy, d_partial_new, d_alpha, d_rstd, d_logit, d_orstd, d_opre):
    q, w_o, partial_new, alpha, rstd, logit, o_rstd, o_pre, *completed = ctx.saved_tensors
    eps, scale, key_offset = ctx.cfg
    if dy is None:
        dy = torch.zeros_like(partial_new)
    g = None if d_partial_new is None else d_partial_new.to(torch.bfloat16)
    dcomp, dpart, dq, dw, _, _ = read_block_bwd(list(completed), partial_new, q, w_o if ctx.has_w else None,
                                                dy.to(torch.bfloat16), g, alpha, rstd, logit, o_rstd, o_pre,
                                                eps, scale, key_offset)
    return list(dcomp) + [dpart], dpart, dq, (dw if ctx.has_w else None), None, None, None


read_block_fwd.register_autograd(_block_backward, setup_context=_block_setup_context)


def attnres_block_read_op(completed, partial: Tensor, delta: Tensor, query: Tensor, *,
                          eps: float = _ops.EPS_DEFAULT, scale: float = 1.0,
                          out_norm_weight: Optional[Tensor] = None, key_offset: Optional[int] = None):
    """The fused block-partial read through the registered operator."""
    if isinstance(completed, Tensor):
        comp = list(completed.unbind(0)) if completed.dim() == partial.dim() + 1 else [completed]
    else:
        comp = list(completed)
    D = partial.shape[-1]
    ko = D - query.numel() if key_offset is None else int(key_offset)
    out = read_block_fwd(comp + [partial], delta, query, out_norm_weight, float(eps), float(scale), ko)
    return out[0], out[1]
