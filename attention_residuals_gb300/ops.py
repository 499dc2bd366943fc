"""Python binding of the C ABI (same names), plus the autograd operator.

PyTorch provides device memory, the current stream and autograd plumbing;
the binding only marshals pointers and sizes.  Every step of the operator
("Fast Attention Residuals", section "Equation", with the optional output
RMSNorm of "[Perf] Parallelize AttnRes long-sequence reduction") runs in the
CUDA library.  There is no CPU path: CPU tensors are rejected.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Optional, Sequence, Union

import torch

from . import _lib

EPS_DEFAULT = 2.0 ** -23
Sources = Union[torch.Tensor, Sequence[torch.Tensor]]


# --------------------------------------------------------------------------
# Source marshalling
# --------------------------------------------------------------------------
@dataclass
class _SourceView:
    rows: List[torch.Tensor]   # S tensors viewed as [N, D] with a common row stride
    packed: bool
    lead_shape: tuple          # leading (token) shape of one source
    N: int
    D: int
    ld: int


def _as_rows(t: torch.Tensor, D: int) -> torch.Tensor:
    if t.shape[-1] != D:
        raise ValueError("every source must have the same last dimension D")
    if t.dim() == 1:
        t = t.unsqueeze(0)
    r = t.reshape(-1, D) if t.is_contiguous() else None
    if r is None:
        try:
            r = t.view(-1, D)
        except RuntimeError:
            r = None
    if r is None or r.stride(1) != 1 or (r.shape[0] > 1 and r.stride(0) < D):
        r = t.contiguous().view(-1, D)
    return r


def _source_view(values: Sources) -> _SourceView:
    if isinstance(values, torch.Tensor):
        if values.dim() < 2:
            raise ValueError("packed values must be [S, ..., D]")
        S, D = values.shape[0], values.shape[-1]
        lead = tuple(values.shape[1:-1])
        rows = [_as_rows(values[s], D) for s in range(S)]
        packed = True
    else:
        vals = list(values)
        if not vals:
            raise ValueError("need at least one source")
        D = vals[0].shape[-1]
        lead = tuple(vals[0].shape[:-1])
        for v in vals:
            if tuple(v.shape[:-1]) != lead:
                raise ValueError("all sources must have the same shape")
        rows = [_as_rows(v, D) for v in vals]
        packed = False
    for r in rows:
        if r.dtype != torch.bfloat16:
            raise TypeError("sources must be torch.bfloat16")
        if not r.is_cuda:
            raise TypeError("sources must be CUDA tensors (the operator has no CPU path)")
    N = rows[0].shape[0]
    lds = {int(r.stride(0)) if r.shape[0] > 1 else D for r in rows}
    if len(lds) != 1 or any(r.data_ptr() % 16 for r in rows) or next(iter(lds)) % 8:
        rows = [r.contiguous() for r in rows]
        lds = {D}
    return _SourceView(rows=rows, packed=packed, lead_shape=lead, N=N, D=D, ld=next(iter(lds)))


def make_params(view: _SourceView, R: int, *, key_offset: Optional[int], eps: float, scale: float,
                out_norm: bool, split_n_threshold: int = 0) -> _lib.AttnresParams:
    S = len(view.rows)
    if S > _lib.MAX_S:
        raise ValueError(f"at most {_lib.MAX_S} sources")
    p = _lib.AttnresParams()
    p.S = S
    p.D = view.D
    p.R = int(R)
    p.key_offset = view.D - int(R) if key_offset is None else int(key_offset)
    p.N = view.N
    p.eps = float(eps)
    p.scale = float(scale)
    p.out_norm = 1 if out_norm else 0
    p.split_n_threshold = int(split_n_threshold)
    p.src_ld = view.ld
    for s, r in enumerate(view.rows):
        p.src[s] = r.data_ptr()
    return p


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check_vec(t: Optional[torch.Tensor], n: int, name: str):
    if t is None:
        return None
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.numel() != n:
        raise TypeError(f"{name} must be a CUDA bf16 tensor with {n} elements")
    return t.contiguous()


def _check_out(t: Optional[torch.Tensor], n: int, dtype: torch.dtype, name: str, device) -> None:
    """A caller-supplied output: contiguous, on the sources' device, n elements of dtype."""
    if t is None:
        return
    if t.dtype != dtype or t.device != device or t.numel() != n or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous {dtype} tensor with {n} elements on {device}")


def _out_rows(t: torch.Tensor, N: int, D: int, name: str) -> torch.Tensor:
    """[N, D] rows of a caller-supplied gradient buffer, without a copy: the
    kernel writes through this view, so a copy would leave the caller's
    buffer untouched."""
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.numel() != N * D:
        raise TypeError(f"{name} must be a CUDA bf16 tensor of {N} rows of {D}")
    try:
        r = t.view(N, D)
    except RuntimeError as e:
        raise ValueError(f"{name}: rows must be addressable as [N, D] with unit column stride") from e
    if N > 1 and r.stride(1) != 1:
        raise ValueError(f"{name}: rows must have unit column stride")
    return r


# --------------------------------------------------------------------------
# C-ABI mirrors
# --------------------------------------------------------------------------
_PLAN_KEYS = ["grid", "consumer_warps", "vectors_per_thread", "bwd_ring", "fwd_ring",
              "bwd_resident", "bwd_smem_bytes", "bwd_split", "bwd_cluster", "bwd_partial_rows"]


def _plan(p: _lib.AttnresParams) -> dict:
    out = (ctypes.c_int64 * 10)()
    _lib.check(_lib.load().attnres_plan_info(ctypes.byref(p), out), "attnres_plan_info")
    return dict(zip(_PLAN_KEYS, list(out)))


def attnres_plan_info(values: Sources, R: int, *, key_offset=None, out_norm=False,
                      split_n_threshold=0) -> dict:
    view = _source_view(values)
    p = make_params(view, R, key_offset=key_offset, eps=EPS_DEFAULT, scale=1.0, out_norm=out_norm,
                    split_n_threshold=split_n_threshold)
    return _plan(p)


def attnres_bwd_workspace_bytes(params: _lib.AttnresParams) -> int:
    return int(_lib.load().attnres_bwd_workspace_bytes(ctypes.byref(params)))


def attnres_check_device_error() -> None:
    _lib.check(_lib.load().attnres_check_device_error(), "attnres_check_device_error")


def attnres_jit_kernel_count() -> int:
    """Forward kernels compiled at run time for exact plan shapes in this process."""
    return int(_lib.load().attnres_jit_kernel_count())


def attnres_fwd(values: Sources, q: torch.Tensor, *, w_o: Optional[torch.Tensor] = None,
                eps: float = EPS_DEFAULT, scale: float = 1.0, key_offset: Optional[int] = None,
                save_o_pre: Optional[bool] = None, stream=None, out: Optional[dict] = None) -> dict:
    """Forward read.  Returns y [..., D] bf16 and the saved statistics
    alpha/rstd/logit [N, S] f32 and, with w_o, o_rstd [N] f32 and optionally
    the FP32 pre-norm mixture o_pre [N, D].  save_o_pre=None saves o_pre only
    when the backward cannot keep a token's rows resident (then it spares the
    backward a pass over the sources).  ``out`` may supply preallocated
    tensors."""
    view = _source_view(values)
    R = q.numel()
    q = _check_vec(q, R, "q")
    w_o = _check_vec(w_o, view.D, "w_o")
    p = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=w_o is not None)
    dev = view.rows[0].device
    S, N, D = len(view.rows), view.N, view.D
    o = dict(out or {})
    y = o.get("y")
    if y is None:
        y = torch.empty((N, D), dtype=torch.bfloat16, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    alpha = o.get("alpha") if o.get("alpha") is not None else torch.empty((N, S), **f32)
    rstd = o.get("rstd") if o.get("rstd") is not None else torch.empty((N, S), **f32)
    logit = o.get("logit") if o.get("logit") is not None else torch.empty((N, S), **f32)
    o_rstd = o_pre = None
    if w_o is not None:
        o_rstd = o.get("o_rstd") if o.get("o_rstd") is not None else torch.empty((N,), **f32)
        if save_o_pre is None:
            save_o_pre = N > 0 and not _plan(p)["bwd_resident"]
        if save_o_pre:
            o_pre = o.get("o_pre") if o.get("o_pre") is not None else torch.empty((N, D), **f32)
    rc = _lib.load().attnres_fwd(ctypes.byref(p), _ptr(q), _ptr(w_o), _ptr(y), _ptr(alpha),
                                 _ptr(rstd), _ptr(logit), _ptr(o_rstd), _ptr(o_pre), _stream(stream))
    _lib.check(rc, "attnres_fwd")
    return {"y": y.view(*view.lead_shape, D) if view.lead_shape else y.view(D),
            "alpha": alpha, "rstd": rstd, "logit": logit, "o_rstd": o_rstd, "o_pre": o_pre,
            "params": p, "view": view}


def attnres_bwd(values: Sources, q: torch.Tensor, dy: torch.Tensor, saved: dict, *,
                w_o: Optional[torch.Tensor] = None, eps: float = EPS_DEFAULT, scale: float = 1.0,
                key_offset: Optional[int] = None, split_n_threshold: int = 0, stream=None,
                dvalues: Optional[Sources] = None, workspace: Optional[torch.Tensor] = None) -> dict:
    """Backward.  ``saved`` is attnres_fwd's result for the same sources.
    Returns dvalues (packed [S, ..., D] if the sources were packed, else a
    list), dq/dw_o in bf16 and fp32."""
    view = saved.get("view") or _source_view(values)
    R = q.numel()
    q = _check_vec(q, R, "q")
    w_o = _check_vec(w_o, view.D, "w_o")
    p = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=w_o is not None,
                    split_n_threshold=split_n_threshold)
    S, N, D = len(view.rows), view.N, view.D
    dev = view.rows[0].device
    if dy.dtype != torch.bfloat16 or not dy.is_cuda or dy.numel() != N * D:
        raise TypeError("dy must be a CUDA bf16 tensor shaped like the output")
    dy2 = dy.reshape(N, D).contiguous()
    if dvalues is None:
        if view.packed:
            dpacked = torch.empty((S, N, D), dtype=torch.bfloat16, device=dev)
            drows = [dpacked[s] for s in range(S)]
        else:
            dpacked = None
            drows = [torch.empty((N, D), dtype=torch.bfloat16, device=dev) for _ in range(S)]
    else:
        if isinstance(dvalues, torch.Tensor):
            dpacked = dvalues
            drows = [_out_rows(dvalues[s], N, D, "dvalues") for s in range(S)]
        else:
            dpacked = None
            drows = [_out_rows(d, N, D, "dvalues") for d in dvalues]
    dld = int(drows[0].stride(0)) if N > 1 else D
    if N > 1 and any(int(r.stride(0)) != dld for r in drows):
        raise ValueError("dvalues: every source's gradient rows need the same row stride")
    dptrs = (ctypes.c_void_p * S)(*[r.data_ptr() for r in drows])
    dq = torch.empty((R,), dtype=torch.bfloat16, device=dev)
    dq32 = torch.empty((R,), dtype=torch.float32, device=dev)
    dw = dw32 = None
    if w_o is not None:
        dw = torch.empty((D,), dtype=torch.bfloat16, device=dev)
        dw32 = torch.empty((D,), dtype=torch.float32, device=dev)
    need = attnres_bwd_workspace_bytes(p)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    rc = _lib.load().attnres_bwd(
        ctypes.byref(p), _ptr(q), _ptr(w_o), _ptr(dy2), _ptr(saved["alpha"]), _ptr(saved["rstd"]),
        _ptr(saved["logit"]), _ptr(saved.get("o_rstd")), _ptr(saved.get("o_pre")), dptrs,
        ctypes.c_int64(dld), _ptr(dq), _ptr(dq32), _ptr(dw), _ptr(dw32), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    _lib.check(rc, "attnres_bwd")
    shape = (*view.lead_shape, D)
    if dpacked is not None:
        dv = dpacked.view(S, *shape)
    else:
        dv = [r.view(*shape) for r in drows]
    return {"dvalues": dv, "dq": dq, "dq_f32": dq32, "dw_o": dw, "dw_o_f32": dw32}


def attnres_bwd_noalloc(values: Sources, q: torch.Tensor, dy: torch.Tensor, saved: dict, *,
                        w_o: Optional[torch.Tensor] = None, eps: float = EPS_DEFAULT,
                        scale: float = 1.0, key_offset: Optional[int] = None,
                        split_n_threshold: int = 0, stream=None, dvalues: Optional[Sources] = None,
                        dq: Optional[torch.Tensor] = None, dq_f32: Optional[torch.Tensor] = None,
                        dw_o: Optional[torch.Tensor] = None,
                        dw_o_f32: Optional[torch.Tensor] = None) -> dict:
    """Backward through the library's fixed scratch array instead of a
    workspace, for callers that must not allocate device memory during the
    call (pass every output preallocated).  Calls sharing the array must not
    overlap on the GPU; see include/attnres.h."""
    view = saved.get("view") or _source_view(values)
    R = q.numel()
    q = _check_vec(q, R, "q")
    w_o = _check_vec(w_o, view.D, "w_o")
    p = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=w_o is not None,
                    split_n_threshold=split_n_threshold)
    S, N, D = len(view.rows), view.N, view.D
    dev = view.rows[0].device
    if dy.dtype != torch.bfloat16 or not dy.is_cuda or dy.numel() != N * D:
        raise TypeError("dy must be a CUDA bf16 tensor shaped like the output")
    if not dy.is_contiguous():
        raise ValueError("dy must be contiguous (the no-allocation path makes no copies)")
    dy2 = dy.view(N, D)
    if dvalues is None or dq is None or (w_o is not None and dw_o is None):
        raise ValueError("the no-allocation path needs preallocated dvalues, dq (and dw_o)")
    _check_out(dq, R, torch.bfloat16, "dq", dev)
    _check_out(dq_f32, R, torch.float32, "dq_f32", dev)
    _check_out(dw_o, D, torch.bfloat16, "dw_o", dev)
    _check_out(dw_o_f32, D, torch.float32, "dw_o_f32", dev)
    if isinstance(dvalues, torch.Tensor):
        drows = [_out_rows(dvalues[s], N, D, "dvalues") for s in range(S)]
    else:
        drows = [_out_rows(d, N, D, "dvalues") for d in dvalues]
    dld = int(drows[0].stride(0)) if N > 1 else D
    if N > 1 and any(int(r.stride(0)) != dld for r in drows):
        raise ValueError("dvalues: every source's gradient rows need the same row stride")
    dptrs = (ctypes.c_void_p * S)(*[r.data_ptr() for r in drows])
    rc = _lib.load().attnres_bwd_noalloc(
        ctypes.byref(p), _ptr(q), _ptr(w_o), _ptr(dy2), _ptr(saved["alpha"]), _ptr(saved["rstd"]),
        _ptr(saved["logit"]), _ptr(saved.get("o_rstd")), _ptr(saved.get("o_pre")), dptrs,
        ctypes.c_int64(dld), _ptr(dq), _ptr(dq_f32), _ptr(dw_o), _ptr(dw_o_f32), _stream(stream))
    _lib.check(rc, "attnres_bwd_noalloc")
    return {"dvalues": dvalues, "dq": dq, "dq_f32": dq_f32, "dw_o": dw_o, "dw_o_f32": dw_o_f32}


# --------------------------------------------------------------------------
# Training step from host memory (pipelined transfers; see attnres_step_host
# in include/attnres.h)
# --------------------------------------------------------------------------
_copy_streams = {}


def _host_rows(values) -> tuple:
    vals = list(values.unbind(0)) if isinstance(values, torch.Tensor) else list(values)
    D = vals[0].shape[-1]
    rows = []
    for v in vals:
        if v.is_cuda or v.dtype != torch.bfloat16:
            raise TypeError("host sources must be CPU bf16 tensors (pinned for full speed)")
        if not v.is_contiguous():
            raise ValueError("host sources must be contiguous")
        rows.append(v.view(-1, D))
    return vals, rows, D


def attnres_step_host_workspace_bytes(params: _lib.AttnresParams, chunk_tokens: int) -> int:
    return int(_lib.load().attnres_step_host_workspace_bytes(ctypes.byref(params), ctypes.c_int64(chunk_tokens)))


def attnres_step_host(values, q: torch.Tensor, dy: torch.Tensor, *, w_o: Optional[torch.Tensor] = None,
                      eps: float = EPS_DEFAULT, scale: float = 1.0, key_offset: Optional[int] = None,
                      chunk_tokens: int = 4096, out: Optional[dict] = None,
                      workspace: Optional[torch.Tensor] = None, device=None) -> dict:
    """Forward + backward of the read with every input and output in host
    memory (page-locked CPU tensors), transfers overlapped with the kernels
    chunk by chunk.  Asynchronous on the current CUDA stream (synchronise it
    before reading the outputs).  Returns host tensors y, dvalues (a list),
    dq, dq_f32, dw_o, dw_o_f32."""
    vals, rows, D = _host_rows(values)
    S = len(rows)
    N = rows[0].shape[0]
    R = q.numel()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    p = _lib.AttnresParams()
    p.S, p.D, p.R = S, D, R
    p.key_offset = D - R if key_offset is None else int(key_offset)
    p.N, p.eps, p.scale = N, float(eps), float(scale)
    p.out_norm = 1 if w_o is not None else 0
    p.split_n_threshold, p.src_ld = 0, D
    for i, r in enumerate(rows):
        p.src[i] = r.data_ptr()
    o = dict(out or {})
    pin = dict(dtype=torch.bfloat16, pin_memory=True)
    y = o.get("y") if o.get("y") is not None else torch.empty((N, D), **pin)
    dv = o.get("dvalues") if o.get("dvalues") is not None else [torch.empty((N, D), **pin) for _ in range(S)]
    dq = o.get("dq") if o.get("dq") is not None else torch.empty((R,), **pin)
    dq32 = o.get("dq_f32") if o.get("dq_f32") is not None else torch.empty((R,), dtype=torch.float32,
                                                                           pin_memory=True)
    dw = dw32 = None
    if w_o is not None:
        dw = o.get("dw_o") if o.get("dw_o") is not None else torch.empty((D,), **pin)
        dw32 = o.get("dw_o_f32") if o.get("dw_o_f32") is not None else torch.empty((D,), dtype=torch.float32,
                                                                                   pin_memory=True)
    need = attnres_step_host_workspace_bytes(p, chunk_tokens)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    if dev.index not in _copy_streams:
        _copy_streams[dev.index] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    s_in, s_out = _copy_streams[dev.index]
    streams = (ctypes.c_void_p * 3)(torch.cuda.current_stream(dev).cuda_stream, s_in.cuda_stream,
                                    s_out.cuda_stream)
    dptrs = (ctypes.c_void_p * S)(*[d.data_ptr() for d in dv])
    # keep every host buffer the enqueued copies read alive with the result
    keep = (q.contiguous(), None if w_o is None else w_o.contiguous(), dy.reshape(N, D).contiguous())
    rc = _lib.load().attnres_step_host(
        ctypes.byref(p), _ptr(keep[0]), _ptr(keep[1]),
        _ptr(keep[2]), ctypes.c_int64(D), _ptr(y), ctypes.c_int64(D), dptrs, ctypes.c_int64(D),
        _ptr(dq), _ptr(dq32), _ptr(dw), _ptr(dw32), ctypes.c_int64(chunk_tokens), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), streams)
    _lib.check(rc, "attnres_step_host")
    return {"y": y, "dvalues": dv, "dq": dq, "dq_f32": dq32, "dw_o": dw, "dw_o_f32": dw32,
            "workspace": workspace, "inputs": (vals, keep)}


# --------------------------------------------------------------------------
# Fused block-partial read ("Fast Attention Residuals", section "Full and
# Block schedules": the caller's partial-block sum formed inside the read)
# --------------------------------------------------------------------------
def _row2d(t: torch.Tensor, N: int, D: int, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.numel() != N * D:
        raise TypeError(f"{name} must be a CUDA bf16 tensor shaped like one source")
    r = t.reshape(N, D)
    return r if (r.is_contiguous() and r.data_ptr() % 16 == 0) else r.contiguous()


def attnres_partial_fwd(completed: Sources, partial: torch.Tensor, delta: torch.Tensor, q: torch.Tensor, *,
                        w_o: Optional[torch.Tensor] = None, eps: float = EPS_DEFAULT, scale: float = 1.0,
                        key_offset: Optional[int] = None, partial_out: Optional[torch.Tensor] = None,
                        stream=None) -> dict:
    """Fused block-partial forward: partial_new = partial + delta (bf16 add)
    is formed inside the read of (completed..., partial_new).  Returns y,
    partial_new and the saved statistics (as attnres_fwd).  partial_out may
    be given (even `partial` itself, for an in-place update)."""
    comp = [completed] if isinstance(completed, torch.Tensor) and completed.dim() == partial.dim() else completed
    comp = list(comp.unbind(0)) if isinstance(comp, torch.Tensor) else list(comp)
    view = _source_view(comp + [partial])
    N, D = view.N, view.D
    R = q.numel()
    q = _check_vec(q, R, "q")
    w_o = _check_vec(w_o, D, "w_o")
    d2 = _row2d(delta, N, D, "delta")
    if partial_out is None:
        pout = torch.empty((N, D), dtype=torch.bfloat16, device=view.rows[0].device)
    else:
        # written in place: a view of the caller's buffer, never a copy
        pout = _out_rows(partial_out, N, D, "partial_out")
        if (N > 1 and pout.stride(0) != D) or pout.data_ptr() % 16:
            raise ValueError("partial_out must be contiguous [.., D] rows starting on 16 bytes")
    p = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=w_o is not None)
    S, dev = len(view.rows), view.rows[0].device
    f32 = dict(dtype=torch.float32, device=dev)
    y = torch.empty((N, D), dtype=torch.bfloat16, device=dev)
    alpha, rstd, logit = (torch.empty((N, S), **f32) for _ in range(3))
    o_rstd = o_pre = None
    if w_o is not None:
        o_rstd = torch.empty((N,), **f32)
        if N > 0 and not _plan(p)["bwd_resident"]:
            o_pre = torch.empty((N, D), **f32)
    rc = _lib.load().attnres_fwd_partial(ctypes.byref(p), _ptr(q), _ptr(w_o), _ptr(d2), ctypes.c_int64(D),
                                         _ptr(pout), ctypes.c_int64(D), _ptr(y), _ptr(alpha), _ptr(rstd),
                                         _ptr(logit), _ptr(o_rstd), _ptr(o_pre), _stream(stream))
    _lib.check(rc, "attnres_fwd_partial")
    shape = (*view.lead_shape, D)
    return {"y": y.view(shape), "partial_new": pout.view(shape), "alpha": alpha, "rstd": rstd,
            "logit": logit, "o_rstd": o_rstd, "o_pre": o_pre}


def attnres_partial_bwd(completed: Sources, partial_new: torch.Tensor, q: torch.Tensor, dy: torch.Tensor,
                        saved: dict, *, g_partial: Optional[torch.Tensor] = None,
                        w_o: Optional[torch.Tensor] = None, eps: float = EPS_DEFAULT, scale: float = 1.0,
                        key_offset: Optional[int] = None, stream=None) -> dict:
    """Backward of the fused block-partial read.  Returns d_completed (a
    list), d_partial (the gradient of both `partial` and `delta`, including
    g_partial, the gradient reaching partial_new from its later uses), dq
    and dw_o (bf16 and fp32)."""
    comp = list(completed.unbind(0)) if (isinstance(completed, torch.Tensor) and
                                         completed.dim() == partial_new.dim() + 1) else list(completed)
    view = _source_view(comp + [partial_new])
    N, D = view.N, view.D
    R = q.numel()
    q = _check_vec(q, R, "q")
    w_o = _check_vec(w_o, D, "w_o")
    p = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=w_o is not None)
    S, dev = len(view.rows), view.rows[0].device
    dy2 = _row2d(dy, N, D, "dy")
    g2 = None if g_partial is None else _row2d(g_partial, N, D, "g_partial")
    drows = [torch.empty((N, D), dtype=torch.bfloat16, device=dev) for _ in range(S)]
    dptrs = (ctypes.c_void_p * S)(*[r.data_ptr() for r in drows])
    dq = torch.empty((R,), dtype=torch.bfloat16, device=dev)
    dq32 = torch.empty((R,), dtype=torch.float32, device=dev)
    dw = dw32 = None
    if w_o is not None:
        dw = torch.empty((D,), dtype=torch.bfloat16, device=dev)
        dw32 = torch.empty((D,), dtype=torch.float32, device=dev)
    need = attnres_bwd_workspace_bytes(p)
    ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    rc = _lib.load().attnres_bwd_partial(
        ctypes.byref(p), _ptr(q), _ptr(w_o), _ptr(dy2), _ptr(saved["alpha"]), _ptr(saved["rstd"]),
        _ptr(saved["logit"]), _ptr(saved.get("o_rstd")), _ptr(saved.get("o_pre")), _ptr(g2),
        ctypes.c_int64(D), dptrs, ctypes.c_int64(D), _ptr(dq), _ptr(dq32), _ptr(dw), _ptr(dw32), _ptr(ws),
        ctypes.c_size_t(ws.numel()), _stream(stream))
    _lib.check(rc, "attnres_bwd_partial")
    shape = (*view.lead_shape, D)
    return {"d_completed": [r.view(shape) for r in drows[:-1]], "d_partial": drows[-1].view(shape),
            "dq": dq, "dq_f32": dq32, "dw_o": dw, "dw_o_f32": dw32}


# --------------------------------------------------------------------------
# Multi-query read ("Fast Attention Residuals", section "Multi-query AttnRes")
# --------------------------------------------------------------------------
_MULTI_PLAN_KEYS = ["grid", "consumer_warps", "vectors_per_thread", "query_blocks", "fwd_ring",
                    "bwd_ring", "dy_slots", "bwd_smem_bytes", "bwd_general", "bwd_token_groups"]


def make_multi_params(view: _SourceView, M: int, R: int, *, key_offset: Optional[int], eps: float,
                      scale: float, token_major: bool) -> _lib.AttnresMultiParams:
    mp = _lib.AttnresMultiParams()
    mp.base = make_params(view, R, key_offset=key_offset, eps=eps, scale=scale, out_norm=False)
    mp.M = int(M)
    N, D = view.N, view.D
    if token_major:             # [N, M, D]
        mp.out_ld_m, mp.out_ld_n = D, M * D
    else:                       # [M, N, D]
        mp.out_ld_m, mp.out_ld_n = N * D, D
    return mp


def _check_queries(queries: torch.Tensor, D: int) -> torch.Tensor:
    if queries.dim() != 2:
        raise ValueError("queries must be [M, R]")
    M, R = queries.shape
    if not (1 <= M <= _lib.MAX_M) or not (1 <= R <= D):
        raise ValueError(f"queries must be [M, R] with 1 <= M <= {_lib.MAX_M}, 1 <= R <= D")
    if queries.dtype != torch.bfloat16 or not queries.is_cuda:
        raise TypeError("queries must be a CUDA bf16 tensor")
    return queries.contiguous()


def attnres_multi_plan_info(values: Sources, M: int, R: int, *, key_offset=None) -> dict:
    view = _source_view(values)
    mp = make_multi_params(view, M, R, key_offset=key_offset, eps=EPS_DEFAULT, scale=1.0,
                           token_major=False)
    out = (ctypes.c_int64 * 10)()
    lib = _lib.load()
    _lib.check(lib.attnres_multi_plan_info(ctypes.byref(mp), out), "attnres_multi_plan_info")
    info = dict(zip(_MULTI_PLAN_KEYS, list(out)))
    info["fwd_tensor_cores"] = int(lib.attnres_multi_fwd_tensor_cores(ctypes.byref(mp), ctypes.c_int32(0)))
    return info


def attnres_multi_bwd_workspace_bytes(params: _lib.AttnresMultiParams) -> int:
    return int(_lib.load().attnres_multi_bwd_workspace_bytes(ctypes.byref(params)))


def _multi_out_shape(view: _SourceView, M: int, token_major: bool):
    return (*view.lead_shape, M, view.D) if token_major else (M, *view.lead_shape, view.D)


def attnres_multi_fwd(values: Sources, queries: torch.Tensor, *, eps: float = EPS_DEFAULT,
                      scale: float = 1.0, key_offset: Optional[int] = None, token_major: bool = False,
                      stream=None) -> dict:
    """Multi-query forward.  Returns y ([M, ..., D], or [..., M, D] when
    token_major) and the saved statistics alpha/logit [N, M, S] and
    rstd [N, S] (f32)."""
    view = _source_view(values)
    queries = _check_queries(queries, view.D)
    M, R = queries.shape
    mp = make_multi_params(view, M, R, key_offset=key_offset, eps=eps, scale=scale,
                           token_major=token_major)
    dev = view.rows[0].device
    S, N, D = len(view.rows), view.N, view.D
    y = torch.empty((N, M, D) if token_major else (M, N, D), dtype=torch.bfloat16, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    alpha = torch.empty((N, M, S), **f32)
    rstd = torch.empty((N, S), **f32)
    logit = torch.empty((N, M, S), **f32)
    rc = _lib.load().attnres_multi_fwd(ctypes.byref(mp), _ptr(queries), _ptr(y), _ptr(alpha),
                                       _ptr(rstd), _ptr(logit), _stream(stream))
    _lib.check(rc, "attnres_multi_fwd")
    return {"y": y.view(_multi_out_shape(view, M, token_major)), "alpha": alpha, "rstd": rstd,
            "logit": logit, "params": mp, "view": view, "token_major": token_major}


def attnres_multi_bwd(values: Sources, queries: torch.Tensor, dy: torch.Tensor, saved: dict, *,
                      eps: float = EPS_DEFAULT, scale: float = 1.0, key_offset: Optional[int] = None,
                      token_major: Optional[bool] = None, stream=None,
                      workspace: Optional[torch.Tensor] = None) -> dict:
    """Multi-query backward.  ``saved`` is attnres_multi_fwd's result; dy
    has the output's shape and layout.  Returns dvalues (packed or a list,
    like the sources; the sum over queries) and dq [M, R] in bf16 and fp32."""
    view = saved.get("view") or _source_view(values)
    queries = _check_queries(queries, view.D)
    M, R = queries.shape
    tm = saved.get("token_major", False) if token_major is None else token_major
    mp = make_multi_params(view, M, R, key_offset=key_offset, eps=eps, scale=scale, token_major=tm)
    S, N, D = len(view.rows), view.N, view.D
    dev = view.rows[0].device
    if dy.dtype != torch.bfloat16 or not dy.is_cuda or dy.numel() != M * N * D:
        raise TypeError("dy must be a CUDA bf16 tensor shaped like the output")
    dy3 = dy.reshape((N, M, D) if tm else (M, N, D)).contiguous()
    if view.packed:
        dpacked = torch.empty((S, N, D), dtype=torch.bfloat16, device=dev)
        drows = [dpacked[s] for s in range(S)]
    else:
        dpacked = None
        drows = [torch.empty((N, D), dtype=torch.bfloat16, device=dev) for _ in range(S)]
    dptrs = (ctypes.c_void_p * S)(*[r.data_ptr() for r in drows])
    dq = torch.empty((M, R), dtype=torch.bfloat16, device=dev)
    dq32 = torch.empty((M, R), dtype=torch.float32, device=dev)
    need = attnres_multi_bwd_workspace_bytes(mp)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    rc = _lib.load().attnres_multi_bwd(
        ctypes.byref(mp), _ptr(queries), _ptr(dy3), _ptr(saved["alpha"]), _ptr(saved["rstd"]),
        _ptr(saved["logit"]), dptrs, ctypes.c_int64(D), _ptr(dq), _ptr(dq32), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    _lib.check(rc, "attnres_multi_bwd")
    shape = (*view.lead_shape, D)
    dv = dpacked.view(S, *shape) if dpacked is not None else [r.view(*shape) for r in drows]
    return {"dvalues": dv, "dq": dq, "dq_f32": dq32}


# --------------------------------------------------------------------------
# Selected-query read ("Fast Attention Residuals", section "Multi-query
# AttnRes": attnres_selected(sources, query_bank, ids) -> [..., K, D])
# --------------------------------------------------------------------------
def _check_bank_ids(bank: torch.Tensor, ids: torch.Tensor, view: _SourceView):
    if bank.dim() != 2 or not (1 <= bank.shape[1] <= view.D):
        raise ValueError("query_bank must be [E, R] with 1 <= R <= D")
    if bank.dtype != torch.bfloat16 or not bank.is_cuda:
        raise TypeError("query_bank must be a CUDA bf16 tensor")
    if ids.dtype not in (torch.int64, torch.int32, torch.int16, torch.uint8, torch.int8) or not ids.is_cuda:
        raise TypeError("ids must be a CUDA integer tensor")
    if tuple(ids.shape[:-1]) != tuple(view.lead_shape) or ids.dim() < 1:
        raise ValueError("ids must be [..., K] with the sources' leading shape")
    K = ids.shape[-1]
    if not (1 <= K <= _lib.MAX_M):
        raise ValueError(f"at most {_lib.MAX_M} selected queries per token")
    return bank.contiguous(), ids.reshape(view.N, K).to(torch.int64).contiguous(), K


def attnres_selected_fwd(values: Sources, bank: torch.Tensor, ids: torch.Tensor, *,
                         eps: float = EPS_DEFAULT, scale: float = 1.0, key_offset: Optional[int] = None,
                         stream=None) -> dict:
    """Selected-query forward: y [..., K, D] and the saved statistics
    alpha/logit [N, K, S], rstd [N, S] (f32).  An id outside [0, E) is
    reported by attnres_check_device_error()."""
    view = _source_view(values)
    bank, ids2, K = _check_bank_ids(bank, ids, view)
    E, R = bank.shape
    mp = make_multi_params(view, K, R, key_offset=key_offset, eps=eps, scale=scale, token_major=True)
    dev = view.rows[0].device
    S, N, D = len(view.rows), view.N, view.D
    y = torch.empty((N, K, D), dtype=torch.bfloat16, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    alpha = torch.empty((N, K, S), **f32)
    rstd = torch.empty((N, S), **f32)
    logit = torch.empty((N, K, S), **f32)
    rc = _lib.load().attnres_selected_fwd(ctypes.byref(mp), _ptr(bank), ctypes.c_int32(E), _ptr(ids2), _ptr(y),
                                          _ptr(alpha), _ptr(rstd), _ptr(logit), _stream(stream))
    _lib.check(rc, "attnres_selected_fwd")
    return {"y": y.view(*view.lead_shape, K, D), "alpha": alpha, "rstd": rstd, "logit": logit,
            "view": view, "ids": ids2}


def attnres_selected_bwd(values: Sources, bank: torch.Tensor, ids: torch.Tensor, dy: torch.Tensor,
                         saved: dict, *, eps: float = EPS_DEFAULT, scale: float = 1.0,
                         key_offset: Optional[int] = None, stream=None,
                         workspace: Optional[torch.Tensor] = None) -> dict:
    """Selected-query backward.  dy has the output's shape [..., K, D].
    Returns dvalues (packed or a list, like the sources) and dbank [E, R]
    in bf16 and fp32."""
    view = saved.get("view") or _source_view(values)
    bank, ids2, K = _check_bank_ids(bank, ids, view)
    E, R = bank.shape
    mp = make_multi_params(view, K, R, key_offset=key_offset, eps=eps, scale=scale, token_major=True)
    S, N, D = len(view.rows), view.N, view.D
    dev = view.rows[0].device
    if dy.dtype != torch.bfloat16 or not dy.is_cuda or dy.numel() != K * N * D:
        raise TypeError("dy must be a CUDA bf16 tensor shaped like the output")
    dy3 = dy.reshape(N, K, D).contiguous()
    if view.packed:
        dpacked = torch.empty((S, N, D), dtype=torch.bfloat16, device=dev)
        drows = [dpacked[s] for s in range(S)]
    else:
        dpacked = None
        drows = [torch.empty((N, D), dtype=torch.bfloat16, device=dev) for _ in range(S)]
    dptrs = (ctypes.c_void_p * S)(*[r.data_ptr() for r in drows])
    db = torch.empty((E, R), dtype=torch.bfloat16, device=dev)
    db32 = torch.empty((E, R), dtype=torch.float32, device=dev)
    need = int(_lib.load().attnres_selected_bwd_workspace_bytes(ctypes.byref(mp), ctypes.c_int32(E)))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    rc = _lib.load().attnres_selected_bwd(
        ctypes.byref(mp), _ptr(bank), ctypes.c_int32(E), _ptr(ids2), _ptr(dy3), _ptr(saved["alpha"]),
        _ptr(saved["rstd"]), _ptr(saved["logit"]), dptrs, ctypes.c_int64(D), _ptr(db), _ptr(db32),
        _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
    _lib.check(rc, "attnres_selected_bwd")
    shape = (*view.lead_shape, D)
    dv = dpacked.view(S, *shape) if dpacked is not None else [r.view(*shape) for r in drows]
    return {"dvalues": dv, "dbank": db, "dbank_f32": db32}


# --------------------------------------------------------------------------
# Autograd operator
# --------------------------------------------------------------------------
def attnres(values: Sources, query: torch.Tensor, *, eps: float = EPS_DEFAULT, scale: float = 1.0,
            out_norm_weight: Optional[torch.Tensor] = None,
            key_offset: Optional[int] = None) -> torch.Tensor:
    """AttnRes read: mix S ordered full-width sources with a softmax over
    scale * <query, RMSNorm(key slice)> and return one [..., D] bf16 residual.

    values: packed [S, ..., D] bf16 or an ordered list/tuple of [..., D]
    tensors (a shared source may appear more than once; its gradients add).
    query: [R], 1 <= R <= D.  key_offset: first key channel (default D - R,
    the final R coordinates).  out_norm_weight: optional [D] weight of an
    output RMSNorm.  Differentiable in values, query and out_norm_weight;
    runs through registered torch operators, so torch.compile(fullgraph=True)
    and CUDA-graph capture work."""
    from .custom_ops import attnres_op
    return attnres_op(values, query, eps=eps, scale=scale, out_norm_weight=out_norm_weight,
                      key_offset=key_offset)


def attnres_multi(values: Sources, queries: torch.Tensor, *, eps: float = EPS_DEFAULT,
                  scale: float = 1.0, key_offset: Optional[int] = None,
                  output_layout: str = "query_major") -> torch.Tensor:
    """Multi-query read: M queries [M, R] (1 <= M <= 16) read the same
    sources, each with its own routing weights and full-width output.
    Returns [M, ..., D] (output_layout="query_major") or [..., M, D]
    ("token_major").  Differentiable in values and queries; registered
    torch operators, so torch.compile(fullgraph=True) and CUDA graphs work."""
    from .custom_ops import attnres_multi_op
    return attnres_multi_op(values, queries, eps=eps, scale=scale, key_offset=key_offset,
                            output_layout=output_layout)


def attnres_selected(values: Sources, query_bank: torch.Tensor, ids: torch.Tensor, *,
                     eps: float = EPS_DEFAULT, scale: float = 1.0,
                     key_offset: Optional[int] = None) -> torch.Tensor:
    """Selected-query read: output [..., K, D], where slot k of token n reads
    the sources with query_bank[ids[n, k]] ([E, R] bank, integer [..., K]
    ids).  Differentiable in values and query_bank; registered torch
    operators, so torch.compile(fullgraph=True) and CUDA graphs work."""
    from .custom_ops import attnres_selected_op
    return attnres_selected_op(values, query_bank, ids, eps=eps, scale=scale, key_offset=key_offset)


def attnres_block_read(completed: Sources, partial: torch.Tensor, delta: torch.Tensor, query: torch.Tensor,
                       *, eps: float = EPS_DEFAULT, scale: float = 1.0,
                       out_norm_weight: Optional[torch.Tensor] = None, key_offset: Optional[int] = None):
    """Block-schedule read with the partial-block sum fused in: returns
    (attnres((*completed, partial + delta), query), partial + delta), the
    sum formed inside the read (one [..., D] pass less than summing first).
    completed: packed [S-1, ..., D] or a list of [..., D] completed block
    sums (the embedding first); partial: the current partial sum; delta:
    the newest writer output.  Differentiable in every tensor argument."""
    from .custom_ops import attnres_block_read_op
    return attnres_block_read_op(completed, partial, delta, query, eps=eps, scale=scale,
                                 out_norm_weight=out_norm_weight, key_offset=key_offset)
