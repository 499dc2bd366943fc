"""The registered operators' backward, called directly, for the autograd tests.

Autograd hands back only the bf16 roundings of the reduced gradients (dq,
dw_o, the bank gradient).  These helpers run the same operator pair that
autograd runs -- forward, then backward on the same saved statistics -- and
return the bf16 gradients with their FP32 sums, so a test can require
  * autograd's gradient == this bf16 gradient, bit for bit (the kernels and
    their reduction orders are deterministic), and
  * the FP32 sum within the tolerance and the bf16 copy its exact
    round-to-nearest-even (parity_utils.check_vec_grad).
"""
import torch

from attention_residuals_gb300 import custom_ops

_ops = torch.ops.attnres_gb300


def read_grads(values, q, dy, *, w_o=None, eps=2.0 ** -23, scale=1.0, key_offset=None):
    vals, packed = custom_ops._pack_args(values)
    vals = [v.detach() for v in vals]
    q, w = q.detach(), None if w_o is None else w_o.detach()
    ko = vals[0].shape[-1] - q.numel() if key_offset is None else int(key_offset)
    y, alpha, rstd, logit, o_rstd, o_pre = _ops.read_fwd(vals, q, w, float(eps), float(scale), ko, packed)
    dv, dq, dw, dq32, dw32 = _ops.read_bwd(vals, q, w, dy.to(torch.bfloat16).contiguous(), alpha, rstd,
                                           logit, o_rstd, o_pre, float(eps), float(scale), ko, packed)
    return {"dq": dq, "dq_f32": dq32, "dw_o": dw if w is not None else None,
            "dw_o_f32": dw32 if w is not None else None}


def multi_grads(values, queries, dy, *, eps=2.0 ** -23, scale=1.0, key_offset=None, token_major=False):
    vals, packed = custom_ops._pack_args(values)
    vals = [v.detach() for v in vals]
    Q = queries.detach()
    ko = vals[0].shape[-1] - Q.shape[-1] if key_offset is None else int(key_offset)
    y, alpha, rstd, logit = _ops.read_multi_fwd(vals, Q, float(eps), float(scale), ko, token_major, packed)
    dv, dq, dq32 = _ops.read_multi_bwd(vals, Q, dy.to(torch.bfloat16).contiguous(), alpha, rstd, logit,
                                       float(eps), float(scale), ko, token_major, packed)
    return {"dq": dq, "dq_f32": dq32}


def selected_grads(values, bank, ids, dy, *, eps=2.0 ** -23, scale=1.0, key_offset=None):
    vals, packed = custom_ops._pack_args(values)
    vals = [v.detach() for v in vals]
    B = bank.detach()
    ko = vals[0].shape[-1] - B.shape[-1] if key_offset is None else int(key_offset)
    y, alpha, rstd, logit = _ops.read_selected_fwd(vals, B, ids, float(eps), float(scale), ko, packed)
    dv, db, db32 = _ops.read_selected_bwd(vals, B, ids, dy.to(torch.bfloat16).contiguous(), alpha, rstd,
                                          logit, float(eps), float(scale), ko, packed)
    return {"dbank": db, "dbank_f32": db32}


def block_grads(completed, partial, delta, q, dy, g_partial, *, w_o=None, eps=2.0 ** -23, scale=1.0,
                key_offset=None):
    comp = list(completed.unbind(0)) if isinstance(completed, torch.Tensor) else list(completed)
    comp = [c.detach() for c in comp]
    q, w = q.detach(), None if w_o is None else w_o.detach()
    D = partial.shape[-1]
    ko = D - q.numel() if key_offset is None else int(key_offset)
    out = _ops.read_block_fwd(comp + [partial.detach()], delta.detach(), q, w, float(eps), float(scale), ko)
    y, pn, alpha, rstd, logit, o_rstd, o_pre = out
    g = None if g_partial is None else g_partial.to(torch.bfloat16)
    res = _ops.read_block_bwd(comp, pn, q, w, dy.to(torch.bfloat16), g, alpha, rstd, logit, o_rstd, o_pre,
                              float(eps), float(scale), ko)
    dcomp, dpart, dq, dw, dq32, dw32 = res
    return {"dq": dq, "dq_f32": dq32, "dw_o": dw if w is not None else None,
            "dw_o_f32": dw32 if w is not None else None}
