"""The operator's two scalar arguments on the GPU: `scale` and `eps`.

"Fast Attention Residuals", sections "Quickstart" (attnres(values, query,
*, eps=2**-23, scale=1.0)) and "Equation" (the logit is scale times the dot
of the query with the RMS-normalised key; eps sits inside the key's root,
and here also inside the output norm's root).  `scale` enters the forward
logit, the backward's query-side key term, the dq partial sums and the
multi-query coefficients -- separate code paths, so every read is run with
scale != 1 and eps != 2^-23, forward and backward, against the FP64 oracle
called with the same values.  Zero rows make eps decide a key's rstd
(1/sqrt(eps)) outright.
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres, attnres_bwd, attnres_check_device_error, attnres_fwd,
                                       attnres_multi_bwd, attnres_multi_fwd, attnres_partial_bwd,
                                       attnres_partial_fwd, attnres_plan_info, attnres_selected_bwd,
                                       attnres_selected_fwd)
from attention_residuals_gb300.workloads import make_multi, make_random, make_selected
from op_grads import read_grads
from oracle import attnres_oracle
from oracle.multi import attnres_multi_oracle, attnres_selected_oracle
from oracle.partial import attnres_partial_oracle, partial_sum_bits
from parity_utils import (ALPHA_ABS, STAT_REL, Y_REL, check_backward, check_dvalues, check_forward,
                          check_vec_grad, to_np, y_rel_err)

pytestmark = pytest.mark.gpu

SCALE_EPS = [(0.7, 1e-5), (2.5, 1e-2)]


def _zero_rows(wl, frac=0.03, seed=0):
    """Zero a few (source, token) rows so eps alone sets their key's rstd."""
    g = torch.Generator().manual_seed(seed)
    mask = torch.rand((wl.S, wl.N), generator=g) < frac
    wl.values[mask] = 0
    return wl


SINGLE = [
    # S, N, D, R, ko, out_norm, split_n_threshold, save_o_pre
    (6, 211, 2048, 2048, 0, True, 10 ** 9, None),  # resident rows, o rebuilt, in-kernel reduction
    (6, 211, 2048, 2048, 0, True, 1, None),        # same shape, finalize kernel
    (6, 173, 2048, 512, 1536, False, 0, None),     # sliced key in the final R channels
    (9, 97, 8192, 8192, 0, True, 0, False),        # streamed rows (three passes: o, dot, write)
    (9, 97, 8192, 2048, 6144, True, 1, True),      # streamed rows, caller's FP32 o
    (40, 60, 1024, 256, 768, False, 0, None),      # more sources than a warp has lanes
    (5, 301, 4096, 1024, 0, False, 1, None),       # the sliced block shape, first R channels
]


@pytest.mark.parametrize("scale,eps", SCALE_EPS)
@pytest.mark.parametrize("S,N,D,R,ko,out_norm,thr,save", SINGLE)
def test_single_read(S, N, D, R, ko, out_norm, thr, save, scale, eps):
    wl = _zero_rows(make_random(S, N, D, R, key_offset=ko, out_norm=out_norm, seed=S + R + int(10 * scale),
                                scale=scale, eps=eps), seed=S)
    v, q, dy = wl.values.cuda(), wl.q.cuda(), wl.dy.cuda()
    w = wl.w_o.cuda() if out_norm else None
    fwd = attnres_fwd(v, q, w_o=w, key_offset=ko, eps=eps, scale=scale, save_o_pre=save)
    bwd = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=ko, eps=eps, scale=scale, split_n_threshold=thr)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=ko, eps=eps, scale=scale)
    tag = f"S{S} D{D} R{R} ko{ko} scale={scale} eps={eps}"
    errs = check_forward(fwd, ref, out_norm=out_norm, tag=tag)
    errs.update(check_backward(bwd, ref, out_norm=out_norm, tag=tag))
    print(tag, attnres_plan_info(v, R, key_offset=ko, out_norm=out_norm), errs)


@pytest.mark.parametrize("scale,eps", SCALE_EPS)
def test_single_read_autograd_compiled(scale, eps):
    torch._dynamo.reset()
    wl = make_random(5, 96, 1024, 256, key_offset=768, out_norm=True, seed=3, scale=scale, eps=eps)
    v = wl.values.cuda().requires_grad_(True)
    q = wl.q.cuda().requires_grad_(True)
    w = wl.w_o.cuda().requires_grad_(True)
    dy = wl.dy.cuda()
    f = torch.compile(lambda vv, qq, ww: attnres(vv, qq, out_norm_weight=ww, eps=eps, scale=scale),
                      fullgraph=True, dynamic=False)
    y = f(v, q, w)
    y.backward(dy)
    torch.cuda.synchronize()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=768, eps=eps, scale=scale)
    assert y_rel_err(to_np(y), ref["y"]) <= Y_REL
    check_dvalues(to_np(v.grad), ref["dvalues"], {}, "compiled")
    g = read_grads(v, q, dy, w_o=w, eps=eps, scale=scale)
    assert torch.equal(q.grad, g["dq"]) and torch.equal(w.grad, g["dw_o"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "compiled", "dq")
    check_vec_grad(g["dw_o"], g["dw_o_f32"], ref["dw_o"], {}, "compiled", "dw_o")


def _check_multi_like(y, alpha, rstd, logit, ref, K):
    errs = {"y": max(y_rel_err(y[k], ref["y"][k]) for k in range(K)),
            "alpha": float(np.max(np.abs(to_np(alpha) - ref["alpha"]))),
            "rstd": float(np.max(np.abs(to_np(rstd) / ref["rstd"] - 1))),
            "logit": float(np.max(np.abs(to_np(logit) - ref["logit"]) / np.maximum(1, np.abs(ref["logit"]))))}
    assert errs["y"] <= Y_REL and errs["alpha"] <= ALPHA_ABS, errs
    assert errs["rstd"] <= STAT_REL and errs["logit"] <= STAT_REL, errs
    return errs


MULTI = [
    # S, N, D, R, M: one register block, several, and an unaligned key slice
    (5, 90, 2048, 512, 2),
    (4, 64, 1024, 1024, 5),
    (7, 61, 256, 100, 3),
]


@pytest.mark.parametrize("scale,eps", SCALE_EPS)
@pytest.mark.parametrize("S,N,D,R,M", MULTI)
def test_multi_read(S, N, D, R, M, scale, eps):
    wl = make_multi(S, N, D, R, M, seed=S * M, scale=scale, eps=eps)
    g = torch.Generator().manual_seed(M)
    wl.values[torch.rand((S, N), generator=g) < 0.03] = 0
    v, Q, dy = wl.values.cuda(), wl.queries.cuda(), wl.dy.cuda()
    fwd = attnres_multi_fwd(v, Q, key_offset=wl.key_offset, eps=eps, scale=scale)
    bwd = attnres_multi_bwd(v, Q, dy, fwd, key_offset=wl.key_offset, eps=eps, scale=scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_multi_oracle(wl.values, wl.queries, dy=wl.dy, key_offset=wl.key_offset, eps=eps, scale=scale)
    errs = _check_multi_like(to_np(fwd["y"]).reshape(M, N, D), fwd["alpha"], fwd["rstd"], fwd["logit"], ref, M)
    check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, "multi")
    check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, "multi", "dq")


@pytest.mark.parametrize("scale,eps", SCALE_EPS)
@pytest.mark.parametrize("S,N,D,R,E,K", [(5, 80, 2048, 512, 6, 2), (4, 50, 1024, 1024, 3, 5)])
def test_selected_read(S, N, D, R, E, K, scale, eps):
    wl = make_selected(S, N, D, R, E, K, seed=E * K, scale=scale, eps=eps)
    v, bank, ids, dy = wl.values.cuda(), wl.bank.cuda(), wl.ids.cuda(), wl.dy.cuda()
    fwd = attnres_selected_fwd(v, bank, ids, key_offset=wl.key_offset, eps=eps, scale=scale)
    bwd = attnres_selected_bwd(v, bank, ids, dy, fwd, key_offset=wl.key_offset, eps=eps, scale=scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=wl.key_offset,
                                  eps=eps, scale=scale)
    y = np.transpose(to_np(fwd["y"]).reshape(N, K, D), (1, 0, 2))
    refy = dict(ref)
    refy["y"] = np.transpose(ref["y"], (1, 0, 2))
    errs = _check_multi_like(y, fwd["alpha"], fwd["rstd"], fwd["logit"], refy, K)
    check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, "selected")
    check_vec_grad(bwd["dbank"], bwd["dbank_f32"], ref["dbank"], errs, "selected", "dbank")


@pytest.mark.parametrize("scale,eps", SCALE_EPS)
@pytest.mark.parametrize("S,N,D,R,ko,out_norm", [(9, 163, 4096, 1024, 3072, False), (5, 121, 2048, 2048, 0, True)])
def test_block_read(S, N, D, R, ko, out_norm, scale, eps):
    wl = make_random(S + 1, N, D, R, key_offset=ko, out_norm=out_norm, seed=S + N, scale=scale, eps=eps)
    completed, partial, delta = wl.values[:S - 1], wl.values[S - 1], wl.values[S]
    gp = torch.randn(N, D, generator=torch.Generator().manual_seed(N)).to(torch.bfloat16)
    q = wl.q.cuda()
    w = wl.w_o.cuda() if out_norm else None
    comp = [c.cuda() for c in completed]
    fwd = attnres_partial_fwd(comp, partial.cuda(), delta.cuda(), q, w_o=w, key_offset=ko, eps=eps, scale=scale)
    bwd = attnres_partial_bwd(comp, fwd["partial_new"], q, wl.dy.cuda(), fwd, g_partial=gp.cuda(), w_o=w,
                              key_offset=ko, eps=eps, scale=scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_partial_oracle(completed, partial, delta, wl.q, w_o=wl.w_o, dy=wl.dy, g_partial=gp,
                                 key_offset=ko, eps=eps, scale=scale)
    pn = fwd["partial_new"].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(pn, partial_sum_bits(partial, delta))
    errs = {"y": y_rel_err(to_np(fwd["y"]), ref["y"]),
            "alpha": float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"])))}
    assert errs["y"] <= Y_REL and errs["alpha"] <= ALPHA_ABS, errs
    check_dvalues(to_np(torch.stack(bwd["d_completed"])), ref["d_completed"], errs, "block", "d_completed")
    check_dvalues(to_np(bwd["d_partial"]), ref["d_partial"], errs, "block", "d_partial")
    check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, "block", "dq")
    if out_norm:
        check_vec_grad(bwd["dw_o"], bwd["dw_o_f32"], ref["dw_o"], errs, "block", "dw_o")
