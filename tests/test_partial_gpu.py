"""GPU parity of the fused block-partial read ("Fast Attention Residuals",
section "Full and Block schedules": the caller's partial-block sum formed
inside the read) through the C ABI, against the FP64 oracle.

partial_new = partial + delta is integer-exact work (one bf16 rounding of an
FP32 sum) and is compared bit for bit; the read and its gradients use the
single-query tolerances (parity_utils).  Shapes cover the block workload
(eight completed block sums plus the partial, sliced key), the output norm,
both key placements, one source only (no completed block), the streaming
backward (rows too large to stay resident), in-place updates of the partial
sum, and autograd through torch.compile with the new partial sum used
downstream.
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres_block_read, attnres_check_device_error,
                                       attnres_partial_bwd, attnres_partial_fwd, attnres_plan_info)
from attention_residuals_gb300.workloads import make_random
from oracle.partial import attnres_partial_oracle, partial_sum_bits
from op_grads import block_grads
from parity_utils import (ALPHA_ABS, GRAD_REL_L2, STAT_REL, Y_REL, bf16_rne, check_dvalues, check_vec_grad,
                          rel_l2, to_np, y_rel_err)

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(S, N, D, R, ko, out_norm, seed):
    wl = make_random(S + 1, N, D, R, key_offset=ko, out_norm=out_norm, seed=seed)
    completed, partial, delta = wl.values[:S - 1], wl.values[S - 1], wl.values[S]
    g = torch.Generator().manual_seed(seed + 1)
    gp = torch.randn(N, D, generator=g).to(torch.bfloat16)
    return wl, completed, partial, delta, gp


SHAPES = [
    # S (sources incl. the partial), N, D, R, ko, out_norm
    (9, 263, 4096, 1024, 0, False),     # block workload shape, first R channels
    (9, 263, 4096, 1024, 3072, False),  # final R channels (the page's placement)
    (10, 157, 4096, 4096, 0, True),     # output norm
    (1, 77, 1024, 1024, 0, False),      # the partial sum alone
    (5, 301, 2048, 512, 1536, True),
    (40, 9, 8192, 8192, 0, True),       # streaming backward
]


@pytest.mark.parametrize("S,N,D,R,ko,out_norm", SHAPES)
def test_partial_matches_oracle(S, N, D, R, ko, out_norm):
    wl, completed, partial, delta, gp = _case(S, N, D, R, ko, out_norm, seed=S * 13 + R)
    q = wl.q.cuda()
    w = wl.w_o.cuda() if out_norm else None
    comp_d = [c.cuda() for c in completed]
    fwd = attnres_partial_fwd(comp_d, partial.cuda(), delta.cuda(), q, w_o=w, key_offset=ko)
    bwd = attnres_partial_bwd(comp_d, fwd["partial_new"], q, wl.dy.cuda(), fwd, g_partial=gp.cuda(), w_o=w,
                              key_offset=ko)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_partial_oracle(completed, partial, delta, wl.q, w_o=wl.w_o, dy=wl.dy, g_partial=gp,
                                 key_offset=ko)
    np.testing.assert_array_equal(_bits(fwd["partial_new"]), partial_sum_bits(partial, delta))
    errs = {"y": y_rel_err(to_np(fwd["y"]), ref["y"]),
            "alpha": float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"]))),
            "rstd": float(np.max(np.abs(to_np(fwd["rstd"]) / ref["rstd"] - 1)))}
    assert errs["y"] <= Y_REL and errs["alpha"] <= ALPHA_ABS and errs["rstd"] <= STAT_REL, errs
    if S > 1:
        check_dvalues(to_np(torch.stack(bwd["d_completed"])), ref["d_completed"], errs, "", "d_completed")
    check_dvalues(to_np(bwd["d_partial"]), ref["d_partial"], errs, "", "d_partial")
    check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, "", "dq")
    if out_norm:
        check_vec_grad(bwd["dw_o"], bwd["dw_o_f32"], ref["dw_o"], errs, "", "dw_o")
    print(attnres_plan_info(comp_d + [fwd["partial_new"]], R, key_offset=ko, out_norm=out_norm), errs)


def test_partial_in_place_update_and_no_extra_gradient():
    wl, completed, partial, delta, gp = _case(6, 500, 2048, 2048, 0, False, seed=5)
    q = wl.q.cuda()
    comp_d = [c.cuda() for c in completed]
    out_of_place = attnres_partial_fwd(comp_d, partial.cuda(), delta.cuda(), q, key_offset=0)
    acc = partial.cuda().clone()
    in_place = attnres_partial_fwd(comp_d, acc, delta.cuda(), q, key_offset=0, partial_out=acc)
    torch.cuda.synchronize()
    assert torch.equal(acc, out_of_place["partial_new"])
    assert torch.equal(in_place["y"], out_of_place["y"])
    # without g_partial the last gradient is the read's alone
    b = attnres_partial_bwd(comp_d, acc, q, wl.dy.cuda(), in_place, key_offset=0)
    ref = attnres_partial_oracle(completed, partial, delta, wl.q, dy=wl.dy, key_offset=0)
    assert rel_l2(to_np(b["d_partial"]), ref["d_partial"]) <= GRAD_REL_L2


@pytest.mark.parametrize("out_norm", [False, True])
def test_block_read_autograd_compile(out_norm):
    torch._dynamo.reset()
    wl, completed, partial, delta, gp = _case(5, 96, 1024, 256, 768, out_norm, seed=31 + out_norm)
    comp = completed.cuda().requires_grad_(True)
    part = partial.cuda().requires_grad_(True)
    dl = delta.cuda().requires_grad_(True)
    q = wl.q.cuda().requires_grad_(True)
    w = wl.w_o.cuda().requires_grad_(True) if out_norm else None

    def step(c, p, d, qq, ww):
        y, pn = attnres_block_read(c, p, d, qq, out_norm_weight=ww)
        return y, pn

    f = torch.compile(step, fullgraph=True, dynamic=False)
    y, pn = f(comp, part, dl, q, w)
    torch.autograd.backward([y, pn], [wl.dy.cuda(), gp.cuda()])
    torch.cuda.synchronize()
    ref = attnres_partial_oracle(completed, partial, delta, wl.q, w_o=wl.w_o, dy=wl.dy, g_partial=gp,
                                 key_offset=768)
    np.testing.assert_array_equal(_bits(pn), partial_sum_bits(partial, delta))
    assert y_rel_err(to_np(y), ref["y"]) <= Y_REL
    check_dvalues(to_np(comp.grad), ref["d_completed"], {}, "autograd", "d_completed")
    check_dvalues(to_np(part.grad), ref["d_partial"], {}, "autograd", "d_partial")
    assert torch.equal(part.grad, dl.grad)
    # autograd's bf16 dq (and dw_o) are the operator's, bit for bit; the FP32
    # sums are held to the tolerance, the bf16 copies must be their RNE roundings
    g = block_grads(comp, part, dl, q, wl.dy.cuda(), gp.cuda(), w_o=w, key_offset=768)
    assert torch.equal(q.grad, g["dq"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "autograd", "dq")
    if out_norm:
        assert torch.equal(w.grad, g["dw_o"])
        check_vec_grad(g["dw_o"], g["dw_o_f32"], ref["dw_o"], {}, "autograd", "dw_o")


def test_block_full_size_sampled():
    # the benchmark's block workload at full size (eight completed block sums,
    # the partial sum, N=16384, D=4096, R=1024): sampled tokens element by
    # element, the new partial sum bit for bit everywhere, dq over every token
    from attention_residuals_gb300.workloads import make_workload
    wl = make_workload(4, seed=404, device="cuda")
    comp = list(wl.values[:-1].unbind(0))
    partial = wl.values[-1]
    g = torch.Generator(device="cuda").manual_seed(405)
    delta = torch.randn(partial.shape, generator=g, device="cuda").to(torch.bfloat16)
    gp = torch.randn(partial.shape, generator=g, device="cuda").to(torch.bfloat16)
    f = attnres_partial_fwd(comp, partial, delta, wl.q, key_offset=wl.key_offset)
    b = attnres_partial_bwd(comp, f["partial_new"], wl.q, wl.dy, f, g_partial=gp, key_offset=wl.key_offset)
    torch.cuda.synchronize()
    attnres_check_device_error()
    np.testing.assert_array_equal(_bits(f["partial_new"]), partial_sum_bits(partial.cpu(), delta.cpu()))
    rng = np.random.default_rng(3)
    idx = np.array(sorted(set(rng.choice(wl.N, 40, replace=False).tolist()) | {0, wl.N - 1}))
    it = torch.as_tensor(idx, device="cuda")
    sel = lambda t: t.index_select(-2, it).cpu()
    ref = attnres_partial_oracle(torch.stack([sel(c) for c in comp]), sel(partial), sel(delta), wl.q.cpu(),
                                 dy=sel(wl.dy), g_partial=sel(gp), key_offset=wl.key_offset)
    assert y_rel_err(to_np(f["y"].index_select(0, it)), ref["y"]) <= Y_REL
    check_dvalues(to_np(torch.stack([c.index_select(0, it) for c in b["d_completed"]])), ref["d_completed"], {},
                  "full", "d_completed")
    check_dvalues(to_np(b["d_partial"].index_select(0, it)), ref["d_partial"], {}, "full", "d_partial")
    full = attnres_partial_oracle(torch.stack([c.cpu() for c in comp]), partial.cpu(), delta.cpu(), wl.q.cpu(),
                                  dy=wl.dy.cpu(), g_partial=gp.cpu(), key_offset=wl.key_offset)
    check_vec_grad(b["dq"], b["dq_f32"], full["dq"], {}, "full", "dq")
