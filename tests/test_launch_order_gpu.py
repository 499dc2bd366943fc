"""The backward and finalize kernels may begin while the kernel before them
on the stream is still running (programmatic dependent launch); they wait for
it before touching global memory.  These tests put ordinary PyTorch kernels
right before them on the same stream -- one writing an input the backward
reads, one reading a buffer the backward then overwrites -- and check that
the results equal a fully synchronised run's bitwise."""
import pytest
import torch

from attention_residuals_gb300 import (attnres_bwd, attnres_check_device_error, attnres_fwd, attnres_multi_bwd,
                                       attnres_multi_fwd)
from attention_residuals_gb300.workloads import make_multi, make_random

pytestmark = pytest.mark.gpu


def _slow_dy(base):
    # several full passes over a large buffer, the last one writing dy
    t = base.float()
    for _ in range(4):
        t = t * 1.0001 + 0.0
    return (t * 0.5).to(torch.bfloat16)


@pytest.mark.parametrize("S,N,D,R,norm,cl", [(10, 4096, 4096, 4096, True, None), (8, 8192, 2048, 2048, False, None),
                                             (64, 300, 8192, 8192, True, None)])
def test_backward_waits_for_the_kernel_before_it(S, N, D, R, norm, cl):
    wl = make_random(S, N, D, R, out_norm=norm, seed=S + N)
    v, q = wl.values.cuda(), wl.q.cuda()
    w = wl.w_o.cuda() if norm else None
    base = (wl.dy.float() * 2.0).to(torch.bfloat16).cuda()
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0)
    torch.cuda.synchronize()
    dy_ref = _slow_dy(base)
    torch.cuda.synchronize()
    ref = attnres_bwd(v, q, dy_ref, fwd, w_o=w, key_offset=0)
    torch.cuda.synchronize()

    dv = torch.full_like(v, 3.0)
    for _ in range(3):
        dv.fill_(3.0)
        torch.cuda.synchronize()
        snap = dv.clone()                      # a kernel reading dv right before the backward writes it
        dy = _slow_dy(base)                    # kernels writing dy right before the backward reads it
        out = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0, dvalues=dv)
        torch.cuda.synchronize()
        assert bool((snap == 3.0).all()), "the backward wrote dvalues before the kernel reading them finished"
        for key in ("dq", "dq_f32") + (("dw_o", "dw_o_f32") if norm else ()):
            assert torch.equal(out[key], ref[key]), key
        assert torch.equal(dv, ref["dvalues"])
    attnres_check_device_error()


def test_multi_backward_waits_for_the_kernel_before_it():
    wl = make_multi(10, 4096, 4096, 1024, 2, seed=7)
    v, Q = wl.values.cuda(), wl.queries.cuda()
    base = wl.dy.cuda()
    fwd = attnres_multi_fwd(v, Q)
    torch.cuda.synchronize()
    dy_ref = _slow_dy(base)
    torch.cuda.synchronize()
    ref = attnres_multi_bwd(v, Q, dy_ref, fwd)
    torch.cuda.synchronize()
    for _ in range(3):
        dy = _slow_dy(base)
        out = attnres_multi_bwd(v, Q, dy, fwd)
        torch.cuda.synchronize()
        for key in ("dvalues", "dq", "dq_f32"):
            assert torch.equal(out[key], ref[key]), key
    attnres_check_device_error()
