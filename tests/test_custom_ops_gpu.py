"""The registered operators: torch.compile(fullgraph=True) and CUDA-graph
capture through `attnres()` ("Fast Attention Residuals", Quickstart and
Validation scope: compiled reads, CUDA Graph replay, packed and list
sources, shared sources), checked against the FP64 oracle."""
import pytest
import torch

from attention_residuals_gb300 import attnres
from attention_residuals_gb300.workloads import make_random
from op_grads import read_grads
from oracle import attnres_oracle
from parity_utils import check_dvalues, check_vec_grad, to_np, y_rel_err

# Autograd hands back the bf16 gradients of q / w_o.  They must equal, bit for
# bit, the operator's bf16 results, whose FP32 sums are held to the gradient
# tolerance and whose bf16 copies must be those sums' RNE roundings
# (parity_utils.check_vec_grad).

pytestmark = pytest.mark.gpu


def _inputs(out_norm, seed, S=6, N=96, D=1024, R=None, ko=None):
    wl = make_random(S, N, D, R, key_offset=0 if ko is None else ko, out_norm=out_norm, seed=seed)
    return wl


@pytest.mark.parametrize("packed", [True, False])
@pytest.mark.parametrize("out_norm", [False, True])
def test_compile_fullgraph_matches_oracle(packed, out_norm):
    torch._dynamo.reset()
    wl = _inputs(out_norm, seed=21 + packed + 2 * out_norm, R=256, ko=768)
    v = wl.values.cuda().requires_grad_(True)
    q = wl.q.cuda().requires_grad_(True)
    w = wl.w_o.cuda().requires_grad_(True) if out_norm else None
    dy = wl.dy.cuda()

    def read(vals, qq, ww):
        return attnres(vals, qq, out_norm_weight=ww, key_offset=768)

    f = torch.compile(read, fullgraph=True, dynamic=False)
    vals = v if packed else list(v.unbind(0))
    y = f(vals, q, w)
    y.backward(dy)
    torch.cuda.synchronize()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=768)
    assert y_rel_err(to_np(y), ref["y"]) <= 1e-2
    check_dvalues(to_np(v.grad), ref["dvalues"], {}, "compiled")
    g = read_grads(vals, q, dy, w_o=w, key_offset=768)
    assert torch.equal(q.grad, g["dq"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "compiled", "dq")
    if out_norm:
        assert torch.equal(w.grad, g["dw_o"])
        check_vec_grad(g["dw_o"], g["dw_o_f32"], ref["dw_o"], {}, "compiled", "dw_o")


def test_cuda_graph_replay_forward_and_backward():
    wl = _inputs(True, seed=31)
    v = wl.values.cuda().requires_grad_(True)
    q = wl.q.cuda().requires_grad_(True)
    w = wl.w_o.cuda().requires_grad_(True)

    def read(vv, qq, ww):
        return attnres(vv, qq, out_norm_weight=ww, key_offset=0)

    graphed = torch.cuda.make_graphed_callables(read, (v, q, w))
    # replay on new inputs (copied into the graph's static buffers)
    wl2 = _inputs(True, seed=32)
    v2 = wl2.values.cuda().requires_grad_(True)
    y = graphed(v2, q, w)
    y.backward(wl2.dy.cuda())
    torch.cuda.synchronize()
    ref = attnres_oracle(wl2.values, wl.q, w_o=wl.w_o, dy=wl2.dy, key_offset=0)
    assert y_rel_err(to_np(y), ref["y"]) <= 1e-2
    check_dvalues(to_np(v2.grad), ref["dvalues"], {}, "graph")
    g = read_grads(v2, q, wl2.dy.cuda(), w_o=w, key_offset=0)
    assert torch.equal(q.grad, g["dq"]) and torch.equal(w.grad, g["dw_o"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "graph", "dq")
    check_vec_grad(g["dw_o"], g["dw_o_f32"], ref["dw_o"], {}, "graph", "dw_o")


def test_shared_source_gradients_add_through_the_op():
    wl = _inputs(False, seed=41, S=4)
    x = [wl.values[i].cuda().requires_grad_(True) for i in range(3)]
    q = wl.q.cuda().requires_grad_(True)
    y = attnres([x[0], x[1], x[0], x[2]], q, key_offset=0)
    y.backward(wl.dy.cuda())
    vref = torch.stack([wl.values[i] for i in (0, 1, 0, 2)])
    ref = attnres_oracle(vref, wl.q, dy=wl.dy, key_offset=0)
    check_dvalues(to_np(x[0].grad), ref["dvalues"][0] + ref["dvalues"][2], {}, "shared x0")
    check_dvalues(to_np(x[2].grad), ref["dvalues"][3], {}, "x2")


def test_leading_dims_and_default_key_offset():
    wl = _inputs(False, seed=51, S=3, N=2 * 40, D=512, R=128)
    v = wl.values.cuda().view(3, 2, 40, 512)
    q = wl.q.cuda()
    y = attnres(v, q)  # key in the final R channels
    assert y.shape == (2, 40, 512)
    ref = attnres_oracle(wl.values, wl.q, key_offset=512 - 128)
    assert y_rel_err(to_np(y.reshape(80, 512)), ref["y"]) <= 1e-2


@pytest.mark.parametrize("compiled", [False, True])
def test_one_source_list_reads_itself(compiled):
    # A list holding one [T, D] source is S = 1 (the read returns the source,
    # dq = 0), not a packed [S, D] tensor of T sources and one token.
    torch._dynamo.reset()
    wl = _inputs(False, seed=61, S=1, N=300, D=512, R=128)
    x = wl.values[0].cuda().requires_grad_(True)
    q = wl.q.cuda().requires_grad_(True)

    def read(xx, qq):
        return attnres([xx], qq)

    f = torch.compile(read, fullgraph=True, dynamic=False) if compiled else read
    y = f(x, q)
    assert y.shape == x.shape
    assert torch.equal(y, x.detach())
    y.backward(wl.dy.cuda())
    torch.cuda.synchronize()
    assert torch.equal(x.grad, wl.dy.cuda())   # dv = alpha * do with alpha = 1
    assert torch.count_nonzero(q.grad).item() == 0
