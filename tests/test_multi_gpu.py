"""GPU parity of the multi-query read ("Fast Attention Residuals", section
"Multi-query AttnRes") through the C ABI, against the FP64 oracle.

Shapes span every kernel variant (1, 2 or 4 vectors per thread; one or
several register blocks of queries), ragged token counts, unaligned key
slices, both output layouts, M from 1 to 16, more sources than a warp has
lanes and the empty input.  The long
workload at full size is checked on sampled tokens plus the full dq.
Tolerances as for the single-query read (parity_utils).
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres_check_device_error, attnres_multi, attnres_multi_bwd,
                                       attnres_multi_fwd, attnres_multi_plan_info)
from attention_residuals_gb300._lib import AttnresError
from attention_residuals_gb300.workloads import make_multi, make_multi_workload
from oracle.multi import attnres_multi_oracle
from op_grads import multi_grads
from parity_utils import (ALPHA_ABS, GRAD_REL_L2, STAT_REL, Y_REL, bf16_rne, check_dvalues, check_vec_grad,
                          rel_l2, to_np,
                          y_rel_err)

pytestmark = pytest.mark.gpu


def _check(wl, fwd, bwd, ref, token_major, tag):
    M, N, D, S = wl.M, wl.N, wl.D, wl.S
    y = to_np(fwd["y"]).reshape((N, M, D) if token_major else (M, N, D))
    if token_major:
        y = np.transpose(y, (1, 0, 2))
    errs = {"y": max(y_rel_err(y[m], ref["y"][m]) for m in range(M)) if N else 0.0}
    if N:
        errs["alpha"] = float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"])))
        errs["rstd"] = float(np.max(np.abs(to_np(fwd["rstd"]) / ref["rstd"] - 1)))
        z = ref["logit"]
        errs["logit"] = float(np.max(np.abs(to_np(fwd["logit"]) - z) / np.maximum(1, np.abs(z))))
        assert errs["alpha"] <= ALPHA_ABS, (tag, errs)
        assert errs["rstd"] <= STAT_REL, (tag, errs)
        assert errs["logit"] <= STAT_REL, (tag, errs)
    assert errs["y"] <= Y_REL, (tag, errs)
    if bwd is not None:
        check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, tag)
        check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, tag, "dq")
    return errs


def run_multi(wl, *, token_major=False, list_sources=False):
    v = wl.values.cuda()
    Q = wl.queries.cuda()
    dy = wl.dy.cuda()
    if token_major:
        dy = dy.transpose(0, 1).contiguous()
    vals = list(v.unbind(0)) if list_sources else v
    fwd = attnres_multi_fwd(vals, Q, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale,
                            token_major=token_major)
    bwd = attnres_multi_bwd(vals, Q, dy, fwd, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_multi_oracle(wl.values, wl.queries, dy=wl.dy, key_offset=wl.key_offset,
                               eps=wl.eps, scale=wl.scale)
    return fwd, bwd, ref


SHAPES = [
    # S, N, D, R, ko, M
    (8, 2, 1024, 64, 960, 2),        # the page's example
    (5, 37, 512, 128, 384, 2),
    (6, 129, 2048, 2048, 0, 3),      # R == D, padded query block
    (4, 200, 4096, 1024, 3072, 4),   # two vectors per thread, two backward blocks
    (3, 64, 1024, 1024, 0, 16),      # M = 16, four register blocks
    (10, 97, 4096, 1024, 3072, 2),   # the long workload's shape, short N
    (2, 50, 8192, 512, 0, 2),        # four vectors per thread
    (7, 61, 256, 100, 13, 5),        # unaligned key slice
    (3, 45, 24, 24, 0, 5),           # tiny rows, partial warp
    (33, 41, 512, 256, 256, 3),      # more sources than lanes
    (1, 30, 1024, 512, 512, 4),      # one source
    (12, 161, 2048, 512, 1536, 8),   # M = 8
    (16, 23, 4096, 1024, 3072, 3),   # forward: several softmax groups and two passes per token
    (9, 77, 2048, 512, 1536, 1),     # one query (the fixed-count kernels for M = 1)
    (5, 90, 1024, 256, 768, 4),      # M = 4 at one vector per thread: four per forward block
]


@pytest.mark.parametrize("form", [None, "resident"])
@pytest.mark.parametrize("S,N,D,R,ko,M", SHAPES)
def test_multi_matches_oracle(S, N, D, R, ko, M, form, monkeypatch):
    # default plan, and the resident backward forced wherever a token fits
    # (by default it serves at most two queries)
    if form is not None:
        monkeypatch.setenv("ATTNRES_MULTI_BWD", form)
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=S * 31 + M, src_scale=(0.5, 2.0))
    fwd, bwd, ref = run_multi(wl)
    errs = _check(wl, fwd, bwd, ref, False, f"S{S} N{N} D{D} R{R} ko{ko} M{M}")
    print(attnres_multi_plan_info(wl.values.cuda(), M, R, key_offset=ko), errs)


@pytest.mark.parametrize("list_sources", [False, True])
def test_multi_token_major_and_list_sources(list_sources):
    wl = make_multi(6, 77, 2048, 512, 3, seed=5)
    fwd, bwd, ref = run_multi(wl, token_major=True, list_sources=list_sources)
    assert fwd["y"].shape == (77, 3, 2048)
    _check(wl, fwd, bwd, ref, True, "token-major")
    if list_sources:
        assert isinstance(bwd["dvalues"], list) and len(bwd["dvalues"]) == 6


def test_multi_one_source_reads_itself_and_dq_is_zero():
    wl = make_multi(1, 40, 1024, 256, 3, seed=9)
    fwd, bwd, ref = run_multi(wl)
    for m in range(3):
        assert torch.equal(fwd["y"][m].cpu(), wl.values[0])
    assert torch.count_nonzero(bwd["dq_f32"]).item() == 0


def test_multi_deterministic():
    wl = make_multi(9, 600, 4096, 1024, 2, seed=13)
    v, Q, dy = wl.values.cuda(), wl.queries.cuda(), wl.dy.cuda()
    f = attnres_multi_fwd(v, Q)
    a = attnres_multi_bwd(v, Q, dy, f)
    b = attnres_multi_bwd(v, Q, dy, f)
    torch.cuda.synchronize()
    assert torch.equal(a["dq_f32"], b["dq_f32"])
    assert torch.equal(a["dvalues"], b["dvalues"])
    wl2 = make_multi(4, 300, 1024, 1024, 12, key_offset=0, seed=14)
    v, Q, dy = wl2.values.cuda(), wl2.queries.cuda(), wl2.dy.cuda()
    f = attnres_multi_fwd(v, Q, key_offset=0)
    a = attnres_multi_bwd(v, Q, dy, f, key_offset=0)
    b = attnres_multi_bwd(v, Q, dy, f, key_offset=0)
    torch.cuda.synchronize()
    assert torch.equal(a["dq_f32"], b["dq_f32"])
    assert torch.equal(a["dvalues"], b["dvalues"])


def test_multi_empty_input():
    v = torch.zeros((3, 0, 512), dtype=torch.bfloat16, device="cuda")
    Q = torch.ones((2, 128), dtype=torch.bfloat16, device="cuda")
    f = attnres_multi_fwd(v, Q)
    assert f["y"].shape == (2, 0, 512)
    g = attnres_multi_bwd(v, Q, torch.zeros((2, 0, 512), dtype=torch.bfloat16, device="cuda"), f)
    torch.cuda.synchronize()
    assert torch.count_nonzero(g["dq_f32"]).item() == 0 and g["dq"].shape == (2, 128)


def test_multi_large_tokens_forward_and_backward():
    # 64 rows of 16 KB and sixteen queries cannot stay resident in shared
    # memory: the forward streams the rows (one pass per query block), the
    # backward takes the general two-kernel path
    wl = make_multi(64, 5, 8192, 8192, 16, key_offset=0, seed=77)
    v, Q = wl.values.cuda(), wl.queries.cuda()
    assert attnres_multi_plan_info(v, 16, 8192, key_offset=0)["bwd_general"] >= 1
    fwd, bwd, ref = run_multi(wl)
    _check(wl, fwd, bwd, ref, False, "S64 D8192 M16")


def test_multi_autograd_compile_and_shared_sources():
    torch._dynamo.reset()
    wl = make_multi(4, 90, 1024, 256, 2, seed=21)
    x = [wl.values[i].cuda().requires_grad_(True) for i in range(3)]
    Q = wl.queries.cuda().requires_grad_(True)
    f = torch.compile(lambda vals, qq: attnres_multi(vals, qq), fullgraph=True, dynamic=False)
    y = f([x[0], x[1], x[0], x[2]], Q)
    y.backward(wl.dy.cuda())
    torch.cuda.synchronize()
    vref = torch.stack([wl.values[i] for i in (0, 1, 0, 2)])
    ref = attnres_multi_oracle(vref, wl.queries, dy=wl.dy, key_offset=1024 - 256)
    assert max(y_rel_err(to_np(y[m]), ref["y"][m]) for m in range(2)) <= Y_REL
    check_dvalues(to_np(x[0].grad), ref["dvalues"][0] + ref["dvalues"][2], {}, "shared x0")
    check_dvalues(to_np(x[2].grad), ref["dvalues"][3], {}, "x2")
    # autograd's bf16 dq is the operator's, bit for bit; its FP32 sum is held to
    # the tolerance and the bf16 copy must be that sum's RNE rounding
    g = multi_grads([x[0], x[1], x[0], x[2]], Q, wl.dy.cuda())
    assert torch.equal(Q.grad, g["dq"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "autograd", "dq")
    yt = attnres_multi(torch.stack([t.detach() for t in x]), Q.detach(), output_layout="token_major")
    assert yt.shape == (90, 2, 1024)


@pytest.mark.parametrize("key", ["long", "sixteen"])
def test_multi_full_size_sampled(key):
    # the bench's multi-query workloads at full size, in its launch
    # configuration: two quarter-rank queries (resident backward) and sixteen
    # full-rank queries (tensor-core forward, general backward with the
    # tensor-core gradient kernel)
    wl = make_multi_workload(key, device="cuda")
    v, Q, dy = wl.values, wl.queries, wl.dy
    info = attnres_multi_plan_info(v, wl.M, wl.R, key_offset=wl.key_offset)
    assert info["bwd_general"] == (2 if key == "sixteen" else 0), info
    assert info["fwd_tensor_cores"] == (1 if key == "sixteen" else 0), info
    fwd = attnres_multi_fwd(v, Q)
    bwd = attnres_multi_bwd(v, Q, dy, fwd)
    bwd2 = attnres_multi_bwd(v, Q, dy, fwd)
    torch.cuda.synchronize()
    attnres_check_device_error()
    assert torch.equal(bwd["dq_f32"], bwd2["dq_f32"]) and torch.equal(bwd["dvalues"], bwd2["dvalues"])
    del bwd2
    g = np.random.default_rng(1)
    idx = np.array(sorted(set(g.choice(wl.N, 40, replace=False).tolist()) | {0, wl.N - 1}))
    it = torch.as_tensor(idx, device="cuda")
    ref = attnres_multi_oracle(v.index_select(1, it).cpu(), Q.cpu(), dy=dy.index_select(1, it).cpu(),
                               key_offset=wl.key_offset)
    y = to_np(fwd["y"].index_select(1, it))
    assert max(y_rel_err(y[m], ref["y"][m]) for m in range(wl.M)) <= Y_REL
    assert float(np.max(np.abs(to_np(fwd["alpha"].index_select(0, it)) - ref["alpha"]))) <= ALPHA_ABS
    check_dvalues(to_np(bwd["dvalues"].index_select(1, it)), ref["dvalues"], {}, "full")
    full = attnres_multi_oracle(v.cpu(), Q.cpu(), dy=dy.cpu(), key_offset=wl.key_offset,
                                want_dvalues=False)
    check_vec_grad(bwd["dq"], bwd["dq_f32"], full["dq"], {}, "full", "dq")
