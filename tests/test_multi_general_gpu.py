"""GPU parity of the general multi-query / selected-query backward (two
kernels over column blocks: tensor-core coefficients, then dvalues and dq),
against the FP64 oracle.

"Fast Attention Residuals", section "Multi-query AttnRes": queries [M, R]
with 1 <= M <= 16, and attnres_selected with K slots per token.  The
general backward serves every shape -- the ones whose token does not fit in
shared memory (many sources, wide rows, many queries) and, by default, every
read with more than two queries.  ATTNRES_MULTI_BWD=general forces it on
any shape, so it is also checked on the shapes of the resident kernels.
Its gradient kernel runs on the tensor cores for fixed queries and at most
16 sources; ATTNRES_MULTI_GRAD=simt keeps the SIMT kernel, and both are
checked.
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres_check_device_error, attnres_multi_bwd, attnres_multi_fwd,
                                       attnres_multi_plan_info, attnres_selected_bwd, attnres_selected_fwd)
from attention_residuals_gb300._lib import AttnresError
from attention_residuals_gb300.workloads import make_multi, make_selected
from oracle.multi import attnres_multi_oracle, attnres_selected_oracle
from parity_utils import (ALPHA_ABS, STAT_REL, Y_REL, check_dvalues, check_vec_grad, to_np, y_rel_err)
from test_multi_gpu import SHAPES as MULTI_SHAPES
from test_selected_gpu import SHAPES as SELECTED_SHAPES

pytestmark = pytest.mark.gpu


def _check_multi(wl, fwd, bwd, ref, tag):
    M, N, D, S = wl.M, wl.N, wl.D, wl.S
    y = to_np(fwd["y"]).reshape(M, N, D)
    errs = {"y": max(y_rel_err(y[m], ref["y"][m]) for m in range(M))}
    errs["alpha"] = float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"])))
    assert errs["y"] <= Y_REL and errs["alpha"] <= ALPHA_ABS, (tag, errs)
    check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, tag)
    check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, tag, "dq")
    return errs


def _run_multi(wl, twice=False):
    v, Q, dy = wl.values.cuda(), wl.queries.cuda(), wl.dy.cuda()
    fwd = attnres_multi_fwd(v, Q, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    bwd = attnres_multi_bwd(v, Q, dy, fwd, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    if twice:
        bwd2 = attnres_multi_bwd(v, Q, dy, fwd, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
        torch.cuda.synchronize()
        for key in ("dvalues", "dq_f32", "dq"):
            assert torch.equal(bwd[key], bwd2[key]), key
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_multi_oracle(wl.values, wl.queries, dy=wl.dy, key_offset=wl.key_offset, eps=wl.eps,
                               scale=wl.scale)
    return fwd, bwd, ref


def _grad_form(monkeypatch, form, S):
    """Force the gradient kernel; the plan's backward form it should give
    (2: tensor-core gradients, for at most 16 sources; 1: SIMT)."""
    monkeypatch.setenv("ATTNRES_MULTI_GRAD", form)
    return 2 if form == "mma" and S <= 16 else 1


@pytest.mark.parametrize("form", ["mma", "simt"])
@pytest.mark.parametrize("S,N,D,R,ko,M", MULTI_SHAPES)
def test_general_on_every_multi_shape(S, N, D, R, ko, M, form, monkeypatch):
    monkeypatch.setenv("ATTNRES_MULTI_BWD", "general")
    want = _grad_form(monkeypatch, form, S)
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=S * 37 + M, src_scale=(0.5, 2.0))
    info = attnres_multi_plan_info(wl.values.cuda(), M, R, key_offset=ko)
    assert info["bwd_general"] == want, info
    fwd, bwd, ref = _run_multi(wl)
    errs = _check_multi(wl, fwd, bwd, ref, f"S{S} N{N} D{D} R{R} ko{ko} M{M} {form}")
    print(info, errs)


WIDE = [
    # S, N, D, R, ko, M: shapes whose token does not fit the resident kernel
    (10, 61, 4096, 1024, 3072, 16),     # sixteen queries over the long workload's rows
    (10, 47, 4096, 4096, 0, 16),
    (10, 50, 8192, 8192, 0, 4),         # four queries over 16 KB rows
    (10, 33, 8192, 2048, 6144, 9),
    (64, 6, 8192, 8192, 0, 16),         # the widest token: 64 x 16 KB rows, sixteen queries
    (128, 4, 2048, 512, 1536, 7),       # the most sources
    (3, 90, 1000, 333, 13, 11),         # width 8 mod 16 (the last MMA step reads zeros), unaligned key
    (5, 70, 24, 24, 0, 16),             # tiny rows
    (1, 40, 4096, 1024, 0, 16),         # one source: dq is zero, dvalues = sum of dy
]


@pytest.mark.parametrize("form", ["mma", "simt"])
@pytest.mark.parametrize("S,N,D,R,ko,M", WIDE)
def test_general_wide_shapes(S, N, D, R, ko, M, form, monkeypatch):
    want = _grad_form(monkeypatch, form, S)
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=S + D + M, src_scale=(0.5, 2.0), scale=1.7, eps=1e-4)
    info = attnres_multi_plan_info(wl.values.cuda(), M, R, key_offset=ko)
    assert info["bwd_general"] == want, info
    fwd, bwd, ref = _run_multi(wl, twice=True)
    errs = _check_multi(wl, fwd, bwd, ref, f"S{S} N{N} D{D} R{R} ko{ko} M{M} {form}")
    print(info, errs)


def _run_selected(wl, ids=None):
    v, bank, dy = wl.values.cuda(), wl.bank.cuda(), wl.dy.cuda()
    ids = wl.ids.cuda() if ids is None else ids.cuda()
    fwd = attnres_selected_fwd(v, bank, ids, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    bwd = attnres_selected_bwd(v, bank, ids, dy, fwd, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    return fwd, bwd


def _check_selected(wl, fwd, bwd, ref, tag):
    N, K, D, S = wl.N, wl.K, wl.D, wl.S
    y = to_np(fwd["y"]).reshape(N, K, D)
    errs = {"y": max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(K))}
    assert errs["y"] <= Y_REL, (tag, errs)
    check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, tag)
    check_vec_grad(bwd["dbank"], bwd["dbank_f32"], ref["dbank"][:wl.E], errs, tag, "dbank")
    return errs


@pytest.mark.parametrize("S,N,D,R,E,K", SELECTED_SHAPES)
def test_general_on_every_selected_shape(S, N, D, R, E, K, monkeypatch):
    monkeypatch.setenv("ATTNRES_MULTI_BWD", "general")
    wl = make_selected(S, N, D, R, E, K, seed=S * 41 + K, unused_rows=1 if E > 2 else 0)
    fwd, bwd = _run_selected(wl)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=wl.key_offset)
    errs = _check_selected(wl, fwd, bwd, ref, f"S{S} N{N} D{D} R{R} E{E} K{K}")
    if E > 2:  # the last bank row is never selected: its gradient is exactly zero
        assert torch.count_nonzero(bwd["dbank_f32"][E - 1]).item() == 0
    print(errs)


@pytest.mark.parametrize("S,N,D,R,E,K", [(10, 40, 8192, 8192, 5, 16), (9, 60, 4096, 1024, 80, 12),
                                         (6, 50, 1000, 300, 7, 5)])
def test_general_selected_wide(S, N, D, R, E, K):
    # sixteen slots over 16 KB rows; a bank too large for shared memory; an
    # unaligned key with a width 8 mod 16
    wl = make_selected(S, N, D, R, E, K, seed=S + E + K)
    fwd, bwd = _run_selected(wl)
    bwd2 = attnres_selected_bwd(wl.values.cuda(), wl.bank.cuda(), wl.ids.cuda(), wl.dy.cuda(), fwd,
                                key_offset=wl.key_offset)
    torch.cuda.synchronize()
    attnres_check_device_error()
    assert torch.equal(bwd["dvalues"], bwd2["dvalues"]) and torch.equal(bwd["dbank_f32"], bwd2["dbank_f32"])
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=wl.key_offset)
    print(_check_selected(wl, fwd, bwd, ref, f"S{S} D{D} E{E} K{K}"))


def test_general_selected_bad_id_reads_a_zero_query():
    wl = make_selected(6, 50, 1024, 256, 4, 6, seed=19)
    ids = wl.ids.clone()
    ids[7, 0] = -3
    ids[20, 5] = 9
    fwd, bwd = _run_selected(wl, ids)
    torch.cuda.synchronize()
    with pytest.raises(AttnresError):
        attnres_check_device_error()
    zbank = torch.cat([wl.bank, torch.zeros(1, wl.bank.shape[1], dtype=wl.bank.dtype)])
    zids = ids.clone().numpy()
    zids[(zids < 0) | (zids >= wl.E)] = wl.E
    ref = attnres_selected_oracle(wl.values, zbank, zids, dy=wl.dy, key_offset=wl.key_offset)
    _check_selected(wl, fwd, bwd, ref, "bad ids")
