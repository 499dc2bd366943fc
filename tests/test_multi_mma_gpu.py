"""GPU parity of the tensor-core multi-query forward (mma.m16n8k16: logits as
queries x key channels x sources, outputs as queries x sources x channels,
FP32 weights entering as three bf16 terms) against the FP64 oracle.

"Fast Attention Residuals", section "Multi-query AttnRes": queries [M, R],
1 <= M <= 16, and attnres_selected with K slots per token.  The form runs by
default from nine queries up when a token's S <= 32 rows fit in shared
memory twice, R is a multiple of 16 and the key starts on an 8-channel
boundary; ATTNRES_MULTI_FWD=mma forces it for every query count and
ATTNRES_MULTI_FWD=simt turns it off.
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres_check_device_error, attnres_multi_bwd, attnres_multi_fwd,
                                       attnres_multi_plan_info, attnres_selected_fwd)
from attention_residuals_gb300._lib import AttnresError
from attention_residuals_gb300.workloads import make_multi, make_selected
from oracle.multi import attnres_multi_oracle, attnres_selected_oracle
from parity_utils import ALPHA_ABS, STAT_REL, Y_REL, check_dvalues, check_vec_grad, to_np, y_rel_err

pytestmark = pytest.mark.gpu

SHAPES = [
    # S, N, D, R, ko, M
    (8, 2, 1024, 64, 960, 2),          # the page's example, forced
    (10, 301, 1024, 1024, 0, 16),      # sixteen queries, R == D
    (10, 257, 4096, 1024, 3072, 8),    # the long workload's rows, eight queries
    (32, 97, 512, 256, 128, 12),       # the most sources the form takes (two K tiles of 16)
    (17, 120, 2048, 512, 1536, 5),     # a source count across a K tile boundary
    (1, 77, 1024, 1024, 0, 16),        # one source: y_m = v
    (3, 60, 16, 16, 0, 16),            # the narrowest rows
    (3, 150, 8192, 4096, 4096, 6),     # the widest rows (one CTA per SM)
    (9, 1000, 2048, 2048, 0, 16),      # many tokens per CTA
]


def _check(wl, fwd, ref, tag):
    M, N, D = wl.M, wl.N, wl.D
    y = to_np(fwd["y"]).reshape(M, N, D)
    errs = {"y": max(y_rel_err(y[m], ref["y"][m]) for m in range(M))}
    errs["alpha"] = float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"])))
    errs["rstd"] = float(np.max(np.abs(to_np(fwd["rstd"]) / ref["rstd"] - 1)))
    z = ref["logit"]
    errs["logit"] = float(np.max(np.abs(to_np(fwd["logit"]) - z) / np.maximum(1, np.abs(z))))
    assert errs["y"] <= Y_REL and errs["alpha"] <= ALPHA_ABS, (tag, errs)
    assert errs["rstd"] <= STAT_REL and errs["logit"] <= STAT_REL, (tag, errs)
    return errs


@pytest.mark.parametrize("S,N,D,R,ko,M", SHAPES)
def test_mma_forward_matches_oracle(S, N, D, R, ko, M, monkeypatch):
    monkeypatch.setenv("ATTNRES_MULTI_FWD", "mma")
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=S * 5 + M, src_scale=(0.5, 2.0), scale=1.3, eps=1e-4)
    v, Q = wl.values.cuda(), wl.queries.cuda()
    info = attnres_multi_plan_info(v, M, R, key_offset=ko)
    assert info["fwd_tensor_cores"] == 1, info
    fwd = attnres_multi_fwd(v, Q, key_offset=ko, eps=wl.eps, scale=wl.scale)
    again = attnres_multi_fwd(v, Q, key_offset=ko, eps=wl.eps, scale=wl.scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    for key in ("y", "alpha", "rstd", "logit"):
        assert torch.equal(fwd[key], again[key]), key  # run to run
    ref = attnres_multi_oracle(wl.values, wl.queries, dy=None, key_offset=ko, eps=wl.eps, scale=wl.scale)
    print(info, _check(wl, fwd, ref, f"S{S} N{N} D{D} R{R} ko{ko} M{M}"))


def test_token_major_output_and_default_choice(monkeypatch):
    monkeypatch.delenv("ATTNRES_MULTI_FWD", raising=False)
    wl = make_multi(10, 211, 2048, 512, 9, key_offset=1536, seed=3)
    v, Q = wl.values.cuda(), wl.queries.cuda()
    assert attnres_multi_plan_info(v, 9, 512, key_offset=1536)["fwd_tensor_cores"] == 1
    assert attnres_multi_plan_info(v, 8, 512, key_offset=1536)["fwd_tensor_cores"] == 0  # eight: the other form
    qm = attnres_multi_fwd(v, Q, key_offset=1536)
    tm = attnres_multi_fwd(v, Q, key_offset=1536, token_major=True)
    torch.cuda.synchronize()
    assert torch.equal(qm["y"], tm["y"].permute(1, 0, 2))
    assert torch.equal(qm["alpha"], tm["alpha"])


@pytest.mark.parametrize("S,N,D,R,ko,M", [(10, 301, 1024, 1024, 0, 16), (10, 257, 4096, 1024, 3072, 8)])
def test_mma_and_simt_forms_agree(S, N, D, R, ko, M, monkeypatch):
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=11)
    v, Q, dy = wl.values.cuda(), wl.queries.cuda(), wl.dy.cuda()
    out = {}
    for form in ("mma", "simt"):
        monkeypatch.setenv("ATTNRES_MULTI_FWD", form)
        assert attnres_multi_plan_info(v, M, R, key_offset=ko)["fwd_tensor_cores"] == (form == "mma")
        f = attnres_multi_fwd(v, Q, key_offset=ko)
        out[form] = (f, attnres_multi_bwd(v, Q, dy, f, key_offset=ko))
    torch.cuda.synchronize()
    a, b = out["mma"][0], out["simt"][0]
    assert float((a["alpha"] - b["alpha"]).abs().max()) <= 2e-6
    ya, yb = a["y"].float(), b["y"].float()
    assert float(((ya - yb).norm() / yb.norm())) <= 2e-3
    # the backward from either forward's statistics matches the oracle
    ref = attnres_multi_oracle(wl.values, wl.queries, dy=wl.dy, key_offset=ko)
    for form in ("mma", "simt"):
        bwd = out[form][1]
        errs = {}
        check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, form)
        check_vec_grad(bwd["dq"], bwd["dq_f32"], ref["dq"], errs, form, "dq")


@pytest.mark.parametrize("S,N,D,R,E,K", [(10, 150, 4096, 1024, 4, 8), (8, 97, 1024, 64, 6, 16),
                                         (12, 80, 512, 512, 16, 5)])
def test_mma_selected_forward_matches_oracle(S, N, D, R, E, K, monkeypatch):
    monkeypatch.setenv("ATTNRES_MULTI_FWD", "mma")
    wl = make_selected(S, N, D, R, E, K, seed=S + K)
    v, bank, ids = wl.values.cuda(), wl.bank.cuda(), wl.ids.cuda()
    fwd = attnres_selected_fwd(v, bank, ids, key_offset=wl.key_offset)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), key_offset=wl.key_offset)
    y = to_np(fwd["y"]).reshape(N, K, D)
    err = max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(K))
    assert err <= Y_REL, err
    assert float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"]))) <= ALPHA_ABS


def test_mma_selected_bad_id_reads_a_zero_query(monkeypatch):
    monkeypatch.setenv("ATTNRES_MULTI_FWD", "mma")
    wl = make_selected(6, 50, 1024, 256, 4, 6, seed=19)
    ids = wl.ids.clone()
    ids[7, 0] = -3
    ids[20, 5] = 9
    fwd = attnres_selected_fwd(wl.values.cuda(), wl.bank.cuda(), ids.cuda(), key_offset=wl.key_offset)
    torch.cuda.synchronize()
    with pytest.raises(AttnresError):
        attnres_check_device_error()
    zbank = torch.cat([wl.bank, torch.zeros(1, wl.bank.shape[1], dtype=wl.bank.dtype)])
    zids = ids.clone().numpy()
    zids[(zids < 0) | (zids >= wl.E)] = wl.E
    ref = attnres_selected_oracle(wl.values, zbank, zids, key_offset=wl.key_offset)
    y = to_np(fwd["y"]).reshape(50, 6, 1024)
    assert max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(6)) <= Y_REL
