"""Full-size parity: each of the five workloads at its full size, in the
launch configuration the benchmark uses (plan chosen by the library for the
shape), against the FP64 oracle.

Per-token outputs (y, alpha, rstd, logit, o_rstd, dvalues) are compared
element by element on a sample of tokens the oracle recomputes one by one
(tokens are independent).  dq and dw_o are sums over all N tokens; the
oracle computes them over every token (it does not materialise dvalues for
that run).
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import attnres_bwd, attnres_fwd, attnres_plan_info
from attention_residuals_gb300.workloads import make_workload
from oracle import attnres_oracle
from parity_utils import check_dvalues, check_forward, check_vec_grad, to_np

pytestmark = pytest.mark.gpu

CASES = [(2, 0), (3, 0), (4, 0), (4, 3072), (5, 0)]


def sample_tokens(N, wl, k=48, seed=0):
    g = np.random.default_rng(seed)
    idx = set(g.choice(N, size=min(k, N), replace=False).tolist())
    idx.update([0, 1, N - 1, N - 2, N // 2])
    idx.update(wl.notes.get("all_zero_tokens", [])[:4])
    return np.array(sorted(i for i in idx if 0 <= i < N))


@pytest.mark.parametrize("cfg,ko", CASES)
def test_full_size(cfg, ko):
    wl = make_workload(cfg, key_offset=ko, device="cuda")
    v, q, w, dy = wl.values, wl.q, wl.w_o, wl.dy
    info = attnres_plan_info(v, wl.R, key_offset=ko, out_norm=wl.out_norm)
    fwd = attnres_fwd(v, q, w_o=w, key_offset=ko)
    bwd = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=ko)
    bwd2 = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=ko)
    torch.cuda.synchronize()
    # run-to-run determinism of every backward output
    assert torch.equal(bwd["dq_f32"], bwd2["dq_f32"])
    assert torch.equal(bwd["dvalues"], bwd2["dvalues"])
    if wl.out_norm:
        assert torch.equal(bwd["dw_o_f32"], bwd2["dw_o_f32"])
    del bwd2

    # sampled tokens, element by element
    idx = sample_tokens(wl.N, wl, seed=cfg)
    it = torch.as_tensor(idx, device="cuda")
    vs = v.index_select(1, it).cpu()
    ref = attnres_oracle(vs, q.cpu(), w_o=None if w is None else w.cpu(),
                         dy=dy.index_select(0, it).cpu(), key_offset=ko)
    sub = {"y": fwd["y"].index_select(0, it), "alpha": fwd["alpha"].index_select(0, it),
           "rstd": fwd["rstd"].index_select(0, it), "logit": fwd["logit"].index_select(0, it),
           "o_rstd": None if fwd["o_rstd"] is None else fwd["o_rstd"].index_select(0, it)}
    errs = check_forward(sub, ref, out_norm=wl.out_norm, tag=f"cfg{cfg} ko={ko}")
    check_dvalues(to_np(bwd["dvalues"].index_select(1, it)), ref["dvalues"], errs, f"cfg{cfg}")

    # dq / dw_o over all tokens
    full = attnres_oracle(v.cpu(), q.cpu(), w_o=None if w is None else w.cpu(), dy=dy.cpu(),
                          key_offset=ko, want_dvalues=False)
    check_vec_grad(bwd["dq"], bwd["dq_f32"], full["dq"], errs, f"cfg{cfg}", "dq")
    if wl.out_norm:
        check_vec_grad(bwd["dw_o"], bwd["dw_o_f32"], full["dw_o"], errs, f"cfg{cfg}", "dw_o")
    print(f"cfg{cfg} ko={ko} plan={info} errs={errs}")
