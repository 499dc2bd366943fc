"""GPU parity of the selected-query read ("Fast Attention Residuals", section
"Multi-query AttnRes": attnres_selected(sources, query_bank, ids) ->
[..., K, D]) through the C ABI, against the FP64 oracle.

Covers one and several query blocks per token, bank rows that no token
selects (zero gradient), repeated ids within a token, unaligned key slices,
the empty input, list sources, autograd through torch.compile, bitwise
determinism, and an out-of-range id (recorded as a device error, never read
out of bounds).  Tolerances as for the single-query read (parity_utils).
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres_check_device_error, attnres_selected, attnres_selected_bwd,
                                       attnres_selected_fwd)
from attention_residuals_gb300._lib import AttnresError
from attention_residuals_gb300.workloads import make_selected
from oracle.multi import attnres_selected_oracle
from op_grads import selected_grads
from parity_utils import (ALPHA_ABS, GRAD_REL_L2, STAT_REL, Y_REL, bf16_rne, check_dvalues, check_vec_grad,
                          rel_l2, to_np,
                          y_rel_err)

pytestmark = pytest.mark.gpu


def run_selected(wl, list_sources=False):
    v = wl.values.cuda()
    vals = list(v.unbind(0)) if list_sources else v
    bank, ids, dy = wl.bank.cuda(), wl.ids.cuda(), wl.dy.cuda()
    fwd = attnres_selected_fwd(vals, bank, ids, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    bwd = attnres_selected_bwd(vals, bank, ids, dy, fwd, key_offset=wl.key_offset, eps=wl.eps,
                               scale=wl.scale)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=wl.key_offset,
                                  eps=wl.eps, scale=wl.scale)
    return fwd, bwd, ref


def check(wl, fwd, bwd, ref, tag):
    N, K, D, S = wl.N, wl.K, wl.D, wl.S
    y = to_np(fwd["y"]).reshape(N, K, D)
    errs = {"y": max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(K)) if N else 0.0}
    assert errs["y"] <= Y_REL, (tag, errs)
    if N:
        errs["alpha"] = float(np.max(np.abs(to_np(fwd["alpha"]) - ref["alpha"])))
        errs["rstd"] = float(np.max(np.abs(to_np(fwd["rstd"]) / ref["rstd"] - 1)))
        z = ref["logit"]
        errs["logit"] = float(np.max(np.abs(to_np(fwd["logit"]) - z) / np.maximum(1, np.abs(z))))
        assert errs["alpha"] <= ALPHA_ABS, (tag, errs)
        assert errs["rstd"] <= STAT_REL, (tag, errs)
        assert errs["logit"] <= STAT_REL, (tag, errs)
    check_dvalues(to_np(bwd["dvalues"]).reshape(S, N, D), ref["dvalues"], errs, tag)
    check_vec_grad(bwd["dbank"], bwd["dbank_f32"], ref["dbank"], errs, tag, "dbank")
    return errs


SHAPES = [
    # S, N, D, R, E, K
    (8, 97, 1024, 64, 6, 2),
    (10, 150, 4096, 1024, 4, 2),
    (6, 129, 2048, 512, 9, 3),       # several query blocks in the backward
    (5, 61, 256, 100, 5, 4),         # unaligned key slice (scalar query gather)
    (12, 40, 512, 512, 16, 1),
    (4, 33, 4096, 4096, 7, 2),       # a bank too large to stay in shared memory
    (6, 70, 512, 100, 6, 2),         # one register block, unaligned key: per-channel dq reductions
]


@pytest.mark.parametrize("S,N,D,R,E,K", SHAPES)
def test_selected_matches_oracle(S, N, D, R, E, K):
    ko = 13 if R == 100 else None
    wl = make_selected(S, N, D, R, E, K, key_offset=ko, seed=S + 7 * E, src_scale=(0.5, 2.0), unused_rows=1)
    fwd, bwd, ref = run_selected(wl)
    errs = check(wl, fwd, bwd, ref, f"S{S} N{N} D{D} R{R} E{E} K{K}")
    # the last bank row is never selected: its gradient is exactly zero
    assert torch.count_nonzero(bwd["dbank_f32"][-1]).item() == 0
    print(errs)


def test_selected_repeated_ids_list_sources_and_determinism():
    wl = make_selected(7, 80, 2048, 256, 3, 3, seed=3)
    wl.ids[:, 1] = wl.ids[:, 0]          # a token reads the same bank row twice
    fwd, bwd, ref = run_selected(wl, list_sources=True)
    check(wl, fwd, bwd, ref, "repeated ids")
    v, bank, ids, dy = wl.values.cuda(), wl.bank.cuda(), wl.ids.cuda(), wl.dy.cuda()
    f = attnres_selected_fwd(v, bank, ids)
    a = attnres_selected_bwd(v, bank, ids, dy, f)
    b = attnres_selected_bwd(v, bank, ids, dy, f)
    torch.cuda.synchronize()
    assert torch.equal(a["dbank_f32"], b["dbank_f32"]) and torch.equal(a["dvalues"], b["dvalues"])


def test_selected_empty_input():
    v = torch.zeros((3, 0, 512), dtype=torch.bfloat16, device="cuda")
    bank = torch.ones((4, 128), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    f = attnres_selected_fwd(v, bank, ids)
    assert f["y"].shape == (0, 2, 512)
    g = attnres_selected_bwd(v, bank, ids, torch.zeros((0, 2, 512), dtype=torch.bfloat16, device="cuda"), f)
    torch.cuda.synchronize()
    assert torch.count_nonzero(g["dbank_f32"]).item() == 0 and g["dbank"].shape == (4, 128)


def test_selected_out_of_range_id_is_reported():
    wl = make_selected(4, 30, 1024, 256, 3, 2, seed=11)
    ids = wl.ids.clone()
    ids[5, 1] = 7                          # outside [0, 3)
    v, bank = wl.values.cuda(), wl.bank.cuda()
    f = attnres_selected_fwd(v, bank, ids.cuda())
    torch.cuda.synchronize()
    with pytest.raises(AttnresError) as e:
        attnres_check_device_error()
    assert e.value.name == "ATTNRES_ERR_DEVICE"
    attnres_check_device_error()           # the record was cleared
    # the backward reports it too; the bad slot adds to no bank row
    g = attnres_selected_bwd(v, bank, ids.cuda(), wl.dy.cuda(), f)
    torch.cuda.synchronize()
    with pytest.raises(AttnresError) as e:
        attnres_check_device_error()
    assert e.value.name == "ATTNRES_ERR_DEVICE"
    assert torch.isfinite(g["dbank_f32"]).all() and torch.isfinite(g["dvalues"].float()).all()


def test_selected_bad_id_reads_a_zero_query():
    # an id outside [0, E) is reported and otherwise acts as a zero query: the
    # results equal the oracle's with that slot pointing at an extra zero bank
    # row, and no bank row receives its gradient
    wl = make_selected(6, 50, 1024, 256, 4, 2, seed=17)
    ids = wl.ids.clone()
    ids[7, 0] = -3
    ids[20, 1] = 9
    v, bank, dy = wl.values.cuda(), wl.bank.cuda(), wl.dy.cuda()
    f = attnres_selected_fwd(v, bank, ids.cuda())
    g = attnres_selected_bwd(v, bank, ids.cuda(), dy, f)
    torch.cuda.synchronize()
    with pytest.raises(AttnresError):
        attnres_check_device_error()
    zbank = torch.cat([wl.bank, torch.zeros(1, wl.bank.shape[1], dtype=wl.bank.dtype)])
    zids = ids.clone().numpy()
    zids[(zids < 0) | (zids >= wl.E)] = wl.E
    ref = attnres_selected_oracle(wl.values, zbank, zids, dy=wl.dy, key_offset=wl.key_offset)
    y = to_np(f["y"]).reshape(wl.N, wl.K, wl.D)
    assert max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(wl.K)) <= Y_REL
    assert float(np.max(np.abs(to_np(f["alpha"]) - ref["alpha"]))) <= ALPHA_ABS
    assert rel_l2(to_np(g["dvalues"]), ref["dvalues"]) <= GRAD_REL_L2
    assert rel_l2(to_np(g["dbank_f32"]), ref["dbank"][:wl.E]) <= GRAD_REL_L2


def test_selected_autograd_compile():
    torch._dynamo.reset()
    wl = make_selected(5, 64, 1024, 128, 4, 2, seed=21)
    v = wl.values.cuda().requires_grad_(True)
    bank = wl.bank.cuda().requires_grad_(True)
    ids = wl.ids.cuda().view(8, 8, 2)
    f = torch.compile(lambda vv, bb, ii: attnres_selected(vv.view(5, 8, 8, 1024), bb, ii), fullgraph=True,
                      dynamic=False)
    y = f(v, bank, ids)
    assert y.shape == (8, 8, 2, 1024)
    y.backward(wl.dy.cuda().view(8, 8, 2, 1024))
    torch.cuda.synchronize()
    ref = attnres_selected_oracle(wl.values, wl.bank, wl.ids.numpy(), dy=wl.dy, key_offset=1024 - 128)
    assert max(y_rel_err(to_np(y).reshape(64, 2, 1024)[:, k], ref["y"][:, k]) for k in range(2)) <= Y_REL
    check_dvalues(to_np(v.grad), ref["dvalues"], {}, "autograd")
    # autograd's bf16 bank gradient is the operator's, bit for bit; its FP32 sum
    # is held to the tolerance and the bf16 copy must be its RNE rounding
    g = selected_grads(v.view(5, 8, 8, 1024), bank, ids, wl.dy.cuda().view(8, 8, 2, 1024))
    assert torch.equal(bank.grad, g["dbank"])
    check_vec_grad(g["dbank"], g["dbank_f32"], ref["dbank"], {}, "autograd", "dbank")


def test_selected_full_size_sampled():
    # the benchmark's selected-query workload at full size: sampled tokens
    # element by element, the bank gradient over every token
    wl = make_selected(10, 32768, 4096, 1024, 8, 2, seed=300, src_scale=(0.5, 2.0), device="cuda")
    v, bank, ids, dy = wl.values, wl.bank, wl.ids, wl.dy
    f = attnres_selected_fwd(v, bank, ids)
    b = attnres_selected_bwd(v, bank, ids, dy, f)
    b2 = attnres_selected_bwd(v, bank, ids, dy, f)
    torch.cuda.synchronize()
    attnres_check_device_error()
    assert torch.equal(b["dbank_f32"], b2["dbank_f32"]) and torch.equal(b["dvalues"], b2["dvalues"])
    del b2
    g = np.random.default_rng(2)
    idx = np.array(sorted(set(g.choice(wl.N, 40, replace=False).tolist()) | {0, wl.N - 1}))
    it = torch.as_tensor(idx, device="cuda")
    ref = attnres_selected_oracle(v.index_select(1, it).cpu(), bank.cpu(), ids.index_select(0, it).cpu().numpy(),
                                  dy=dy.index_select(0, it).cpu(), key_offset=wl.key_offset)
    y = to_np(f["y"].index_select(0, it))
    assert max(y_rel_err(y[:, k], ref["y"][:, k]) for k in range(2)) <= Y_REL
    check_dvalues(to_np(b["dvalues"].index_select(1, it)), ref["dvalues"], {}, "full")
    full = attnres_selected_oracle(v.cpu(), bank.cpu(), ids.cpu().numpy(), dy=dy.cpu(), key_offset=wl.key_offset,
                                   want_dvalues=False)
    check_vec_grad(b["dbank"], b["dbank_f32"], full["dbank"], {}, "full", "dbank")
