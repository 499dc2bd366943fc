"""GPU parity of the cluster backward: tokens whose S source rows do not fit
one SM's shared memory are shared by a thread-block cluster of 2, 4 or 8
CTAs, each holding a column slice of every row, with the two full-width
reductions (<g, yhat> under the output norm, and the S dots <do, v_s>)
exchanged through distributed shared memory.

Checked against the FP64 oracle: both output-norm modes, R == D and sliced
keys at both placements, S below and above a warp's 32 lanes, every cluster
size, token counts below the number of clusters, bitwise run-to-run
determinism, and agreement with the one-CTA streaming backward that
ATTNRES_BWD_CLUSTER=0 selects for the same shapes.  ATTNRES_BWD_CLUSTER
selects each form: "<n>" resident slices on clusters of n, "s<n>" streamed
slices, "h<n>" streamed slices with two CTAs per SM, "0" no cluster.
"""
import os

import pytest
import torch

from attention_residuals_gb300 import attnres_bwd, attnres_fwd, attnres_plan_info
from attention_residuals_gb300.workloads import make_random
from oracle import attnres_oracle
from parity_utils import check_backward, check_forward, cuda_copy

pytestmark = pytest.mark.gpu

CASES = [
    # S, N, D, R, ko, out_norm, ATTNRES_BWD_CLUSTER, cluster size, resident
    (9, 97, 8192, 8192, 0, True, "2", 2, 1),         # two CTAs, two vectors per thread
    (24, 70, 8192, 8192, 0, True, "4", 4, 1),
    (64, 40, 8192, 8192, 0, True, "8", 8, 1),        # the deep workload's rows, four groups of 32 sources
    (64, 33, 8192, 2048, 6144, False, "8", 8, 1),    # sliced key in the final channels, no norm
    (40, 61, 6144, 1536, 0, False, "4", 4, 1),       # key in the first channels
    (65, 50, 2048, 2048, 0, True, "4", 4, 1),
    (33, 300, 4096, 1000, 3, True, "4", 4, 1),       # unaligned key slice
    (64, 3, 8192, 8192, 0, True, "8", 8, 1),         # fewer tokens than clusters
    (64, 40, 8192, 8192, 0, True, "s2", 2, 0),       # streamed slices, the caller's o or o rebuilt
    (64, 45, 8192, 8192, 0, True, "s4", 4, 0),
    (40, 61, 6144, 1536, 0, True, "s8", 8, 0),       # three vectors' worth of warps per slice
    (24, 70, 8192, 2048, 6144, False, "s2", 2, 0),
    (33, 300, 4096, 1000, 3, False, "s4", 4, 0),
    (64, 77, 2064, 2064, 0, True, "s2", 2, 0),       # a slice of 129 vectors: not every thread owns one
    (24, 77, 4112, 1024, 3088, False, "2", 2, 1),     # 257 vectors of two per thread
    (64, 45, 8192, 8192, 0, True, "h4", 4, 0),       # streamed slices, two CTAs per SM
    (40, 61, 6144, 1536, 0, False, "h8", 8, 0),
    (33, 300, 4096, 1000, 3, True, "h4", 4, 0),
    (9, 97, 8192, 8192, 0, True, None, 1, 0),        # the planner's own choice: short tokens stream on one CTA,
    (64, 160, 8192, 8192, 0, True, None, 2, 0),      # 1 MB tokens on clusters of two
]


@pytest.mark.parametrize("save_o_pre", [None, False])
@pytest.mark.parametrize("S,N,D,R,ko,out_norm,env,cl,resident", CASES)
def test_cluster_backward_matches_oracle(S, N, D, R, ko, out_norm, env, cl, resident, save_o_pre, monkeypatch):
    if save_o_pre is False and not (out_norm and not resident):
        pytest.skip("o is only saved for the streamed form with the output norm")
    if env is None:
        monkeypatch.delenv("ATTNRES_BWD_CLUSTER", raising=False)
    else:
        monkeypatch.setenv("ATTNRES_BWD_CLUSTER", env)
    wl = make_random(S, N, D, R, key_offset=ko, out_norm=out_norm, seed=S * 7 + D + N, scale=1.3)
    v, q, w, dy = cuda_copy(wl)
    info = attnres_plan_info(v, R, key_offset=ko, out_norm=out_norm)
    assert info["bwd_cluster"] == cl and info["bwd_resident"] == resident, info
    if cl == 1:
        pytest.skip("one CTA per token: covered by the streaming tests in test_parity_gpu.py")
    assert info["grid"] == info["bwd_partial_rows"] * cl and info["bwd_partial_rows"] <= N, info
    fwd = attnres_fwd(v, q, w_o=w, key_offset=ko, scale=wl.scale, save_o_pre=save_o_pre)
    # o is saved by default only when the backward streams the rows
    assert (fwd["o_pre"] is not None) == bool(out_norm and not resident and save_o_pre is None)
    outs = [attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=ko, scale=wl.scale) for _ in range(2)]
    torch.cuda.synchronize()
    for key in ("dvalues", "dq_f32", "dq") + (("dw_o_f32",) if out_norm else ()):
        assert torch.equal(outs[0][key], outs[1][key]), key
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=ko, scale=wl.scale)
    tag = f"S{S} N{N} D{D} R{R} ko{ko} cl{cl} resident={resident} o_pre={fwd['o_pre'] is not None}"
    check_forward(fwd, ref, out_norm=out_norm, tag=tag)
    errs = check_backward(outs[0], ref, out_norm=out_norm, tag=tag)
    print(tag, info, errs)


@pytest.mark.parametrize("S,D,out_norm", [(64, 8192, True), (40, 6144, False)])
def test_cluster_and_streaming_backward_agree(S, D, out_norm, monkeypatch):
    wl = make_random(S, 45, D, out_norm=out_norm, seed=S + D)
    v, q, w, dy = cuda_copy(wl)
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0, save_o_pre=False)
    clus = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0)
    monkeypatch.setenv("ATTNRES_BWD_CLUSTER", "0")
    assert attnres_plan_info(v, D, key_offset=0, out_norm=out_norm)["bwd_cluster"] == 1
    strm = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0)
    torch.cuda.synchronize()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=0)
    check_backward(clus, ref, out_norm=out_norm, tag="cluster")
    check_backward(strm, ref, out_norm=out_norm, tag="streaming")
    # the two reduction orders differ only by FP32 rounding
    d = (clus["dvalues"].float() - strm["dvalues"].float()).norm() / strm["dvalues"].float().norm()
    assert d.item() < 2e-3
