"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Sizes here finish in the oracle within seconds yet span many CTAs of the
persistent grid and leave a ragged tail (N not a multiple of the grid).
Full-size workloads are in test_parity_full_gpu.py.
"""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import (attnres, attnres_bwd, attnres_check_device_error,
                                       attnres_fwd, attnres_plan_info)
from attention_residuals_gb300.workloads import make_random, make_workload
from oracle import attnres_oracle
from op_grads import read_grads
from parity_utils import check_backward, check_dvalues, check_forward, check_vec_grad, cuda_copy, rel_l2, to_np

pytestmark = pytest.mark.gpu


def run_both(wl, *, split_n_threshold=0, list_sources=False):
    v, q, w, dy = cuda_copy(wl)
    vals = list(v.unbind(0)) if list_sources else v
    fwd = attnres_fwd(vals, q, w_o=w, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale)
    bwd = attnres_bwd(vals, q, dy, fwd, w_o=w, key_offset=wl.key_offset, eps=wl.eps,
                      scale=wl.scale, split_n_threshold=split_n_threshold)
    torch.cuda.synchronize()
    attnres_check_device_error()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=wl.key_offset,
                         eps=wl.eps, scale=wl.scale)
    return fwd, bwd, ref


@pytest.mark.parametrize("cfg,N", [(1, None), (2, 301), (3, 157), (4, 263), (5, 40)])
@pytest.mark.parametrize("ko_mode", ["first", "final"])
def test_workload_shapes_small_N(cfg, N, ko_mode):
    from attention_residuals_gb300.workloads import CONFIGS
    c = CONFIGS[cfg]
    if ko_mode == "final" and c["R"] == c["D"]:
        pytest.skip("key offset only matters when R < D")
    ko = 0 if ko_mode == "first" else c["D"] - c["R"]
    wl = make_workload(cfg, N=N, key_offset=ko)
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=wl.out_norm, tag=wl.name)
    check_backward(bwd, ref, out_norm=wl.out_norm, tag=wl.name)


@pytest.mark.parametrize("S", [1, 3, 7, 10, 15, 29])
def test_source_count_matrix(S):
    wl = make_random(S, 211, 1024, out_norm=(S % 2 == 1), seed=S)
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=wl.out_norm, tag=f"S={S}")
    check_backward(bwd, ref, out_norm=wl.out_norm, tag=f"S={S}")


@pytest.mark.parametrize("R,ko", [(16, 0), (16, 2048 - 16), (64, 512), (384, 0), (640, 1408),
                                  (512, 0), (2048, 0), (100, 3), (7, 2041), (1, 1000)])
def test_ranks_and_offsets(R, ko):
    wl = make_random(6, 173, 2048, R, key_offset=ko, out_norm=True, seed=R + ko)
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=True, tag=f"R={R} ko={ko}")
    check_backward(bwd, ref, out_norm=True, tag=f"R={R} ko={ko}")


@pytest.mark.parametrize("D", [8, 24, 520, 1000, 3072, 8192])
def test_odd_widths(D):
    wl = make_random(4, 67, D, out_norm=True, seed=D)
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=True, tag=f"D={D}")
    check_backward(bwd, ref, out_norm=True, tag=f"D={D}")


@pytest.mark.parametrize("N", [1, 2, 3, 17, 152, 153, 305])
def test_token_counts(N):
    wl = make_random(5, N, 512, out_norm=True, seed=N)
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=True, tag=f"N={N}")
    check_backward(bwd, ref, out_norm=True, tag=f"N={N}")


@pytest.mark.parametrize("save_o_pre", [None, False, True])
def test_streaming_backward_many_sources(save_o_pre, monkeypatch):
    # 64 rows of 8 KB do not fit one SM: with the cluster backward switched off
    # the backward streams the rows once per pass (o rebuild unless o_pre was
    # saved, dot pass, key slices).
    monkeypatch.setenv("ATTNRES_BWD_CLUSTER", "0")
    wl = make_random(64, 90, 4096, 1024, key_offset=1024, out_norm=True, seed=64)
    v, q, w, dy = cuda_copy(wl)
    info = attnres_plan_info(v, 1024, key_offset=1024, out_norm=True)
    assert info["bwd_resident"] == 0 and info["bwd_cluster"] == 1
    fwd = attnres_fwd(v, q, w_o=w, key_offset=1024, save_o_pre=save_o_pre)
    assert (fwd["o_pre"] is not None) == (save_o_pre is not False)
    bwd = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=1024)
    bwd2 = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=1024)
    torch.cuda.synchronize()
    for key in ("dvalues", "dq_f32", "dw_o_f32"):
        assert torch.equal(bwd[key], bwd2[key]), key
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=1024)
    check_forward(fwd, ref, out_norm=True, tag="S64 streaming")
    check_backward(bwd, ref, out_norm=True, tag="S64 streaming")
    if fwd["o_pre"] is not None:
        o_ref = ref["y"] / (wl.w_o.double().numpy() * ref["o_rstd"][:, None])
        assert rel_l2(to_np(fwd["o_pre"]), o_ref) < 1e-5


@pytest.mark.parametrize("cluster", ["0", "s2"])
@pytest.mark.parametrize("S,D,outn", [(24, 8192, True), (40, 6144, False), (130 // 2, 2048, True)])
def test_streaming_wide_rows_deterministic(S, D, outn, cluster, monkeypatch):
    # rows too many to stay resident in one SM: streamed by one CTA (4 vectors
    # per thread for D > 4096) or held as column slices by a cluster
    monkeypatch.setenv("ATTNRES_BWD_CLUSTER", cluster)
    wl = make_random(S, 70, D, out_norm=outn, seed=S + D)
    v, q, w, dy = cuda_copy(wl)
    info = attnres_plan_info(v, D, key_offset=0, out_norm=outn)
    assert (info["bwd_cluster"] > 1) == (cluster != "0"), info
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0)
    outs = [attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0) for _ in range(3)]
    torch.cuda.synchronize()
    for b in outs[1:]:
        assert torch.equal(b["dvalues"], outs[0]["dvalues"])
        assert torch.equal(b["dq_f32"], outs[0]["dq_f32"])
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=0)
    check_forward(fwd, ref, out_norm=outn, tag=f"S{S} D{D} {info}")
    check_backward(outs[0], ref, out_norm=outn, tag=f"S{S} D{D} {info}")


def test_resident_backward_with_saved_o_pre():
    wl = make_random(10, 120, 4096, out_norm=True, seed=65)
    v, q, w, dy = cuda_copy(wl)
    assert attnres_plan_info(v, 4096, key_offset=0, out_norm=True)["bwd_resident"] == 1
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0, save_o_pre=True)
    assert fwd["o_pre"] is not None and fwd["o_pre"].dtype == torch.float32
    bwd = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0)
    torch.cuda.synchronize()
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=0)
    check_backward(bwd, ref, out_norm=True, tag="resident + o_pre")


@pytest.mark.parametrize("thr", [1, 10 ** 9])
def test_both_reduction_paths(thr):
    wl = make_random(8, 500, 2048, out_norm=True, seed=5)
    fwd, bwd, ref = run_both(wl, split_n_threshold=thr)
    check_backward(bwd, ref, out_norm=True, tag=f"threshold={thr}")


def test_reduction_paths_deterministic():
    wl = make_random(8, 700, 1024, out_norm=True, seed=6)
    v, q, w, dy = cuda_copy(wl)
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0)
    outs = []
    for thr in (1, 1, 10 ** 9, 10 ** 9):  # finalize kernel twice, in-kernel reduction twice
        b = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0, split_n_threshold=thr)
        outs.append((b["dq_f32"].clone(), b["dw_o_f32"].clone(), b["dvalues"].clone()))
    torch.cuda.synchronize()
    for a, b in ((outs[0], outs[1]), (outs[2], outs[3])):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_list_sources_and_shared_source():
    wl = make_random(5, 129, 1024, out_norm=False, seed=11)
    v, q, _, dy = cuda_copy(wl)
    srcs = [v[0], v[1], v[0], v[2]]          # v[0] read twice
    packed = torch.stack([s for s in srcs])
    vref = torch.stack([wl.values[i] for i in (0, 1, 0, 2)])
    fwd = attnres_fwd(srcs, q, key_offset=0)
    bwd = attnres_bwd(srcs, q, dy, fwd, key_offset=0)
    ref = attnres_oracle(vref, wl.q, dy=wl.dy, key_offset=0)
    check_forward(fwd, ref, out_norm=False, tag="list")
    check_backward(bwd, ref, out_norm=False, tag="list")
    # autograd adds the two gradients of the shared source
    x0 = v[0].clone().requires_grad_(True)
    x1 = v[1].clone().requires_grad_(True)
    x2 = v[2].clone().requires_grad_(True)
    qq = q.clone().requires_grad_(True)
    y = attnres([x0, x1, x0, x2], qq, key_offset=0)
    y.backward(dy)
    g0 = ref["dvalues"][0] + ref["dvalues"][2]
    check_dvalues(to_np(x0.grad), g0, {}, "shared x0")
    g = read_grads([x0, x1, x0, x2], qq, dy, key_offset=0)
    assert torch.equal(qq.grad, g["dq"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "autograd", "dq")
    del packed


def test_strided_sources():
    # Sources that are column slices of a wider buffer (row stride > D).
    wl = make_random(4, 133, 1024, out_norm=True, seed=12)
    v, q, w, dy = cuda_copy(wl)
    wide = torch.zeros((4, 133, 1536), dtype=torch.bfloat16, device="cuda")
    wide[:, :, 256:1280] = v
    srcs = [wide[s, :, 256:1280] for s in range(4)]
    assert srcs[0].stride(0) == 1536
    fwd = attnres_fwd(srcs, q, w_o=w, key_offset=0)
    assert fwd["params"].src_ld == 1536
    bwd = attnres_bwd(srcs, q, dy, fwd, w_o=w, key_offset=0)
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=0)
    check_forward(fwd, ref, out_norm=True, tag="strided")
    check_backward(bwd, ref, out_norm=True, tag="strided")


def test_poisoned_outputs_and_workspace():
    wl = make_random(6, 211, 2048, out_norm=True, seed=13)
    v, q, w, dy = cuda_copy(wl)
    nan = float("nan")
    N, D, S = 211, 2048, 6
    out = {"y": torch.full((N, D), nan, dtype=torch.bfloat16, device="cuda"),
           "alpha": torch.full((N, S), nan, device="cuda"),
           "rstd": torch.full((N, S), nan, device="cuda"),
           "logit": torch.full((N, S), nan, device="cuda"),
           "o_rstd": torch.full((N,), nan, device="cuda"),
           "o_pre": torch.full((N, D), nan, device="cuda")}
    fwd = attnres_fwd(v, q, w_o=w, key_offset=0, out=out, save_o_pre=True)
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=0)
    for thr in (1, 10 ** 9):
        ws = torch.full((1 << 22,), 0xFF, dtype=torch.uint8, device="cuda")
        dvals = torch.full((S, N, D), nan, dtype=torch.bfloat16, device="cuda")
        bwd = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=0, split_n_threshold=thr,
                          workspace=ws, dvalues=dvals)
        torch.cuda.synchronize()
        check_forward(fwd, ref, out_norm=True, tag="poison")
        check_backward(bwd, ref, out_norm=True, tag=f"poison thr={thr}")


def test_zero_rows_eps_floor():
    wl = make_workload(4, N=300, key_offset=0)
    assert wl.notes["zero_rows"] > 0
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=False, tag="zero rows")
    check_backward(bwd, ref, out_norm=False, tag="zero rows")
    for n in wl.notes["all_zero_tokens"]:
        np.testing.assert_allclose(to_np(fwd["alpha"])[n], 1.0 / wl.S, atol=1e-6)


def test_cuda_graph_replay():
    wl = make_random(8, 400, 2048, out_norm=True, seed=14)
    v, q, w, dy = cuda_copy(wl)
    fwd0 = attnres_fwd(v, q, w_o=w, key_offset=0)
    ws = torch.empty((1 << 24,), dtype=torch.uint8, device="cuda")
    dv = torch.empty_like(v)
    attnres_bwd(v, q, dy, fwd0, w_o=w, key_offset=0, workspace=ws, dvalues=dv)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = {k: torch.empty_like(fwd0[k]) for k in ("y", "alpha", "rstd", "logit", "o_rstd")}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            f = attnres_fwd(v, q, w_o=w, key_offset=0, out=out)
            b = attnres_bwd(v, q, dy, f, w_o=w, key_offset=0, workspace=ws, dvalues=dv)
    # change the inputs in place, replay, compare with the oracle on the new inputs
    wl2 = make_random(8, 400, 2048, out_norm=True, seed=15)
    v.copy_(wl2.values.cuda())
    dy.copy_(wl2.dy.cuda())
    g.replay()
    torch.cuda.synchronize()
    ref = attnres_oracle(wl2.values, wl.q, w_o=wl.w_o, dy=wl2.dy, key_offset=0)
    check_forward(f, ref, out_norm=True, tag="graph")
    check_backward(b, ref, out_norm=True, tag="graph")


def test_empty_input_is_noop():
    v = torch.empty((3, 0, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.randn(64, device="cuda").to(torch.bfloat16)
    fwd = attnres_fwd(v, q)
    assert fwd["y"].shape == (0, 64)
    bwd = attnres_bwd(v, q, torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), fwd)
    assert bwd["dvalues"].shape == (3, 0, 64)


def test_autograd_matches_explicit_calls():
    wl = make_random(5, 64, 512, 128, key_offset=384, out_norm=True, seed=16)
    v, q, w, dy = cuda_copy(wl)
    vv = v.clone().requires_grad_(True)
    qq = q.clone().requires_grad_(True)
    ww = w.clone().requires_grad_(True)
    y = attnres(vv, qq, out_norm_weight=ww)      # default key_offset = D - R = 384
    y.backward(dy)
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=384)
    check_dvalues(to_np(vv.grad), ref["dvalues"], {}, "autograd")
    g = read_grads(vv, qq, dy, w_o=ww)
    assert torch.equal(qq.grad, g["dq"]) and torch.equal(ww.grad, g["dw_o"])
    check_vec_grad(g["dq"], g["dq_f32"], ref["dq"], {}, "autograd", "dq")
    check_vec_grad(g["dw_o"], g["dw_o_f32"], ref["dw_o"], {}, "autograd", "dw_o")


@pytest.mark.parametrize("S,N,D,R,norm", [(8, 700, 2048, 2048, False), (10, 613, 2048, 512, True),
                                          (16, 900, 1024, 1024, False), (12, 500, 1536, 1536, True),
                                          (6, 400, 520, 136, True)])
def test_narrow_rows_two_ctas_per_sm(S, N, D, R, norm):
    # resident rows of at most 2048 channels: two backward CTAs share each SM
    wl = make_random(S, N, D, R, key_offset=D - R, out_norm=norm, seed=S + D)
    info = attnres_plan_info(wl.values.cuda(), R, key_offset=D - R, out_norm=norm)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert info["bwd_resident"] == 1 and info["grid"] == min(N, 2 * sms), info
    assert info["consumer_warps"] % 1000 <= 4, info
    fwd, bwd, ref = run_both(wl)
    check_forward(fwd, ref, out_norm=norm, tag="narrow")
    print(check_backward(bwd, ref, out_norm=norm, tag=f"narrow S{S} D{D}"))
