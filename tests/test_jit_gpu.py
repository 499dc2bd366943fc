"""The forward compiled at run time for a plan's exact shape (NVRTC; the
source count, rows per chunk, softmax group rows and ring depth fixed at
compile time) against the precompiled kernels on the same inputs, and the
FP64 oracle.  The two kernels do the same arithmetic in the same order, so
their outputs must agree bit for bit."""
import pytest
import torch

from attention_residuals_gb300 import (attnres_check_device_error, attnres_fwd, attnres_jit_kernel_count,
                                       attnres_partial_fwd)
from attention_residuals_gb300.workloads import make_workload
from oracle import attnres_oracle
from parity_utils import check_forward

pytestmark = pytest.mark.gpu


def _fwd(monkeypatch, jit, *args, **kw):
    monkeypatch.setenv("ATTNRES_JIT", "1" if jit else "0")
    out = attnres_fwd(*args, **kw)
    torch.cuda.synchronize()
    attnres_check_device_error()
    return out


@pytest.mark.parametrize("cfg,N,save_o", [(3, 2048, False), (3, 1536, True), (2, 4096, False), (4, 3000, False)])
def test_runtime_compiled_forward_matches_precompiled(monkeypatch, cfg, N, save_o):
    wl = make_workload(cfg, N=N, seed=70 + cfg, device="cuda")
    w = wl.w_o if wl.out_norm else None
    kw = dict(w_o=w, key_offset=wl.key_offset)
    if save_o:
        kw["save_o_pre"] = True
    ref = _fwd(monkeypatch, False, wl.values, wl.q, **kw)
    before = attnres_jit_kernel_count()
    got = _fwd(monkeypatch, True, wl.values, wl.q, **kw)
    assert attnres_jit_kernel_count() >= max(before, 1), "the run-time compiled kernel did not run"
    for k in ("y", "alpha", "rstd", "logit", "o_rstd", "o_pre"):
        if ref.get(k) is not None:
            assert torch.equal(ref[k], got[k]), k


def test_runtime_compiled_forward_matches_oracle(monkeypatch):
    wl = make_workload(3, N=1024, seed=7, device="cuda")
    got = _fwd(monkeypatch, True, wl.values, wl.q, w_o=wl.w_o, key_offset=wl.key_offset, eps=wl.eps,
               scale=wl.scale)
    assert attnres_jit_kernel_count() >= 1
    ref = attnres_oracle(wl.values.cpu(), wl.q.cpu(), w_o=wl.w_o.cpu(), key_offset=wl.key_offset, eps=wl.eps,
                         scale=wl.scale)
    check_forward(got, ref, out_norm=True, tag="run-time compiled forward")


def test_runtime_compiled_fused_partial_forward(monkeypatch):
    wl = make_workload(4, N=2048, seed=9, device="cuda")
    comp = list(wl.values[:-1].unbind(0))
    g = torch.Generator(device="cuda").manual_seed(10)
    delta = torch.randn(wl.values[-1].shape, generator=g, device="cuda").to(torch.bfloat16)
    outs = []
    for jit in (False, True):
        monkeypatch.setenv("ATTNRES_JIT", "1" if jit else "0")
        outs.append(attnres_partial_fwd(comp, wl.values[-1], delta, wl.q, key_offset=wl.key_offset))
        torch.cuda.synchronize()
    attnres_check_device_error()
    for k in ("y", "alpha", "partial_new"):
        assert torch.equal(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("selected", [False, True])
def test_runtime_compiled_multi_forward_matches_precompiled(monkeypatch, selected):
    from attention_residuals_gb300 import attnres_multi_fwd, attnres_selected_fwd
    from attention_residuals_gb300.workloads import make_multi, make_selected
    outs = []
    if selected:
        wl = make_selected(10, 2048, 4096, 1024, 8, 2, seed=12, src_scale=(0.5, 2.0), device="cuda")
        run = lambda: attnres_selected_fwd(wl.values, wl.bank, wl.ids)
    else:
        wl = make_multi(10, 2048, 4096, 1024, 2, seed=13, src_scale=(0.5, 2.0), device="cuda")
        run = lambda: attnres_multi_fwd(wl.values, wl.queries)
    for jit in (False, True):
        monkeypatch.setenv("ATTNRES_JIT", "1" if jit else "0")
        before = attnres_jit_kernel_count()
        outs.append(run())
        torch.cuda.synchronize()
        if jit:
            assert attnres_jit_kernel_count() >= max(before, 1)
    attnres_check_device_error()
    for k in ("y", "alpha", "rstd", "logit"):
        assert torch.equal(outs[0][k], outs[1][k]), k
