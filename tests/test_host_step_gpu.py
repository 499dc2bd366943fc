"""The host-buffer training step (attnres_step_host): sources and dy in
page-locked host memory, every result copied back, transfers overlapped
with the kernels chunk by chunk.  Per-token results (y, dvalues) must equal
the device path's bit for bit (same kernels, same plan per token); dq and
dw_o add the chunks' FP32 sums in chunk order and are checked against the
FP64 oracle.  Covers a ragged last chunk, one chunk larger than N, many
small chunks, the output norm and the empty input."""
import numpy as np
import pytest
import torch

from attention_residuals_gb300 import attnres_bwd, attnres_fwd, attnres_step_host
from attention_residuals_gb300.workloads import make_random
from oracle import attnres_oracle
from parity_utils import check_vec_grad

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,N,D,R,ko,out_norm,chunk", [
    (10, 5000, 4096, 4096, 0, True, 2048),     # ragged last chunk, output norm
    (6, 700, 2048, 512, 1536, False, 4096),    # one chunk larger than N
    (4, 333, 1024, 1024, 0, True, 64),         # many small chunks
])
def test_step_host_matches_device_path_and_oracle(S, N, D, R, ko, out_norm, chunk):
    wl = make_random(S, N, D, R, key_offset=ko, out_norm=out_norm, seed=N + S)
    hv = wl.values.pin_memory()
    hdy = wl.dy.pin_memory()
    res = attnres_step_host(hv, wl.q, hdy, w_o=wl.w_o, key_offset=ko, chunk_tokens=chunk)
    torch.cuda.synchronize()
    v, q, dy = wl.values.cuda(), wl.q.cuda(), wl.dy.cuda()
    w = wl.w_o.cuda() if out_norm else None
    f = attnres_fwd(v, q, w_o=w, key_offset=ko)
    b = attnres_bwd(v, q, dy, f, w_o=w, key_offset=ko)
    torch.cuda.synchronize()
    assert torch.equal(res["y"], f["y"].cpu())
    for s in range(S):
        assert torch.equal(res["dvalues"][s], b["dvalues"][s].cpu()), s
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, dy=wl.dy, key_offset=ko, want_dvalues=False)
    check_vec_grad(res["dq"], res["dq_f32"], ref["dq"], {}, "host step", "dq")
    if out_norm:
        check_vec_grad(res["dw_o"], res["dw_o_f32"], ref["dw_o"], {}, "host step", "dw_o")


def test_step_host_empty():
    v = torch.zeros((3, 0, 512), dtype=torch.bfloat16).pin_memory()
    q = torch.ones((512,), dtype=torch.bfloat16)
    res = attnres_step_host(v, q, torch.zeros((0, 512), dtype=torch.bfloat16), chunk_tokens=128)
    torch.cuda.synchronize()
    assert torch.count_nonzero(res["dq_f32"]).item() == 0
