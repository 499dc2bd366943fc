"""The backward entry point that allocates nothing (attnres_bwd_noalloc).

Callers that cannot allocate device memory during the call -- code being
captured into a CUDA graph, plugins that must stay off the host process's
allocator, latency-critical paths that cannot afford cudaMalloc's implicit
synchronisation -- use the library's fixed scratch array instead of a
workspace.  It runs the same plan and the same kernels as the workspace
entry point, with fixed reduction orders, so its results must equal that
entry point's bit for bit -- on consecutive calls that reuse the shared
array (a stale ticket or a wrong scratch offset shows up as a difference).
This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import pytest
import torch

from attention_residuals_gb300 import _lib, attnres_bwd, attnres_fwd
from attention_residuals_gb300.ops import _ptr, _stream, make_params
from attention_residuals_gb300.workloads import make_random

pytestmark = pytest.mark.gpu


def call_noalloc(wl, v, q, w, dy, fwd, thr, outs):
    """Call attnres_bwd_noalloc through the C ABI with preallocated outputs."""
    lib = _lib.load()
    view = fwd["view"]
    p = make_params(view, wl.R, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale,
                    out_norm=w is not None, split_n_threshold=thr)
    dvals, dq, dq32, dw, dw32 = outs
    S = wl.S
    dptrs = (ctypes.c_void_p * S)(*[dvals[s].data_ptr() for s in range(S)])
    rc = lib.attnres_bwd_noalloc(
        ctypes.byref(p), _ptr(q), _ptr(w), _ptr(dy), _ptr(fwd["alpha"]), _ptr(fwd["rstd"]),
        _ptr(fwd["logit"]), _ptr(fwd["o_rstd"]), _ptr(fwd["o_pre"]), dptrs, ctypes.c_int64(wl.D),
        _ptr(dq), _ptr(dq32), _ptr(dw), _ptr(dw32), _stream(None))
    assert rc == 0, _lib.STATUS.get(rc, rc)


@pytest.mark.parametrize("thr", [10 ** 9, 1])  # in-kernel reduction (tickets) and finalize kernel
def test_noalloc_matches_workspace_path_twice(thr):
    wl = make_random(6, 301, 2048, out_norm=True, seed=77)
    v = wl.values.cuda()
    q = wl.q.cuda()
    w = wl.w_o.cuda()
    dy = wl.dy.cuda()
    fwd = attnres_fwd(v, q, w_o=w, key_offset=wl.key_offset)
    ref = attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=wl.key_offset, split_n_threshold=thr)
    for _ in range(2):  # two calls in a row reuse the shared scratch array
        outs = (torch.full_like(v, float("nan")),
                torch.full((wl.R,), float("nan"), dtype=torch.bfloat16, device="cuda"),
                torch.full((wl.R,), float("nan"), device="cuda"),
                torch.full((wl.D,), float("nan"), dtype=torch.bfloat16, device="cuda"),
                torch.full((wl.D,), float("nan"), device="cuda"))
        call_noalloc(wl, v, q, w, dy, fwd, thr, outs)
        torch.cuda.synchronize()
        dvals, dq, dq32, dw, dw32 = outs
        assert torch.equal(dvals, ref["dvalues"])
        assert torch.equal(dq32, ref["dq_f32"]) and torch.equal(dq, ref["dq"])
        assert torch.equal(dw32, ref["dw_o_f32"]) and torch.equal(dw, ref["dw_o"])


def test_noalloc_largest_shape_fits_and_bad_args_rejected():
    # The widest shape (R + D = 16384 partial-sum columns per CTA) with a
    # full grid (one partial row per SM: N at least the SM count) fits the
    # fixed array on this device, on both reduction paths; arguments that
    # break the contract are refused before anything is enqueued.
    lib = _lib.load()
    p = _lib.AttnresParams()
    p.S, p.D, p.R, p.key_offset, p.N = 2, 8192, 8192, 0, 32768
    p.eps, p.scale, p.out_norm, p.src_ld = 2.0 ** -23, 1.0, 1, 8192
    p.src[0] = p.src[1] = 256  # non-NULL, aligned; a size query dereferences nothing
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for thr in (1, 10 ** 9):
        p.split_n_threshold = thr
        need = lib.attnres_bwd_workspace_bytes(ctypes.byref(p))
        assert sms * 16384 * 4 <= need <= _lib.NOALLOC_SCRATCH_BYTES, (thr, need)
    v = torch.zeros((2, 4, 8192), dtype=torch.bfloat16, device="cuda")
    from attention_residuals_gb300.ops import _source_view
    view = _source_view(v)
    p = make_params(view, 8192, key_offset=0, eps=2.0 ** -23, scale=1.0, out_norm=True)
    p.S = 0  # invalid shape: rejected as an argument error
    rc = lib.attnres_bwd_noalloc(ctypes.byref(p), None, None, None, None, None, None, None, None,
                                 None, ctypes.c_int64(8192), None, None, None, None, None)
    assert rc == 1
