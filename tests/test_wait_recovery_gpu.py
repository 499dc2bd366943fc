"""The bounded-wait recovery path, forced on the GPU without a fault.

Every wait on a shared-memory barrier in the kernels gives up after a time
limit, records where, and lets the kernel run to its end without waiting
again; attnres_check_device_error() reports it.  The test hook of
include/attnres_testing.h makes that happen on purpose: CTA 0's producer
never issues one chunk fill (every earlier fill is issued and consumed, so no
copy is left in flight) and the wait limit is 1 ms.  The launch must finish
quickly, the error must be reported once, and the next ordinary launch must
be bitwise equal to one made before the failure (and match the oracle).
"""
import ctypes
import time

import pytest
import torch

from attention_residuals_gb300 import _lib, attnres_check_device_error, attnres_fwd
from attention_residuals_gb300._lib import AttnresError
from attention_residuals_gb300.ops import _ptr, _source_view, _stream, make_params
from attention_residuals_gb300.workloads import make_random
from oracle import attnres_oracle
from parity_utils import check_forward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("withhold", [1, 2])
@pytest.mark.parametrize("out_norm", [False, True])
def test_withheld_fill_times_out_and_the_next_launch_is_clean(withhold, out_norm):
    wl = make_random(8, 900, 1024, out_norm=out_norm, seed=91 + withhold)
    v, q = wl.values.cuda(), wl.q.cuda()
    w = wl.w_o.cuda() if out_norm else None
    before = attnres_fwd(v, q, w_o=w, key_offset=0)
    torch.cuda.synchronize()
    attnres_check_device_error()

    # the forced failure
    lib = _lib.load()
    p = make_params(_source_view(v), wl.R, key_offset=0, eps=wl.eps, scale=wl.scale, out_norm=out_norm)
    N, S, D = wl.N, wl.S, wl.D
    f32 = dict(dtype=torch.float32, device="cuda")
    y = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    alpha, rstd, logit = (torch.empty((N, S), **f32) for _ in range(3))
    o_rstd = torch.empty((N,), **f32) if out_norm else None
    t0 = time.perf_counter()
    rc = lib.attnres_fwd_withhold_for_test(ctypes.byref(p), _ptr(q), _ptr(w), _ptr(y), _ptr(alpha), _ptr(rstd),
                                           _ptr(logit), _ptr(o_rstd), ctypes.c_int64(withhold),
                                           ctypes.c_uint32(1000), _stream(None))
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, elapsed  # the 1 ms limit, not the default two seconds
    with pytest.raises(AttnresError) as e:
        attnres_check_device_error()
    assert e.value.name == "ATTNRES_ERR_DEVICE"
    attnres_check_device_error()  # reported once, then cleared

    # the next ordinary launch: the same bits as before the failure, and the oracle's values
    after = attnres_fwd(v, q, w_o=w, key_offset=0)
    torch.cuda.synchronize()
    attnres_check_device_error()
    for key in ("y", "alpha", "rstd", "logit") + (("o_rstd",) if out_norm else ()):
        assert torch.equal(before[key], after[key]), key
    ref = attnres_oracle(wl.values, wl.q, w_o=wl.w_o, key_offset=0)
    check_forward(after, ref, out_norm=out_norm, tag="after the forced timeout")


def test_hook_rejects_bad_arguments():
    lib = _lib.load()
    v = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    p = make_params(_source_view(v), 64, key_offset=0, eps=2.0 ** -23, scale=1.0, out_norm=False)
    for withhold, wait_us in ((0, 1000), (1, 0), (1, 2_000_000)):
        rc = lib.attnres_fwd_withhold_for_test(ctypes.byref(p), None, None, None, None, None, None, None,
                                               ctypes.c_int64(withhold), ctypes.c_uint32(wait_us), _stream(None))
        assert rc == 1  # ATTNRES_ERR_INVALID_ARG, nothing launched
