"""Every output a call writes sits inside guard bands, and no byte of a band
may change: a canary check of each entry point's stores (the bounds a
memory checker would watch), run on the shapes that reach each kernel form.

Each output is carved out of a larger device buffer whose other bytes hold a
sentinel: GUARD bytes before and after it, and for source gradients a row
pitch wider than D (the pad columns between rows are sentinel too).  The
workspaces are exactly the size the library asks for, with the same bands.
The guarded results must also be bitwise equal to an ordinary call's.
"""
import ctypes
import math

import pytest
import torch

from attention_residuals_gb300 import (_lib, attnres_bwd, attnres_bwd_noalloc, attnres_check_device_error,
                                       attnres_fwd, attnres_partial_fwd)
from attention_residuals_gb300.ops import (_ptr, _source_view, _stream, attnres_bwd_workspace_bytes,
                                           attnres_multi_bwd_workspace_bytes, make_multi_params, make_params)
from attention_residuals_gb300.workloads import make_multi, make_random, make_selected

pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes of sentinel on each side of an output
SENTINEL = 0xA5   # every byte of a band
ROW_PAD = 64      # extra bf16 columns between gradient rows (keeps 16-byte aligned rows)


class Guarded:
    """An output of `shape` inside a sentinel-filled buffer; the last
    dimension may be padded (a strided view with sentinel columns)."""

    def __init__(self, shape, dtype, row_pad=0):
        self.shape, self.dtype = tuple(shape), dtype
        self.esz = torch.tensor([], dtype=dtype).element_size()
        self.inner = (self.shape[-1] if self.shape else 1) + row_pad
        self.rows = math.prod(self.shape[:-1]) if len(self.shape) > 1 else 1
        self.body = self.rows * self.inner * self.esz
        self.raw = torch.full((GUARD + self.body + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        core = self.raw[GUARD:GUARD + self.body].view(dtype)
        if len(self.shape) > 1:
            self.t = core.view(*self.shape[:-1], self.inner)[..., :self.shape[-1]]
        else:
            self.t = core[:self.shape[0]] if self.shape else core
        assert self.t.data_ptr() % 16 == 0

    @property
    def ld(self):
        return self.inner

    def check(self, name):
        torch.cuda.synchronize()
        head, tail = self.raw[:GUARD], self.raw[GUARD + self.body:]
        assert bool((head == SENTINEL).all()), f"{name}: a store landed before the output"
        assert bool((tail == SENTINEL).all()), f"{name}: a store landed after the output"
        width = self.shape[-1] if self.shape else 1
        if self.inner > width:
            pad = self.raw[GUARD:GUARD + self.body].view(self.rows, self.inner * self.esz)[:, width * self.esz:]
            assert bool((pad == SENTINEL).all()), f"{name}: a store landed between rows"


def _guard_ws(nbytes):
    return Guarded((max(int(nbytes), 16),), torch.uint8)


SINGLE = [
    # S, N, D, R, ko, out_norm, cluster switch: resident, ragged, streaming and cluster plans
    (9, 301, 1000, 300, 13, True, None),
    (12, 1030, 4096, 1024, 3072, False, None),
    (12, 700, 2048, 2048, 0, True, None),
    (40, 96, 8192, 8192, 0, True, "0"),
    (40, 96, 8192, 8192, 0, False, "s2"),
    (20, 130, 8192, 4096, 4096, False, "4"),
]


@pytest.mark.parametrize("S,N,D,R,ko,out_norm,cl", SINGLE)
def test_single_query_stores_stay_inside(S, N, D, R, ko, out_norm, cl, monkeypatch):
    if cl is not None:
        monkeypatch.setenv("ATTNRES_BWD_CLUSTER", cl)
    wl = make_random(S, N, D, R, key_offset=ko, out_norm=out_norm, seed=S * 7 + N)
    v, q, dy = wl.values.cuda(), wl.q.cuda(), wl.dy.cuda()
    w = wl.w_o.cuda() if out_norm else None
    f32 = torch.float32
    g = {"y": Guarded((N, D), torch.bfloat16), "alpha": Guarded((N, S), f32), "rstd": Guarded((N, S), f32),
         "logit": Guarded((N, S), f32)}
    if out_norm:
        g["o_rstd"] = Guarded((N,), f32)
        g["o_pre"] = Guarded((N, D), f32)
    fwd = attnres_fwd(v, q, w_o=w, key_offset=ko, save_o_pre=out_norm, out={k: x.t for k, x in g.items()})
    plain = attnres_fwd(v, q, w_o=w, key_offset=ko, save_o_pre=out_norm)
    for k, x in g.items():
        x.check(k)
        assert torch.equal(x.t, plain[k]), k

    # attnres_bwd: strided source gradients and an exact-size workspace
    p = make_params(_source_view(v), R, key_offset=ko, eps=wl.eps, scale=wl.scale, out_norm=out_norm)
    ws = _guard_ws(attnres_bwd_workspace_bytes(p))
    dv = Guarded((S, N, D), torch.bfloat16, row_pad=ROW_PAD)
    attnres_bwd(v, q, dy, fwd, w_o=w, key_offset=ko, dvalues=dv.t, workspace=ws.t)
    ref = attnres_bwd(v, q, dy, plain, w_o=w, key_offset=ko)
    dv.check("dvalues")
    ws.check("workspace")
    assert torch.equal(dv.t, ref["dvalues"])

    # attnres_bwd_noalloc: every output guarded
    o = {"dq": Guarded((R,), torch.bfloat16), "dq_f32": Guarded((R,), f32)}
    if out_norm:
        o["dw_o"], o["dw_o_f32"] = Guarded((D,), torch.bfloat16), Guarded((D,), f32)
    dv2 = Guarded((S, N, D), torch.bfloat16, row_pad=ROW_PAD)
    attnres_bwd_noalloc(v, q, dy, fwd, w_o=w, key_offset=ko, dvalues=dv2.t, **{k: x.t for k, x in o.items()})
    dv2.check("dvalues (no-allocation path)")
    assert torch.equal(dv2.t, ref["dvalues"])
    for k, x in o.items():
        x.check(k)
        assert torch.equal(x.t, ref[k]), k
    attnres_check_device_error()


def test_block_partial_store_stays_inside():
    wl = make_random(6, 515, 2048, 512, key_offset=1536, seed=5)
    v = wl.values.cuda()
    delta = (torch.randn((wl.N, wl.D), generator=torch.Generator().manual_seed(3)) * 0.5).to(torch.bfloat16).cuda()
    pout = Guarded((wl.N, wl.D), torch.bfloat16)
    out = attnres_partial_fwd(list(v[:-1]), v[-1], delta, wl.q.cuda(), key_offset=1536, partial_out=pout.t)
    plain = attnres_partial_fwd(list(v[:-1]), v[-1], delta, wl.q.cuda(), key_offset=1536)
    pout.check("partial_out")
    assert torch.equal(pout.t, plain["partial_new"].view(wl.N, wl.D))
    assert torch.equal(out["y"], plain["y"])


MULTI = [
    # S, N, D, R, ko, M: the resident kernels, then the general form
    (9, 257, 1024, 256, 768, 4),
    (10, 61, 4096, 1024, 3072, 16),
    (10, 50, 8192, 8192, 0, 4),
    (3, 90, 1000, 333, 13, 11),
]


def _multi_call(lib, mp, queries, dy, S, N, D, M, R, E=0, ids=None):
    f32 = torch.float32
    g = {"y": Guarded((N, M, D) if ids is not None else (M, N, D), torch.bfloat16),
         "alpha": Guarded((N, M, S), f32), "rstd": Guarded((N, S), f32), "logit": Guarded((N, M, S), f32)}
    if ids is None:
        rc = lib.attnres_multi_fwd(ctypes.byref(mp), _ptr(queries), _ptr(g["y"].t), _ptr(g["alpha"].t),
                                   _ptr(g["rstd"].t), _ptr(g["logit"].t), _stream(None))
    else:
        rc = lib.attnres_selected_fwd(ctypes.byref(mp), _ptr(queries), ctypes.c_int32(E), _ptr(ids),
                                      _ptr(g["y"].t), _ptr(g["alpha"].t), _ptr(g["rstd"].t), _ptr(g["logit"].t),
                                      _stream(None))
    _lib.check(rc, "forward")
    rows = E if ids is not None else M
    dv = Guarded((S, N, D), torch.bfloat16, row_pad=ROW_PAD)
    dptrs = (ctypes.c_void_p * S)(*[dv.t[s].data_ptr() for s in range(S)])
    dq, dq32 = Guarded((rows, R), torch.bfloat16), Guarded((rows, R), f32)
    if ids is None:
        need = attnres_multi_bwd_workspace_bytes(mp)
        ws = _guard_ws(need)
        rc = lib.attnres_multi_bwd(ctypes.byref(mp), _ptr(queries), _ptr(dy), _ptr(g["alpha"].t), _ptr(g["rstd"].t),
                                   _ptr(g["logit"].t), dptrs, ctypes.c_int64(dv.ld), _ptr(dq.t), _ptr(dq32.t),
                                   _ptr(ws.t), ctypes.c_size_t(need), _stream(None))
    else:
        need = int(lib.attnres_selected_bwd_workspace_bytes(ctypes.byref(mp), ctypes.c_int32(E)))
        ws = _guard_ws(need)
        rc = lib.attnres_selected_bwd(ctypes.byref(mp), _ptr(queries), ctypes.c_int32(E), _ptr(ids), _ptr(dy),
                                      _ptr(g["alpha"].t), _ptr(g["rstd"].t), _ptr(g["logit"].t), dptrs,
                                      ctypes.c_int64(dv.ld), _ptr(dq.t), _ptr(dq32.t), _ptr(ws.t),
                                      ctypes.c_size_t(need), _stream(None))
    _lib.check(rc, "backward")
    for k, x in g.items():
        x.check(k)
    dv.check("dvalues")
    dq.check("dq")
    dq32.check("dq_f32")
    ws.check("workspace")
    return g, dv, dq, dq32


@pytest.mark.parametrize("S,N,D,R,ko,M", MULTI)
@pytest.mark.parametrize("form", [None, "resident", "general"])
def test_multi_query_stores_stay_inside(S, N, D, R, ko, M, form, monkeypatch):
    if form is not None:
        monkeypatch.setenv("ATTNRES_MULTI_BWD", form)
    from attention_residuals_gb300 import attnres_multi_bwd, attnres_multi_fwd
    wl = make_multi(S, N, D, R, M, key_offset=ko, seed=S + M + D, src_scale=(0.5, 2.0))
    v, Q, dy = wl.values.cuda(), wl.queries.cuda(), wl.dy.cuda()
    mp = make_multi_params(_source_view(v), M, R, key_offset=ko, eps=wl.eps, scale=wl.scale, token_major=False)
    g, dv, dq, dq32 = _multi_call(_lib.load(), mp, Q, dy, S, N, D, M, R)
    fwd = attnres_multi_fwd(v, Q, key_offset=ko)
    bwd = attnres_multi_bwd(v, Q, dy, fwd, key_offset=ko)
    assert torch.equal(g["y"].t, fwd["y"]) and torch.equal(g["alpha"].t, fwd["alpha"])
    assert torch.equal(dv.t, bwd["dvalues"])
    assert torch.equal(dq.t, bwd["dq"]) and torch.equal(dq32.t, bwd["dq_f32"])
    attnres_check_device_error()


@pytest.mark.parametrize("S,N,D,R,E,K", [(8, 200, 1024, 256, 6, 3), (10, 40, 8192, 8192, 5, 16),
                                         (6, 50, 1000, 300, 7, 5)])
def test_selected_query_stores_stay_inside(S, N, D, R, E, K):
    from attention_residuals_gb300 import attnres_selected_bwd, attnres_selected_fwd
    wl = make_selected(S, N, D, R, E, K, seed=S + E + K)
    v, bank, ids, dy = wl.values.cuda(), wl.bank.cuda(), wl.ids.cuda(), wl.dy.cuda()
    mp = make_multi_params(_source_view(v), K, R, key_offset=wl.key_offset, eps=wl.eps, scale=wl.scale,
                           token_major=True)
    g, dv, db, db32 = _multi_call(_lib.load(), mp, bank, dy, S, N, D, K, R, E=E, ids=ids)
    fwd = attnres_selected_fwd(v, bank, ids, key_offset=wl.key_offset)
    bwd = attnres_selected_bwd(v, bank, ids, dy, fwd, key_offset=wl.key_offset)
    assert torch.equal(g["y"].t, fwd["y"].view(N, K, D))
    assert torch.equal(dv.t, bwd["dvalues"])
    assert torch.equal(db.t, bwd["dbank"]) and torch.equal(db32.t, bwd["dbank_f32"])
    attnres_check_device_error()


def test_debug_build_flag_matches_the_loaded_library():
    import os
    lib = _lib.load()
    want = 1 if os.environ.get("ATTNRES_DEBUG_LIB") == "1" else 0
    assert lib.attnres_debug_checks() == want
