"""C-ABI checks that need no GPU: the library builds, loads and exports every
function the headers in include/ declare, and arguments that break the
contract are rejected before anything is planned or launched."""
import ctypes
import os
import re

import pytest
import torch

from attention_residuals_gb300 import _lib
from attention_residuals_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attnres.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(attnres_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(_lib.EXPORTED) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_params_struct_layout_matches_header():
    # offsets follow the C struct: 4 x int32, int64, 2 x float, 2 x int32, int64, pointer array
    P = _lib.AttnresParams
    assert P.N.offset == 16 and P.eps.offset == 24 and P.src_ld.offset == 40 and P.src.offset == 48
    assert ctypes.sizeof(P) == 48 + 8 * _lib.MAX_S


def test_status_strings(lib):
    for code in range(0, 8):
        s = lib.attnres_status_string(code)
        assert s and len(s) > 1


def _params(S=4, N=8, D=64, R=64, ko=0, ld=None, out_norm=0, fake=0x100000):
    p = _lib.AttnresParams()
    p.S, p.D, p.R, p.key_offset, p.N = S, D, R, ko, N
    p.eps, p.scale, p.out_norm, p.split_n_threshold = 2.0 ** -23, 1.0, out_norm, 0
    p.src_ld = D if ld is None else ld
    for s in range(min(max(S, 0), _lib.MAX_S)):
        p.src[s] = fake + s * 0x10000
    return p


BAD = [
    (dict(S=0), 1), (dict(S=129), 1), (dict(D=4), 1), (dict(D=12, R=12), 2),
    (dict(D=16384, R=16), 1), (dict(R=0), 1), (dict(R=65), 1), (dict(R=32, ko=33), 1),
    (dict(ko=-1), 1), (dict(N=-1), 1), (dict(out_norm=2), 1), (dict(ld=32), 1),
    (dict(ld=68), 2), (dict(fake=0x100002), 2),
]


@pytest.mark.parametrize("kw,code", BAD)
def test_forward_rejects_bad_shapes_before_launch(lib, kw, code):
    p = _params(**kw)
    fake = ctypes.c_void_p(0x200000)
    rc = lib.attnres_fwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", BAD)
def test_backward_rejects_bad_shapes_before_launch(lib, kw, code):
    p = _params(**kw)
    fake = ctypes.c_void_p(0x200000)
    d = (ctypes.c_void_p * 4)(*[0x300000 + i * 0x10000 for i in range(4)])
    rc = lib.attnres_bwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, d,
                         ctypes.c_int64(64), fake, None, None, None, fake, ctypes.c_size_t(1 << 20), None)
    assert rc == code
    assert lib.attnres_bwd_workspace_bytes(ctypes.byref(p)) == 0


def test_nan_eps_and_scale_rejected(lib):
    fake = ctypes.c_void_p(0x200000)
    for field, val in (("eps", float("nan")), ("eps", -1.0), ("scale", float("inf"))):
        p = _params()
        setattr(p, field, val)
        rc = lib.attnres_fwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, None)
        assert rc == 1


def test_missing_pointers_rejected(lib):
    p = _params(out_norm=1)
    fake = ctypes.c_void_p(0x200000)
    # out_norm without w_o / o_rstd / o_pre
    assert lib.attnres_fwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, None) == 1
    p = _params()
    assert lib.attnres_fwd(ctypes.byref(p), None, None, fake, fake, fake, fake, None, None, None) == 1
    # misaligned output row pointer
    odd = ctypes.c_void_p(0x200008)
    assert lib.attnres_fwd(ctypes.byref(p), fake, None, odd, fake, fake, fake, None, None, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only used without a GPU")
def test_backward_rejects_aliasing_outputs(lib):
    p = _params(S=2, N=8, D=64)
    fake = ctypes.c_void_p(0x200000)
    # dvalues of source 1 overlaps source 0's rows
    d = (ctypes.c_void_p * 2)(0x100000 + 64, 0x500000)
    rc = lib.attnres_bwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, d,
                         ctypes.c_int64(64), fake, None, None, None, fake, ctypes.c_size_t(1 << 20), None)
    assert rc == 1
    d = (ctypes.c_void_p * 2)(0x500000, 0x500000 + 128)  # the two outputs overlap
    rc = lib.attnres_bwd(ctypes.byref(p), fake, None, fake, fake, fake, fake, None, None, d,
                         ctypes.c_int64(64), fake, None, None, None, fake, ctypes.c_size_t(1 << 20), None)
    assert rc == 1


def test_binding_refuses_cpu_tensors():
    from attention_residuals_gb300 import attnres_fwd
    v = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    q = torch.zeros((64,), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        attnres_fwd(v, q)


# --------------------------------------------------------------- multi-query
def test_multi_params_struct_layout_matches_header():
    MP = _lib.AttnresMultiParams
    base = ctypes.sizeof(_lib.AttnresParams)
    assert MP.M.offset == base and MP.out_ld_m.offset == base + 8 and MP.out_ld_n.offset == base + 16
    assert ctypes.sizeof(MP) == base + 24


def _mparams(M=2, ld_m=None, ld_n=None, **kw):
    mp = _lib.AttnresMultiParams()
    mp.base = _params(**kw)
    mp.M = M
    N, D = mp.base.N, mp.base.D
    mp.out_ld_m = N * D if ld_m is None else ld_m
    mp.out_ld_n = D if ld_n is None else ld_n
    return mp


MULTI_BAD = BAD + [
    (dict(M=0), 1), (dict(M=17), 1), (dict(out_norm=1), 3), (dict(ld_m=4), 2), (dict(ld_n=-8), 1),
]


@pytest.mark.parametrize("kw,code", MULTI_BAD)
def test_multi_forward_rejects_bad_shapes_before_launch(lib, kw, code):
    mp = _mparams(**kw)
    fake = ctypes.c_void_p(0x200000)
    rc = lib.attnres_multi_fwd(ctypes.byref(mp), fake, fake, fake, fake, fake, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", MULTI_BAD)
def test_multi_backward_rejects_bad_shapes_before_launch(lib, kw, code):
    mp = _mparams(**kw)
    fake = ctypes.c_void_p(0x200000)
    d = (ctypes.c_void_p * 4)(*[0x300000 + i * 0x10000 for i in range(4)])
    rc = lib.attnres_multi_bwd(ctypes.byref(mp), fake, fake, fake, fake, fake, d, ctypes.c_int64(64),
                               fake, None, fake, ctypes.c_size_t(1 << 20), None)
    assert rc == code
    assert lib.attnres_multi_bwd_workspace_bytes(ctypes.byref(mp)) == 0


def test_multi_missing_or_misaligned_pointers_rejected(lib):
    mp = _mparams()
    fake = ctypes.c_void_p(0x200000)
    assert lib.attnres_multi_fwd(ctypes.byref(mp), None, fake, fake, fake, fake, None) == 1
    assert lib.attnres_multi_fwd(ctypes.byref(mp), fake, ctypes.c_void_p(0x200008), fake, fake, fake,
                                 None) == 2
    d = (ctypes.c_void_p * 4)(*[0x300000 + i * 0x10000 for i in range(4)])
    assert lib.attnres_multi_bwd(ctypes.byref(mp), fake, fake, fake, fake, fake, d, ctypes.c_int64(64),
                                 None, None, fake, ctypes.c_size_t(1 << 20), None) == 1


# ------------------------------------------------------------ selected-query
@pytest.mark.parametrize("kw,code", MULTI_BAD)
def test_selected_rejects_bad_shapes_before_launch(lib, kw, code):
    mp = _mparams(**kw)
    fake = ctypes.c_void_p(0x200000)
    assert lib.attnres_selected_fwd(ctypes.byref(mp), fake, 4, fake, fake, fake, fake, fake, None) == code
    d = (ctypes.c_void_p * 4)(*[0x300000 + i * 0x10000 for i in range(4)])
    rc = lib.attnres_selected_bwd(ctypes.byref(mp), fake, 4, fake, fake, fake, fake, fake, d,
                                  ctypes.c_int64(64), fake, None, fake, ctypes.c_size_t(1 << 20), None)
    assert rc == code
    assert lib.attnres_selected_bwd_workspace_bytes(ctypes.byref(mp), 4) == 0


def test_selected_bank_and_ids_checked(lib):
    mp = _mparams()
    fake = ctypes.c_void_p(0x200000)
    # no bank rows, missing ids, misaligned ids
    assert lib.attnres_selected_fwd(ctypes.byref(mp), fake, 0, fake, fake, fake, fake, fake, None) == 1
    assert lib.attnres_selected_fwd(ctypes.byref(mp), fake, 4, None, fake, fake, fake, fake, None) == 1
    assert lib.attnres_selected_fwd(ctypes.byref(mp), fake, 4, ctypes.c_void_p(0x200004), fake, fake, fake,
                                    fake, None) == 2
    assert lib.attnres_selected_bwd_workspace_bytes(ctypes.byref(mp), 0) == 0
