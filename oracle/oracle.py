"""ctypes wrapper around the FP64 C oracle (test infrastructure only).

The oracle follows "Fast Attention Residuals", section "Equation" (key slice,
key RMS with eps inside the square root, scaled dot with the query, softmax
over sources, weighted full-width sum), plus the optional output RMSNorm that
"[Perf] Parallelize AttnRes long-sequence reduction" (Summary) saves o_rstd
for, and the chain-rule backward.  All arithmetic happens in the C file in
IEEE double; this module only converts arrays and calls it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attnres_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_attnres.so")
_lock = threading.Lock()
_lib = None


def oracle_library_path() -> str:
    return _LIB


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", _SRC, "-o", tmp,
             "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            for name, ip in (("attnres_oracle_bf16", ctypes.c_void_p),
                             ("attnres_oracle_f64", ctypes.c_void_p)):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                               ip, ip, ip, ip,
                               dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as_bits(x):
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bit patterns."""
    if x is None:
        return None
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be torch.bfloat16 or uint16 bit patterns")
    return a


def attnres_oracle(values, q, *, eps=2.0 ** -23, scale=1.0, w_o=None, dy=None,
                   key_offset=None, nthreads=None, precision="bf16", want_dvalues=True):
    """Run the oracle.

    values: packed sources [S, N, D] (bf16 tensor / uint16 bits, or float64 when
            precision == "f64").  q: [R].  w_o: [D] or None (no output norm).
    dy: [N, D] upstream gradient, or None for forward only.
    key_offset: first channel of the key slice (default D - R, the page's
            "final R coordinates").
    Returns a dict of float64 numpy arrays: y [N,D], alpha/rstd/logit [N,S],
    o_rstd [N] (1.0 without out-norm), and when dy is given dvalues [S,N,D],
    dq [R], dw_o [D] (zeros without out-norm).
    """
    lib = _load()
    if precision == "bf16":
        v = _as_bits(values)
        qq = _as_bits(q)
        ww = _as_bits(w_o)
        gg = _as_bits(dy)
        fn = lib.attnres_oracle_bf16
    elif precision == "f64":
        v = np.ascontiguousarray(values, dtype=np.float64)
        qq = np.ascontiguousarray(q, dtype=np.float64)
        ww = None if w_o is None else np.ascontiguousarray(w_o, dtype=np.float64)
        gg = None if dy is None else np.ascontiguousarray(dy, dtype=np.float64)
        fn = lib.attnres_oracle_f64
    else:
        raise ValueError(precision)
    if v.ndim != 3:
        raise ValueError("values must be packed [S, N, D]")
    S, N, D = v.shape
    R = int(qq.shape[0])
    ko = D - R if key_offset is None else int(key_offset)
    out_norm = 1 if ww is not None else 0
    if gg is not None and gg.shape != (N, D):
        raise ValueError("dy must be [N, D]")
    if nthreads is None:
        nthreads = max(1, min(os.cpu_count() or 1, 64, N if N > 0 else 1))
    y = np.empty((N, D), np.float64)
    alpha = np.empty((N, S), np.float64)
    rstd = np.empty((N, S), np.float64)
    logit = np.empty((N, S), np.float64)
    o_rstd = np.empty((N,), np.float64)
    dsrc = np.empty((S, N, D), np.float64) if (gg is not None and want_dvalues) else None
    dq = np.zeros((R,), np.float64) if gg is not None else None
    dw = np.zeros((D,), np.float64) if gg is not None else None
    rc = fn(S, N, D, R, ko, float(eps), float(scale), out_norm, _ptr(v), _ptr(qq), _ptr(ww),
            _ptr(gg), _dptr(y), _dptr(alpha), _dptr(rstd), _dptr(logit), _dptr(o_rstd),
            _dptr(dsrc), _dptr(dq), _dptr(dw), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (S/N/D/R/key_offset or missing w_o)")
    out = {"y": y, "alpha": alpha, "rstd": rstd, "logit": logit, "o_rstd": o_rstd}
    if gg is not None:
        out["dq"] = dq
        out["dw_o"] = dw
        if dsrc is not None:
            out["dvalues"] = dsrc
    return out
