"""ctypes view of the C ABI declared in include/attnres.h.

Argument marshalling only: every step of the operator runs in the CUDA
library.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

MAX_S = 128
MAX_D = 8192
MAX_M = 16
NOALLOC_SCRATCH_BYTES = 16 << 20
DEFAULT_SPLIT_N = 1

STATUS = {
    0: "ATTNRES_OK",
    1: "ATTNRES_ERR_INVALID_ARG",
    2: "ATTNRES_ERR_ALIGNMENT",
    3: "ATTNRES_ERR_UNSUPPORTED",
    4: "ATTNRES_ERR_WORKSPACE",
    5: "ATTNRES_ERR_CUDA",
    6: "ATTNRES_ERR_DEVICE",
}

EXPORTED = [
    "attnres_fwd",
    "attnres_bwd",
    "attnres_bwd_noalloc",
    "attnres_bwd_workspace_bytes",
    "attnres_check_device_error",
    "attnres_jit_kernel_count",
    "attnres_debug_checks",
    "attnres_multi_fwd_tensor_cores",
    "attnres_status_string",
    "attnres_plan_info",
    "attnres_multi_fwd",
    "attnres_multi_bwd",
    "attnres_multi_bwd_workspace_bytes",
    "attnres_multi_plan_info",
    "attnres_selected_fwd",
    "attnres_selected_bwd",
    "attnres_selected_bwd_workspace_bytes",
    "attnres_fwd_partial",
    "attnres_bwd_partial",
    "attnres_step_host",
    "attnres_step_host_workspace_bytes",
    "attnres_fwd_withhold_for_test",
]


class AttnresParams(ctypes.Structure):
    _fields_ = [
        ("S", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("R", ctypes.c_int32),
        ("key_offset", ctypes.c_int32),
        ("N", ctypes.c_int64),
        ("eps", ctypes.c_float),
        ("scale", ctypes.c_float),
        ("out_norm", ctypes.c_int32),
        ("split_n_threshold", ctypes.c_int32),
        ("src_ld", ctypes.c_int64),
        ("src", ctypes.c_void_p * MAX_S),
    ]


class AttnresMultiParams(ctypes.Structure):
    _fields_ = [
        ("base", AttnresParams),
        ("M", ctypes.c_int32),
        ("out_ld_m", ctypes.c_int64),
        ("out_ld_n", ctypes.c_int64),
    ]


class _Partial:
    """A library handle that lacks some entry points (an explicitly loaded
    older build): declaring a missing function is a no-op, calling it fails."""

    def __init__(self, lib, missing):
        self._lib = lib
        self._missing = set(missing)

    def __getattr__(self, name):
        if name in self._missing:
            return _Missing(name)
        return getattr(self._lib, name)


class _Missing:
    def __init__(self, name):
        self.name = name
        self.argtypes = self.restype = None

    def __call__(self, *args):
        raise RuntimeError(f"this build of the library has no {self.name}")


class AttnresError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        msg = _status_string(code)
        super().__init__(f"{where}: {self.name}: {msg}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """The release build, or with ATTNRES_DEBUG_LIB=1 in the environment the
    bounds-checked build (python -m attention_residuals_gb300.build --debug)."""
    from .build import DEBUG_LIB_PATH, LIB_PATH
    return DEBUG_LIB_PATH if os.environ.get("ATTNRES_DEBUG_LIB") == "1" else LIB_PATH


def load(path: str | None = None):
    """Load the library (no build, no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"AttnRes CUDA library not found at {p}; build it with "
                "`python -m attention_residuals_gb300.build` (needs nvcc for sm_103a)")
        lib = ctypes.CDLL(p)
        missing = [n for n in EXPORTED if not hasattr(lib, n)]
        if missing and path is None:
            raise RuntimeError(f"AttnRes CUDA library at {p} lacks {missing}; rebuild it")
        if missing:  # an explicitly given older build: declare what it has
            lib = _Partial(lib, missing)
        P = ctypes.POINTER(AttnresParams)
        vp, fp, i64, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        lib.attnres_fwd.restype = ctypes.c_int
        lib.attnres_fwd.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, vp, vp]
        lib.attnres_bwd_workspace_bytes.restype = sz
        lib.attnres_bwd_workspace_bytes.argtypes = [P]
        lib.attnres_bwd.restype = ctypes.c_int
        lib.attnres_bwd.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, vp,
                                    ctypes.POINTER(ctypes.c_void_p), i64, vp, fp, vp, fp, vp, sz, vp]
        lib.attnres_bwd_noalloc.restype = ctypes.c_int
        lib.attnres_bwd_noalloc.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, fp,
                                            ctypes.POINTER(ctypes.c_void_p), i64, vp, fp, vp, fp, vp]
        lib.attnres_fwd_withhold_for_test.restype = ctypes.c_int
        lib.attnres_fwd_withhold_for_test.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, i64, ctypes.c_uint32, vp]
        lib.attnres_check_device_error.restype = ctypes.c_int
        lib.attnres_check_device_error.argtypes = []
        lib.attnres_jit_kernel_count.restype = ctypes.c_int
        lib.attnres_jit_kernel_count.argtypes = []
        lib.attnres_debug_checks.restype = ctypes.c_int
        lib.attnres_debug_checks.argtypes = []
        lib.attnres_multi_fwd_tensor_cores.restype = ctypes.c_int
        lib.attnres_status_string.restype = ctypes.c_char_p
        lib.attnres_status_string.argtypes = [ctypes.c_int]
        lib.attnres_plan_info.restype = ctypes.c_int
        lib.attnres_plan_info.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
        MP = ctypes.POINTER(AttnresMultiParams)
        lib.attnres_multi_fwd_tensor_cores.argtypes = [MP, ctypes.c_int32]
        lib.attnres_multi_fwd.restype = ctypes.c_int
        lib.attnres_multi_fwd.argtypes = [MP, vp, vp, fp, fp, fp, vp]
        lib.attnres_multi_bwd_workspace_bytes.restype = sz
        lib.attnres_multi_bwd_workspace_bytes.argtypes = [MP]
        lib.attnres_multi_bwd.restype = ctypes.c_int
        lib.attnres_multi_bwd.argtypes = [MP, vp, vp, fp, fp, fp, ctypes.POINTER(ctypes.c_void_p), i64,
                                          vp, fp, vp, sz, vp]
        lib.attnres_multi_plan_info.restype = ctypes.c_int
        lib.attnres_multi_plan_info.argtypes = [MP, ctypes.POINTER(ctypes.c_int64)]
        lib.attnres_fwd_partial.restype = ctypes.c_int
        lib.attnres_fwd_partial.argtypes = [P, vp, vp, vp, i64, vp, i64, vp, fp, fp, fp, fp, vp, vp]
        lib.attnres_bwd_partial.restype = ctypes.c_int
        lib.attnres_bwd_partial.argtypes = [P, vp, vp, vp, fp, fp, fp, fp, vp, vp, i64,
                                            ctypes.POINTER(ctypes.c_void_p), i64, vp, fp, vp, fp, vp, sz, vp]
        lib.attnres_step_host_workspace_bytes.restype = sz
        lib.attnres_step_host_workspace_bytes.argtypes = [P, i64]
        lib.attnres_step_host.restype = ctypes.c_int
        lib.attnres_step_host.argtypes = [P, vp, vp, vp, i64, vp, i64, ctypes.POINTER(ctypes.c_void_p), i64, vp,
                                          fp, vp, fp, i64, vp, sz, ctypes.POINTER(ctypes.c_void_p)]
        i32 = ctypes.c_int32
        lib.attnres_selected_fwd.restype = ctypes.c_int
        lib.attnres_selected_fwd.argtypes = [MP, vp, i32, vp, vp, fp, fp, fp, vp]
        lib.attnres_selected_bwd_workspace_bytes.restype = sz
        lib.attnres_selected_bwd_workspace_bytes.argtypes = [MP, i32]
        lib.attnres_selected_bwd.restype = ctypes.c_int
        lib.attnres_selected_bwd.argtypes = [MP, vp, i32, vp, vp, fp, fp, fp, ctypes.POINTER(ctypes.c_void_p),
                                             i64, vp, fp, vp, sz, vp]
        _lib = lib
        return lib


def _status_string(code: int) -> str:
    try:
        return load().attnres_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return STATUS.get(code, "unknown")


def check(code: int, where: str):
    if code != 0:
        raise AttnresError(code, where)
