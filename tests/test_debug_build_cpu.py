"""The bounds-checked build (-DATTNRES_DEBUG) compiles for sm_103a, exports
every symbol the release build does and says it is the checked one.  Its GPU
use: ATTNRES_DEBUG_LIB=1 python -m pytest tests -m gpu runs the whole parity
suite against it, where any store outside a call's sizes is skipped and
reported by attnres_check_device_error() (every GPU test asserts a clear
record at its end)."""
import ctypes
import os
import shutil

import pytest

from attention_residuals_gb300 import _lib
from attention_residuals_gb300.build import DEBUG_LIB_PATH, build


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="needs nvcc")
def test_debug_build_compiles_and_exports_everything():
    path = build(debug=True)
    assert path == DEBUG_LIB_PATH
    lib = ctypes.CDLL(path)
    missing = [n for n in _lib.EXPORTED if not hasattr(lib, n)]
    assert not missing, missing
    lib.attnres_debug_checks.restype = ctypes.c_int
    assert lib.attnres_debug_checks() == 1
    rel = ctypes.CDLL(build())
    rel.attnres_debug_checks.restype = ctypes.c_int
    assert rel.attnres_debug_checks() == 0
