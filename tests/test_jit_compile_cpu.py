"""The sources embedded for run-time compilation compile with NVRTC for
sm_103a (no GPU needed to compile), for the long-sequence forward's plan
shape and a multi-query one, without register spills.  A header change that
broke this would otherwise only show as a silent fall-back to the
precompiled kernels on a GPU machine."""
import ctypes
import os
import re
import tempfile

import pytest

from attention_residuals_gb300 import build


def _nvrtc():
    for name in ("libnvrtc.so.13", os.path.join(build._cuda_lib_dir(), "libnvrtc.so")):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("NVRTC is not available here")


def _embedded():
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "attnres_jit_sources.inc")
        build._write_jit_sources(path)
        text = open(path).read()
    return dict(re.findall(r'\{"([^"]+)", R"ATTNRES_SRC\((.*?)\)ATTNRES_SRC"\}', text, flags=re.S))


INT_TYPES = ("#pragma once\ntypedef unsigned char uint8_t; typedef unsigned short uint16_t; "
             "typedef unsigned int uint32_t; typedef unsigned long long uint64_t; typedef signed char int8_t; "
             "typedef short int16_t; typedef int int32_t; typedef long long int64_t; typedef unsigned long size_t; "
             "typedef unsigned long uintptr_t; typedef long ptrdiff_t;\n")


@pytest.mark.parametrize("header,expr", [
    ("attnres_fwd_kernel.cuh", "attnres::jit::attnres_fwd_kernel<2, true, false, 1, 10, 5, 5, 2>"),
    ("attnres_multi_fwd_kernel.cuh", "attnres::jit::attnres_multi_fwd_kernel<2, 2, true, 2, 10, 5, 5, 2>"),
])
def test_embedded_forward_compiles_without_spills(header, expr):
    lib = _nvrtc()
    files = _embedded()
    # the same stand-ins for toolkit headers the library gives NVRTC
    files.update({"cstdint": INT_TYPES, "stdint.h": INT_TYPES, "cstddef": INT_TYPES, "stddef.h": INT_TYPES,
                  "cfloat": "#pragma once\n#define FLT_MAX 3.402823466e+38F\n", "cuda_runtime.h": "#pragma once\n"})
    names = list(files)
    arr = ctypes.c_char_p * len(names)
    prog = ctypes.c_void_p()
    src = f'#define ATTNRES_FWD_NS jit\n#include "{header}"\n'.encode()
    assert lib.nvrtcCreateProgram(ctypes.byref(prog), src, b"probe.cu", len(names),
                                  arr(*[files[n].encode() for n in names]), arr(*[n.encode() for n in names])) == 0
    assert lib.nvrtcAddNameExpression(prog, expr.encode()) == 0
    opts = [b"-arch=sm_103a", b"-std=c++17", b"-default-device", b"--ptxas-options=-v"]
    rc = lib.nvrtcCompileProgram(prog, len(opts), (ctypes.c_char_p * len(opts))(*opts))
    size = ctypes.c_size_t()
    lib.nvrtcGetProgramLogSize(prog, ctypes.byref(size))
    buf = ctypes.create_string_buffer(size.value)
    lib.nvrtcGetProgramLog(prog, buf)
    log = buf.value.decode(errors="replace")
    lib.nvrtcDestroyProgram(ctypes.byref(prog))
    assert rc == 0, log
    spills = [int(x) for x in re.findall(r"(\d+) bytes spill stores", log)]
    assert spills and max(spills) == 0, log
