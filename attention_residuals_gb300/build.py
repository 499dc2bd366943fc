"""Build the sm_103a AttnRes shared library in-tree with nvcc.

    python -m attention_residuals_gb300.build

compiles csrc/*.cu in parallel (one -gencode for compute_103a/sm_103a) and
links attention_residuals_gb300/libattnres_gb300.so against the shared CUDA
runtime.  No PyTorch headers or libraries are involved.

    python -m attention_residuals_gb300.build --debug

writes libattnres_gb300_debug.so instead, compiled with -DATTNRES_DEBUG:
every output store is checked against the call's sizes and a bad one is
skipped and reported by attnres_check_device_error().  ATTNRES_DEBUG_LIB=1
makes the Python binding load it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libattnres_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
DEBUG_LIB_NAME = "libattnres_gb300_debug.so"
DEBUG_LIB_PATH = os.path.join(PKG, DEBUG_LIB_NAME)
SOURCES = ["attnres_fwd.cu", "attnres_bwd.cu", "attnres_bwd_norm.cu", "attnres_bwd_opre.cu", "attnres_bwd_cluster.cu",
           "attnres_multi_fwd.cu", "attnres_multi_fwd_mma.cu", "attnres_multi_bwd.cu", "attnres_multi_general.cu", "attnres_multi_grad_mma.cu", "attnres_api.cu", "attnres_host.cu", "attnres_jit.cu"]
# Sources the library compiles again at run time for exact plan shapes
# (attnres_jit.cu): embedded as string literals under their include names.
JIT_FILES = [("attnres_fwd_kernel.cuh", CSRC), ("attnres_multi_fwd_kernel.cuh", CSRC), ("device_utils.cuh", CSRC),
             ("kernels.cuh", CSRC), ("attnres.h", INCLUDE)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dir() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(cuda, sub)
        if os.path.isdir(d):
            return d
    return os.path.join(cuda, "lib64")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return any(os.path.getmtime(d) > t for d in deps if os.path.isfile(d))


def _write_jit_sources(path: str) -> None:
    delim = "ATTNRES_SRC"
    parts = ["struct JitFile { const char* name; const char* text; };",
             "static const JitFile kJitFiles[] = {"]
    for name, folder in JIT_FILES:
        with open(os.path.join(folder, name)) as f:
            text = f.read()
        if f"){delim}\"" in text:
            raise RuntimeError(f"{name} contains the raw-string delimiter")
        parts.append(f'    {{"{name}", R"{delim}({text}){delim}"}},')
    parts.append("};")
    with open(path, "w") as f:
        f.write("\n".join(parts) + "\n")


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    lib_path, lib_name = (DEBUG_LIB_PATH, DEBUG_LIB_NAME) if debug else (LIB_PATH, LIB_NAME)
    if not force and not _stale(lib_path):
        return lib_path
    nvcc = _nvcc()
    tmp = tempfile.mkdtemp(prefix="attnres_build_")
    libdir = _cuda_lib_dir()
    flags = ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "-I", CSRC, "-I", tmp, f'-DATTNRES_CUDA_LIBDIR="{libdir}"'] + (["-DATTNRES_DEBUG"] if debug else []) + list(extra_flags or [])
    if verbose:
        flags += ["-Xptxas", "-v"]
    try:
        _write_jit_sources(os.path.join(tmp, "attnres_jit_sources.inc"))
        def compile_one(src):
            obj = os.path.join(tmp, src.replace(".cu", ".o"))
            cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                sys.stderr.write(r.stderr)
            return obj

        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        out_tmp = os.path.join(tmp, lib_name)
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", out_tmp,
               "-Xlinker", f"-rpath={libdir}", "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        shutil.move(out_tmp, lib_path + ".tmp")
        os.replace(lib_path + ".tmp", lib_path)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
