"""Build libggq.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel into ``_build/`` and linked into
``gguf_block_quantized_q8_gb300/libggq.so``.  No cmake, one -gencode.
"""
from __future__ import annotations

import concurrent.futures as cf
import contextlib
import os
import resource
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libggq.so")

SOURCES = ["api.cu", "gemv.cu", "gemv_rows.cu", "gemv_stream.cu", "gemv_noalloc.cu", "smallm.cu", "dequant.cu", "prefill.cu",
           "gguf_loader.cpp"]
HEADERS = ["ggq_internal.h", "ptx.cuh", "gemv_tile.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found")
    return found


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "ggq.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, verbose: bool) -> str:
    nvcc = _nvcc()
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", "-c", src, "-o", obj]
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


@contextlib.contextmanager
def _compiler_stack():
    """Let the compilers started meanwhile grow their stack to 1 GB (or the hard
    limit): the device compiler recurses deeply over the largest kernels, and
    with line info their build needed more than the usual 8 MB on aarch64."""
    soft, hard = resource.getrlimit(resource.RLIMIT_STACK)
    want = (1 << 30) if hard == resource.RLIM_INFINITY else min(hard, 1 << 30)
    raised = soft != resource.RLIM_INFINITY and soft < want
    if raised:
        try:
            resource.setrlimit(resource.RLIMIT_STACK, (want, hard))
        except (ValueError, OSError):
            raised = False
    try:
        yield
    finally:
        if raised:
            resource.setrlimit(resource.RLIMIT_STACK, (soft, hard))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libggq.so."""
    if not force and not is_stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with _compiler_stack(), cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
