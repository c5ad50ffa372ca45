"""Build the CUDA library in place: one nvcc per translation unit (in parallel), one link.

Produces ``libfa_gb300.so`` next to this file, compiled for sm_103a only.  Run as
``python -m exact_tiled_attention_07_gb300.build`` or through ``__graft_entry__.build()``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libfa_gb300_debug.so")

SOURCES = ["api.cu", "simt.cu", "fwd_tc.cu", "bwd_tc.cu", "noalloc.cu", "decode.cu", "decode_tc.cu", "fp8.cu", "selftest.cu",
           "pipeline.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _compile(nvcc: str, src: str, verbose: bool, build_dir: str = BUILD_DIR, extra=()) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v", "-c", os.path.join(CSRC, src),
           "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(build_dir, os.path.splitext(src)[0] + ".ptxas.log")
    with open(log, "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
    if verbose:
        print(f"[build] {src} ok")
    return obj


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link the shared library; returns its path.

    debug=True builds ``libfa_gb300_debug.so`` instead, with FA_DEBUG defined: the kernels then
    check their work-item, tile and row indices and record a device error on a failed check.
    """
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    extra = ["-DFA_DEBUG=1"] if debug else []
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "fa.h"))
    if not force and os.path.exists(lib_path):
        newest = max(os.path.getmtime(p) for p in srcs + headers)
        if os.path.getmtime(lib_path) >= newest:
            return lib_path
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose, build_dir, extra), SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, lib_path)
    if verbose:
        print(f"[build] linked {lib_path}")
    return lib_path


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)
