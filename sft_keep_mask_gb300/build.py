"""Build the fused LM-head library (sm_103a) in-tree.

Compiles every ``csrc/*.cu`` translation unit with nvcc in parallel and links
them into ``sft_keep_mask_gb300/_lib/liblmhead.so`` (CUDA runtime linked
statically; the driver API is reached through the runtime's entry-point
query, so no libcuda link is needed).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "liblmhead.so")
# The same sources with -DLMHEAD_DEBUG: device-side index checks that report
# LMHEAD_EBOUNDS instead of touching memory outside an array.
DEBUG_BUILD = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(LIBDIR, "liblmhead_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(ROOT, "include", "lmhead.h")]


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library; with
    `debug` the LMHEAD_DEBUG variant (liblmhead_debug.so)."""
    build_dir = DEBUG_BUILD if debug else BUILD
    lib_path = DEBUG_LIB if debug else LIB
    if debug:
        extra_flags = list(extra_flags) + ["-DLMHEAD_DEBUG"]
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    nvcc = _nvcc()
    newest_dep = max(os.path.getmtime(p) for p in _deps())
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest_dep:
        return lib_path

    def compile_one(src):
        obj = os.path.join(build_dir, src[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


EXAMPLE_SRC = os.path.join(PKG, "examples", "lmhead_c_example.c")
EXAMPLE_BIN = os.path.join(BUILD, "lmhead_c_example")


def build_example() -> str:
    """Compile the plain-C example caller of the C ABI against liblmhead.so."""
    lib = build()
    cuda_home = os.path.dirname(os.path.dirname(_nvcc()))
    cmd = ["gcc", "-O2", "-std=c11", EXAMPLE_SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda_home, "include"), "-L", LIBDIR, "-llmhead",
           f"-Wl,-rpath,{LIBDIR}", "-L", os.path.join(cuda_home, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{os.path.join(cuda_home, 'lib64')}", "-o", EXAMPLE_BIN]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"example build failed:\n{r.stdout}\n{r.stderr}")
    return EXAMPLE_BIN


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [],
                debug="--debug" in sys.argv))
