"""Build libfa.so in-tree with nvcc for sm_103a (no GPU needed to build).

Each translation unit under csrc/ is compiled in parallel, then linked into a
shared library with the CUDA runtime linked statically, so the library loads
on a machine without a GPU (calls then return FA_ERR_CUDA).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libfa.so")
# Ablation builds of the same sources (loaded only when asked for by name):
#   unfused      two scalar FMAs instead of one packed fma.rn.f32x2
#   threshold0   rescale on every rise of the row max (no lazy skip)
#   trace        clock64 pipeline trace of the first CTA (fa_debug_trace_read)
VARIANTS = {
    "unfused": ["-DFA_UNFUSE_FMA"],
    "threshold0": ["-DFA_RESCALE_THRESHOLD=0.0f"],
    "trace": ["-DFA_TRACE"],
}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cuh", ".h"))) + [os.path.join(INCLUDE, "fa.h")]


def variant_path(variant=None) -> str:
    return LIB_PATH if not variant else os.path.join(PKG, f"libfa_{variant}.so")


def up_to_date(lib_path=LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant=None) -> str:
    """Compile and link libfa.so (or an ablation variant); returns its path."""
    lib_path = variant_path(variant)
    if variant:
        extra_flags = list(extra_flags) + VARIANTS[variant]
    build_dir = BUILD_DIR if not variant else BUILD_DIR + "_" + variant
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC] + list(extra_flags)
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            print(log)
    objs = [o for o, _ in results]
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libfa.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    var = next((a.split("=", 1)[1] for a in sys.argv if a.startswith("--variant=")), None)
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, variant=var))
