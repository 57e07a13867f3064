"""Builds libdsa.so (the C-ABI library) from csrc/ with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``sparse_attention_gemm_gb300/_build/libdsa.so``.  No cmake, no torch
extension machinery: the library has a plain C ABI (include/dsa.h).
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdsa.so")
# The checked build (-DDSA_CHECKED: in-kernel range checks that record
# DSA_STATUS_CHECK_FAILED and skip the access) goes to its own directory.
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libdsa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "small_ops.cu", "topk.cu", "indexer.cu", "attention.cu", "attention_bwd.cu", "pipeline.cu"]
HEADERS = ["common.cuh", "block_sort.cuh", "topk_select.cuh"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compiles libdsa.so (or, with checked=True, the range-checked build into
    _build_checked/) and returns its path."""
    out_dir = BUILD_CHECKED if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "dsa.h")]
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    "--expt-relaxed-constexpr", *(["-DDSA_CHECKED"] if checked else []), *extra_flags]
    objs = []

    def compile_one(src):
        path = os.path.join(CSRC, src)
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        if force or _stale(obj, [path, *hdrs]):
            cmd = [nvcc, *flags, "-c", path, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-lpthread", "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
