"""In-tree build of ``libbip.so`` (sm_103a) with nvcc, translation units in parallel.

``python -m invariant_paged_prefill_gb300.build`` builds (or rebuilds when a
source is newer than the library).
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
SOURCES = ["bip_host.cpp", "bip_attn.cu", "bip_attn_gather.cu", "bip_attn_mask.cu", "bip_merge.cu", "bip_append.cu",
           "bip_plan_dev.cu", "bip_mask_skip.cu", "bip_upload.cu", "bip_no_alloc.cu"]
HEADERS = ["bip_internal.h", "bip_numerics.cuh", "bip_ptx.cuh", "bip_attn_impl.cuh"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
# -fmad=false: no silent contraction of a*b+c in device code; the numerics
# use explicitly rounded intrinsics, and the same bits must come out of the
# attention kernel's fold and the merge kernel.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", ARCH, "-Xcompiler", "-fPIC,-O2",
              "-I" + os.path.join(ROOT, "include")]


def library_path() -> str:
    return os.path.join(PKG, "libbip.so")


def _nvcc() -> str:
    nv = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nv):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbip.so")
    return nv


def _inputs() -> list[str]:
    return [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "bip.h")]


def is_stale() -> bool:
    lib = library_path()
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build_library(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD_DIR, src + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for (_, log), src in zip(results, SOURCES):
            if log.strip():
                print(f"--- {src}\n{log}", file=sys.stderr)
    tmp = library_path() + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, library_path())
    return library_path()


def ensure_built() -> str:
    if is_stale():
        build_library()
    return library_path()


if __name__ == "__main__":
    print(build_library(verbose=True, ptxas_info="-v" in sys.argv))
