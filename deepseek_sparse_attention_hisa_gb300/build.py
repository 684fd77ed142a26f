"""In-tree build of libhisa.so for sm_103a (nvcc, no cmake).

Each .cu translation unit under csrc/ compiles in parallel to an object file in
_build/, then nvcc links them into deepseek_sparse_attention_hisa_gb300/libhisa.so
(CUDA runtime linked statically, so the library needs only the driver at run time).
A stamp of the sources and flags skips the build when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libhisa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                     "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhisa.so")


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp() -> str:
    h = hashlib.sha256()
    files = _sources() + sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                if f.endswith((".cuh", ".h")))
    files.append(os.path.join(INCLUDE, "hisa.h"))
    for f in files:
        h.update(os.path.basename(f).encode())          # independent of where the tree lives
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


# The sources each profiled kernel is compiled from: its translation unit and the headers it
# includes. A profile's counters stay valid while these bytes (and the flags) are unchanged.
KERNEL_SOURCES = {
    "k_attend_tc": ["k_attend_tc.cu", "hisa_internal.cuh", "tc_ptx.cuh"],
    "k_score_pipe": ["k_score_pipe.cu", "pipe_common.cuh", "select_core.cuh", "hisa_internal.cuh", "tc_ptx.cuh"],
    "k_score_gemm": ["k_score_gemm.cu", "hisa_internal.cuh", "tc_ptx.cuh"],
}


def kernel_stamp(kernel: str) -> str:
    """Hash of one kernel's sources and the compile flags (see KERNEL_SOURCES)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(f for f in NVCC_FLAGS if f != INCLUDE).encode())   # not where the tree lives
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libhisa.so in-tree if the sources changed; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp_file = os.path.join(BUILD, "libhisa.stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIB
    nvcc = _nvcc()
    srcs = _sources()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, "-c", src, "-o", obj] + NVCC_FLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
