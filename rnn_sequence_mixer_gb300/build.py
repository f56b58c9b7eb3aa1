"""Compile libhla.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

nvcc compiles every translation unit of ``csrc/`` in parallel and links them
into ``rnn_sequence_mixer_gb300/_build/libhla.so`` (CUDA runtime linked
statically, so the library depends only on the driver).  Rebuilds only when a
source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libhla.so")
# Measurement-only companion: the tensor-core rate of the prefill's MMA sequence
# with shared-memory-resident operands (bench.py); not part of the C ABI.
MMABENCH_SRC = os.path.join(CSRC, "microbench", "mma_rate.cu")
MMABENCH_LIB = os.path.join(BUILD, "libhla_mmabench.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
    "-Xptxas", "-warn-spills", "-I", INCLUDE, "-I", CSRC,
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhla.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    obj_dir = os.path.join(BUILD, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link of libhla.so failed:\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))


def build_mmabench(force: bool = False) -> str:
    """Compile libhla_mmabench.so (one translation unit) next to libhla.so."""
    deps = [MMABENCH_SRC, os.path.join(CSRC, "umma.cuh"), os.path.join(CSRC, "hla_internal.cuh")]
    if (not force and os.path.exists(MMABENCH_LIB)
            and all(os.path.getmtime(p) <= os.path.getmtime(MMABENCH_LIB) for p in deps)):
        return MMABENCH_LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = MMABENCH_LIB + ".tmp"
    cmd = [_nvcc(), *NVCC_FLAGS, "-shared", MMABENCH_SRC, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on mma_rate.cu:\n{res.stderr}")
    os.replace(tmp, MMABENCH_LIB)
    return MMABENCH_LIB
