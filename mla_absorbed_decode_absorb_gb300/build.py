"""Builds libmla_decode.so in-tree for sm_103a with nvcc (no cmake).

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into
``mla_absorbed_decode_absorb_gb300/libmla_decode.so`` against the shared CUDA
runtime (the same ``libcudart.so`` PyTorch loads).  Usage:
``python -m mla_absorbed_decode_absorb_gb300.build``.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmla_decode.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla_decode")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, " ".join(cmd), p.stdout


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile and link the library if any source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = NVCC_FLAGS + ARCH + list(extra_flags or [])
    jobs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.splitext(os.path.basename(src))[0] + ".o")
        jobs.append((obj, [nvcc, *flags, "-c", src, "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda j: _run(j[1]), jobs))
    for rc, cmd, out in results:
        if verbose or rc != 0:
            sys.stderr.write(cmd + "\n" + out)
        if rc != 0:
            raise RuntimeError("nvcc failed:\n" + cmd + "\n" + out)
    tmp = LIB + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in jobs],
            "-Xlinker", "-rpath=" + _cuda_lib_dir(nvcc)]
    rc, cmd, out = _run(link)
    if verbose or rc != 0:
        sys.stderr.write(cmd + "\n" + out)
    if rc != 0:
        raise RuntimeError("link failed:\n" + cmd + "\n" + out)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
