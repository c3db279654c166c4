"""Builds libmk.so (the megakernel and its C ABI) in-tree for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmk.so")
SOURCES = ["mk_kernel.cu", "mk_host.cpp"]
DEPS = SOURCES + ["mk_plan.h"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmk.so")


def flags() -> list[str]:
    return ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", f"-I{os.path.join(ROOT, 'include')}"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in DEPS] + [os.path.join(ROOT, "include", "mk.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    procs, objs = [], []
    for s in SOURCES:
        obj = os.path.join(BUILD, s + ".o")
        extra = ["-Xptxas", "-v"] if (verbose and s.endswith(".cu")) else []
        cmd = [nv, *flags(), *extra, "-c", os.path.join(CSRC, s), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode:
            print(out.decode(errors="replace"))
        if pr.returncode:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nv, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
