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
LIB_CHECKED = os.path.join(BUILD, "libmk_checked.so")
SOURCES = ["mk_kernel_hd64.cu", "mk_kernel_hd128.cu", "mk_kernel.cu", "mk_host.cpp", "mk_noalloc.cu", "mk_w2a8.cu",
           "mk_prefill.cu", "mk_twell.cu"]
DEPS = SOURCES + ["mk_kernel.cuh", "mk_plan.h", "mk_internal.h", "mk_prefill.h"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmk.so")


def flags() -> list[str]:
    return ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", f"-I{os.path.join(ROOT, 'include')}"]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in DEPS] + [os.path.join(ROOT, "include", "mk.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """checked=True builds libmk_checked.so: every device-side access is
    validated against the registered buffers (slow; for diagnosing faults)."""
    lib = LIB_CHECKED if checked else LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    procs, objs = [], []
    tag = ".chk" if checked else ""
    for s in SOURCES:
        obj = os.path.join(BUILD, s + tag + ".o")
        extra = ["-Xptxas", "-v"] if (verbose and s.endswith(".cu")) else []
        if checked:
            extra += ["-DMK_CHECKED"]
        cmd = [nv, *flags(), *extra, "-c", os.path.join(CSRC, s), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode:
            print(out.decode(errors="replace"))
        if pr.returncode:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nv, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs],
                   check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
