"""Ahead-of-time build of libdg.so (the C-ABI library) for sm_103a with nvcc.

Run as ``python -m fp8_gemm_nt_gb300.build`` or call ``build()``. The library is
built in-tree, next to this file. The build fails if ptxas reports any register
spill or stack frame in a kernel (local memory on the hot path).
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libdg.so")
SOURCES = [os.path.join(CSRC, "dg_api.cu"), os.path.join(CSRC, "dg_no_alloc.cu"), os.path.join(CSRC, "dg_diag.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(verbose: bool = False, out: str = LIB) -> str:
    deps = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dg.h")]
    if os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(d) for d in deps):
        return out
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-diag-suppress", "177", "-I", INCLUDE, "-I", CSRC, "-o", out + ".tmp", *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = res.stdout + res.stderr
    if verbose or res.returncode != 0:
        sys.stderr.write(log)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed building libdg.so")
    bad = [m for m in re.finditer(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", log)
           if any(int(x) for x in m.groups())]
    if bad:
        sys.stderr.write(log)
        raise RuntimeError("a kernel uses local memory (stack frame or register spills)")
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
