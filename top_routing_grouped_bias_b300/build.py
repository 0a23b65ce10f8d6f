"""Builds libmoe_b300.so in this package directory with nvcc for sm_103a.

    python -m top_routing_grouped_bias_b300.build [--verbose-ptxas]

Static cudart is linked in, and the driver's tensor-map encoder is reached
through the runtime's driver entry-point query, so the library loads on a
machine without a GPU driver (the symbols can be listed there; nothing runs).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmoe_b300.so")
SOURCES = ["api.cu", "route.cu", "dispatch.cu", "combine.cu", "grouped_gemm.cu",
           "dispatch_noalloc.cu", "stats.cu", "expert_choice.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "moe.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose_ptxas: bool = False, out: str = LIB,
          defines: tuple = ()) -> str:
    """Compile the library to `out`; `defines` are extra -D tuning constants
    (stage counts, CTA-pair threshold) for measurement builds."""
    if not force and not verbose_ptxas and not defines and out == LIB and not _stale():
        return LIB
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", out + ".tmp"]
    cmd += [f"-D{d}" for d in defines]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="--verbose-ptxas" in sys.argv))
