"""Build libspec_verify.so in-tree with nvcc for sm_103a.

One translation unit, one -gencode, no cmake (about 30 s of nvcc).  The
checked variant, libspec_verify_checked.so, is the same source compiled
with -DSV_CHECKED: every global index the verify kernel forms is tested
against its buffer before the access (a failure sets SV_DEV_OUT_OF_BOUNDS
instead of faulting); the tests run it on small and odd shapes.  Both
compile in parallel.
``python -m speculative_decoding_verification_25_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libspec_verify.so")
LIB_CHECKED = os.path.join(PKG, "libspec_verify_checked.so")
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    srcs = [os.path.join(PKG, "csrc", f) for f in os.listdir(os.path.join(PKG, "csrc"))]
    srcs.append(os.path.join(INCLUDE, "spec_verify.h"))
    return (not os.path.exists(lib)
            or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs))


def _cmd(lib: str, checked: bool, verbose: bool):
    cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I" + INCLUDE, "-o", lib + ".tmp", SRC]
    if checked:
        cmd.insert(1, "-DSV_CHECKED")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(verbose: bool = False, force: bool = False, checked: bool = True) -> str:
    """Compile the library (and, with ``checked``, its checked variant)
    when a source is newer than it or ``force``; returns the library path."""
    jobs = [(LIB, False)] + ([(LIB_CHECKED, True)] if checked else [])
    jobs = [(lib, chk) for lib, chk in jobs if force or _stale(lib)]
    procs = [(lib, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                         text=True))
             for lib, cmd in ((lib, _cmd(lib, chk, verbose)) for lib, chk in jobs)]
    errors = []
    for lib, cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
            continue
        if verbose:
            sys.stderr.write(out)
        os.replace(lib + ".tmp", lib)
    if errors:
        raise RuntimeError("\n".join(errors))
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force=True))
