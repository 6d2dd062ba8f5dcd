"""Compile libmla_verify.so in-tree for sm_103a with nvcc (no CMake, one TU)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(_HERE)
SRC = os.path.join(_HERE, "csrc", "mla_verify.cu")
SRC_NOALLOC = os.path.join(_HERE, "csrc", "mla_verify_noalloc.cu")
HEADERS = [os.path.join(_HERE, "csrc", f) for f in os.listdir(os.path.join(_HERE, "csrc"))
           if f.endswith((".cuh", ".h"))] + [os.path.join(ROOT, "include", "mla_verify.h")]
OUT = os.path.join(_HERE, "libmla_verify.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(OUT):
        return False
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(f) <= t for f in [SRC, SRC_NOALLOC] + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return OUT
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-O3", "-std=c++17", ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), SRC, SRC_NOALLOC, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


OUT_FAULTS = os.path.join(_HERE, "libmla_verify_faults.so")


def build_fault_injection(force: bool = False) -> str:
    """The same library compiled with MLA_FAULT_INJECTION: 5 ms pipeline waits and
    mla_debug_set_fault(kind), for the tests of the timeout paths.  Never the
    library the package loads unless MLA_VERIFY_LIBRARY names it."""
    if not force and os.path.exists(OUT_FAULTS) and all(
            os.path.getmtime(f) <= os.path.getmtime(OUT_FAULTS) for f in [SRC, SRC_NOALLOC] + HEADERS):
        return OUT_FAULTS
    tmp = OUT_FAULTS + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-O3", "-std=c++17", ARCH, "-lineinfo", "-DMLA_FAULT_INJECTION", "-Xcompiler", "-fPIC",
           "-shared", "-I", os.path.join(ROOT, "include"), SRC, SRC_NOALLOC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT_FAULTS)
    return OUT_FAULTS


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
