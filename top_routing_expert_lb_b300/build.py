"""Builds libmoe_b300.so in-tree with nvcc for sm_103a.

With MOE_BUILD_BOUNDS_CHECK=1 in the environment of the build, the library is
compiled with -DMOE_BOUNDS_CHECK: every data-dependent index in the kernels is
range-checked, a failed check is reported as MOE_ERR_BOUNDS by
moe_check_status and the access is skipped (a debug build that stands in for a
device memory checker).  The recorded source hash covers the flags, so
switching the variable rebuilds the library."""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libmoe_b300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe.h")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
]


def flags():
    extra = ["-DMOE_BOUNDS_CHECK"] if os.environ.get("MOE_BUILD_BOUNDS_CHECK") == "1" else []
    return NVCC_FLAGS + extra


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.h")) + [HEADER])


def source_hash() -> str:
    h = hashlib.sha256()
    for s in sources():
        h.update(os.path.basename(s).encode())
        with open(s, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(flags()).encode())
    return h.hexdigest()


def is_stale() -> bool:
    """True when the library is missing or was built from other sources
    (compared by content, since copies of the tree need not keep mtimes)."""
    if not os.path.exists(LIB) or not os.path.exists(LIB + ".srchash"):
        return True
    with open(LIB + ".srchash") as fh:
        return fh.read().strip() != source_hash()


def build(verbose: bool = False, extra=(), out: str | None = None) -> str:
    """Compiles the library into the package (or into `out`, without touching
    the in-tree copy); `extra` adds nvcc flags."""
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = os.environ.get("NVCC", "nvcc")
    if not os.path.exists(nvcc) and os.path.exists("/usr/local/cuda/bin/nvcc"):
        nvcc = "/usr/local/cuda/bin/nvcc"
    cus = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    target = out or LIB
    tmp = target + ".tmp"
    cmd = [nvcc, *flags(), *extra, "-o", tmp, *cus]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    if out is None:
        with open(LIB + ".srchash", "w") as fh:
            fh.write(source_hash() + "\n")
    return target


def ensure_built() -> str:
    if is_stale():
        build()
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
