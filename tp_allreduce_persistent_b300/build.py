"""Build the C-ABI library libllar.so in-tree with nvcc for sm_103a.

Usage: python -m tp_allreduce_persistent_b300.build [--force]
The library lands next to this file, so it travels with the source tree.
"""

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libllar.so")
# diagnostic build: the same library with poll counting compiled in
POLLS_LIB = os.path.join(HERE, "libllar_polls.so")
SOURCES = ["llar_runtime.cu", "llar_kernels.cu", "llar_llbuffer.cu"]
HEADERS = ["llar_internal.h", "llar_device.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    for name in ("llar.h", "llar_llbuffer.h", "llar_llbuffer.cuh"):
        files.append(os.path.join(INCLUDE, name))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_poll_stats(force=False):
    """The poll-counting variant (LLAR_POLL_STATS), next to the library."""
    if not force and up_to_date(POLLS_LIB):
        return POLLS_LIB
    return build(defines=["LLAR_POLL_STATS=1"], out=POLLS_LIB)


def build(force=False, verbose=False, defines=(), out=None):
    """Compile every CUDA source into libllar.so (skipped when up to date).

    `defines` (e.g. ["LLAR_BULK_TILE=4096"]) and `out` build a variant
    library elsewhere, for tuning sweeps; the default build is LIB."""
    if out is None and not defines and not force and up_to_date():
        return LIB
    nvcc = nvcc_path()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    target = out or LIB
    tmp = target + ".tmp"
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "--threads", "3",
           "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
           "-cudart", "shared", "-Xlinker", "-rpath=" + cuda_lib,
           "-o", tmp] + ["-D" + d for d in defines] + [os.path.join(CSRC, f) for f in SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


if __name__ == "__main__":
    if "--poll-stats" in sys.argv:
        print(build_poll_stats(force="--force" in sys.argv))
    else:
        build(force="--force" in sys.argv, verbose="-v" in sys.argv)
        print(LIB)
