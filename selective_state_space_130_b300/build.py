"""Build libssscan.so (the sm_103a kernels and their C ABI) in the package dir.

nvcc cross-compiles for sm_103a without a GPU. The CUDA runtime is linked as
the shared libcudart.so.13, so a process that already loaded it (PyTorch does)
shares one runtime instance and one notion of the current device with the
library; the driver's tensor-map encoder is resolved at run time, so the
library loads on a machine without a GPU (its calls then fail cleanly).
"""

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libssscan.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(os.path.dirname(HERE), "include", "ss_scan.h")]


def up_to_date(out=LIB):
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in deps())


def build(force=False, verbose=False, out=LIB, extra=()):
    if not force and up_to_date(out):
        return out
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2",
           "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-I", os.path.join(os.path.dirname(HERE), "include"),
           *(["-Xptxas", "-v"] if verbose else []), *extra, *sources(), "-o", out]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
