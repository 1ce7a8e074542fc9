"""Build libssscan.so (the sm_103a kernels and their C ABI) in the package dir.

nvcc cross-compiles for sm_103a without a GPU. Each .cu file in csrc/ is
compiled to an object in parallel (the scan kernel's dtype instantiations live
in separate files for this), then linked into one shared library. The CUDA
runtime is linked as the shared libcudart.so.13, so a process that already
loaded it (PyTorch does) shares one runtime instance and one notion of the
current device with the library; the driver's tensor-map encoder is resolved
at run time, so the library loads on a machine without a GPU (its calls then
fail cleanly).
"""

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(HERE, "libssscan.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(ROOT, "include", "ss_scan.h")]


def _newest(paths):
    return max(os.path.getmtime(f) for f in paths)


def up_to_date(out=LIB):
    return os.path.exists(out) and _newest(sources() + headers()) <= os.path.getmtime(out)


def build(force=False, verbose=False, out=LIB, jobs=0):
    if not force and up_to_date(out):
        return out
    nvcc = os.environ.get("NVCC", "nvcc")
    os.makedirs(OBJ, exist_ok=True)
    hdr_time = _newest(headers())

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.basename(src)[:-3] + ".o")
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
            return obj, ""
        cmd = [nvcc, *ARCH, *FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    n = jobs or min(len(sources()), os.cpu_count() or 1)
    with ThreadPoolExecutor(n) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    # no rpath: libcudart.so.13 is found through the loader's search path, or is
    # already loaded by the host process (PyTorch), which this library then shares
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", out]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
