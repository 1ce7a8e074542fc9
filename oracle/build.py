"""Compile the float64 CPU oracle (ss_oracle.c) into oracle/libssoracle.so.

Test infrastructure only: the library is loaded by the tests, the smoke check
and the benchmark's CPU-baseline leg.
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ss_oracle.c")
LIB = os.path.join(HERE, "libssoracle.so")


def build(src: str = SRC, out: str = LIB, extra=()) -> str:
    """Build `src` into the shared library `out` (rebuilt when older than src)."""
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra:
        return out
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
           "-fno-fast-math", "-ffp-contract=off", *extra, src, "-o", out, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    print(build())
    sys.exit(0)
