"""Build the C oracle into oracle/libssd_oracle.so (test infrastructure only).

Plain gcc, -O2 without fast-math, with floating-point contraction off so that
the oracle rounds the same way on x86_64 and aarch64 hosts, and OpenMP over
(sequence, head) pairs.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ssd_oracle.c")
LIB = os.path.join(HERE, "libssd_oracle.so")


def build(force: bool = False, extra_flags=(), out: str = LIB) -> str:
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC) and not extra_flags):
        return out
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", *extra_flags, SRC, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
