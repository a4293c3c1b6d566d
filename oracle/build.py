"""Compile the CPU oracle (gemm_ref.c -> liboracle.so) with the host C compiler.

Test infrastructure: builds the checker, never the product.  Portable flags only
(the same source builds on x86-64 and aarch64); -ffp-contract=off keeps every
multiply and add a separately rounded binary64 operation.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))


def build(verbose: bool = False) -> str:
    src = os.path.join(_HERE, "gemm_ref.c")
    out = os.path.join(_HERE, "liboracle.so")
    tmp = out + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
