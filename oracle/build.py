"""Builds the fp64 CPU oracle (``libsdpa_oracle.so``) beside its source with gcc.

Portable flags only (no -march), so the same source builds on x86_64 and on
aarch64 hosts. Test infrastructure: see ``oracle/__init__.py``.
"""
from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")


def library_path() -> str:
    return os.path.join(_HERE, "libsdpa_oracle.so")


def is_stale() -> bool:
    lib = library_path()
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(_SRC)


def build(verbose: bool = False) -> str:
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           _SRC, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
