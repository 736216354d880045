"""Compile the fp64 CPU oracle (``oracle.c``) into a shared library with gcc.

Test infrastructure only: the product never loads what this builds.

The build keeps IEEE fp64 semantics: no ``-ffast-math`` and ``-ffp-contract=off`` so that x86
and Arm hosts round every operation the same way.  ``mutant=k`` builds a copy with one planted
mistake (``-DORACLE_MUTANT=k``) for the tests that show the pins catch such mistakes.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if not mutant else f"liboracle_mutant{mutant}.so"
    if mutant:
        return os.path.join(HERE, "_build", name)
    return os.path.join(HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)
            and os.path.getmtime(out) >= os.path.getmtime(__file__)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))
