"""Builds the CPU oracle (dflash_oracle.c) into oracle/_build/liboracle.so with gcc.

Test infrastructure: see the package docstring. Rebuilds when the source is newer than
the library, so a fresh checkout (or another CPU architecture) builds on first use.
"""

from __future__ import annotations

import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dflash_oracle.c")
OUT_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(OUT_DIR, "liboracle.so")


def compile_oracle(source: str, library: str) -> str:
    """gcc -O2 one C source into a shared library (written atomically)."""
    os.makedirs(os.path.dirname(library), exist_ok=True)
    tmp = f"{library}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC", "-pthread",
           "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, library)   # concurrent builders never load a partial file
    return library


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if needed and return the path of the shared library."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    return compile_oracle(SOURCE, LIBRARY)


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
