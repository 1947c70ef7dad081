"""Compile the fp64 oracle (``pa_oracle.c``) into a shared library with gcc.

TEST INFRASTRUCTURE ONLY: the oracle is the checker for the CUDA library, never a
part of it.  ``-ffp-contract=off`` keeps the double arithmetic identical on x86-64
and aarch64 (no fused multiply-add contraction); no ``-ffast-math``.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pa_oracle.c")
LIBRARY = os.path.join(HERE, "libpa_oracle.so")

CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]


def build(source: str = SOURCE, output: str = LIBRARY, quiet: bool = True,
          werror: bool = True) -> str:
    """Compile ``source`` to ``output`` and return the library path."""
    cmd = ["gcc", *CFLAGS, *(["-Werror"] if werror else []), source, "-o", output, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{res.stdout}{res.stderr}")
    if not quiet:
        print(" ".join(cmd), file=sys.stderr)
    return output


def needs_build(output: str = LIBRARY, source: str = SOURCE) -> bool:
    return (not os.path.exists(output)) or os.path.getmtime(output) < os.path.getmtime(source)


if __name__ == "__main__":
    print(build(quiet=False))
