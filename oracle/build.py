"""Compile the oracle's C source into a shared library (test infrastructure).

The oracle is plain single-threaded C built with every binary32 operation
rounded on its own (``-ffp-contract=off``; no fast-math), so that its
results are the IEEE results of the operations as written.  Run as a
script, or call :func:`build`.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "cc_oracle.c")
LIBRARY = os.path.join(HERE, "libcc_oracle.so")

CFLAGS = [
    "-O2",
    "-std=c11",
    "-ffp-contract=off",
    "-fno-fast-math",
    "-fPIC",
    "-shared",
    "-Wall",
    "-Wextra",
]


def build(force: bool = False) -> str:
    """Build ``libcc_oracle.so`` beside its source if missing or stale."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    cc = os.environ.get("CC", "gcc")
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    try:
        subprocess.run([cc, *CFLAGS, SOURCE, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, LIBRARY)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
