"""Builds the CPU oracle (test infrastructure): moe_oracle.cpp -> lib/libmoe_oracle.so.

Plain g++ with OpenMP and floating-point contraction off, so that every
operation of the oracle rounds once, as written.  ``build(source=...)``
compiles a modified copy of the source elsewhere (the mutation tests use it
to plant mistakes in the oracle).

    python -m oracle.build
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "lib", "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def _cxx() -> str:
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("g++ not found: the CPU oracle needs a C++17 compiler")
    return cxx


def build(out: str = LIB, source: str | None = None, force: bool = False) -> str:
    """Compile the oracle (or `source`, a modified copy of its text) into `out`; returns `out`."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if source is None:
        src = SRC
        if not force and os.path.exists(out) and os.path.getmtime(out) >= max(os.path.getmtime(SRC),
                                                                              os.path.getmtime(__file__)):
            return out
    else:
        fd, src = tempfile.mkstemp(suffix=".cpp", dir=os.path.dirname(out))
        with os.fdopen(fd, "w") as fh:
            fh.write(source)
    tmp = out + f".tmp{os.getpid()}"
    try:
        res = subprocess.run([_cxx(), *FLAGS, src, "-o", tmp], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, out)
    finally:
        if source is not None:
            os.unlink(src)
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
