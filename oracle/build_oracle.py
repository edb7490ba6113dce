"""Compile the CPU oracle (``lora_oracle.c``) into ``liblora_oracle.so``.

Test infrastructure: building the checker is not using it.  Plain gcc, -O2,
no fast-math and no fused multiply-add (``-ffp-contract=off``) so that the
oracle's fp32 rounding sequence is exactly the one written in the source.
OpenMP parallelises over independent rows only; results do not depend on the
thread count.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lora_oracle.c")


def library_path() -> str:
    return os.path.join(HERE, "liblora_oracle.so")


def override_path() -> str | None:
    """A prebuilt oracle library to load instead (used by the mutation tests,
    which plant a mistake in a copy of the source and check the pins fail)."""
    return os.environ.get("LORA_ORACLE_LIBRARY") or None


def build(force: bool = False) -> str:
    out = library_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
