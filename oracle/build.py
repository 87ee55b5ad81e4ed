"""Compile the CPU oracle (test infrastructure) into ``oracle/_build/liblq_oracle.so``.

Plain gcc, C11, -O2, -ffp-contract=off and no fast-math, so that every fp32
multiply, add and fmaf rounds exactly where the source says it does.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def library_path() -> str:
    return os.path.join(OUT_DIR, "liblq_oracle.so")


def stale() -> bool:
    out = library_path()
    return (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    out = library_path()
    if not force and not stale():
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *FLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
