"""Builds the oracle's C primitives (``liboracle_clo.so``) -- test infrastructure."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "clo_oracle.c")
LIB = os.path.join(HERE, "liboracle_clo.so")


def build_oracle(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB):
        cc = os.environ.get("CC", "gcc")
        tmp = LIB + ".tmp"
        subprocess.run([cc, "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"],
                       check=True)
        os.replace(tmp, LIB)
    return LIB
