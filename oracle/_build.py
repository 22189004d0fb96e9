"""Compile liboracle.so (plain C, gcc) next to this file.  Building the
checker is not using it: only tests/, smoke() and bench.py's CPU-baseline leg
load the library."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")


def build_cmd():
    return ["gcc", "-O2", "-fPIC", "-shared", "-o", LIB,
            os.path.join(HERE, "oracle.c"), os.path.join(HERE, "replay.c"), "-lm"]


def build():
    subprocess.run(build_cmd(), check=True)
    return LIB
