"""Compile libsynth.so (plain C, gcc) next to this file."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")


def build_cmd():
    return ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", LIB,
            os.path.join(HERE, "synth.c"), "-lm"]


def build():
    subprocess.run(build_cmd(), check=True)
    return LIB
