"""Build libmk.so in-tree with nvcc for sm_103a (no torch extension machinery:
the library is a plain C ABI)."""
import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmk.so")
SOURCES = ["mk_kernel.cu", "mk_stream.cu", "mk_runtime.cu", "mk_plan.cpp", "mk_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include"), "-I", os.path.join(HERE, "csrc")]


def nvcc():
    return shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


def build(verbose=False):
    tmp = tempfile.mkdtemp(prefix="mk_build_")
    try:
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(tmp, src + ".o")
            cmd = [nvcc()] + ARCH + FLAGS + ["-c", os.path.join(HERE, "csrc", src), "-o", obj]
            if verbose and src.endswith("kernel.cu"):
                cmd += ["-Xptxas", "-v"]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
            objs.append(obj)
        for cmd, pr in procs:
            out, _ = pr.communicate()
            if pr.returncode != 0 or verbose:
                print(out.decode(errors="replace"))
            if pr.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
        tmp_lib = os.path.join(tmp, "libmk.so")
        subprocess.run([nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp_lib] + objs,
                       check=True)
        os.replace(tmp_lib, LIB)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return LIB
