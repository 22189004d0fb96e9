"""Seeded synthetic inputs shared by the oracle tests and the CUDA path.

Holds no decoder arithmetic: it maps (seed, tensor id, index) to numbers with a
counter-based generator (splitmix64 + Box-Muller, see synth.c) and lays them
out as the tensors a Llama-style decoder takes.  Neither the oracle nor the
CUDA library is imported here.
"""
import ctypes
import os

import numpy as np

from ._build import LIB, build

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        L = ctypes.CDLL(LIB)
        L.synth_splitmix64.restype = ctypes.c_uint64
        L.synth_splitmix64.argtypes = [ctypes.c_uint64]
        L.synth_normal.restype = ctypes.c_double
        L.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64]
        L.synth_f32_to_bf16.restype = ctypes.c_uint16
        L.synth_f32_to_bf16.argtypes = [ctypes.c_float]
        L.synth_normal_bf16.restype = None
        L.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                                        ctypes.c_int]
        L.synth_kv_bf16.restype = None
        L.synth_kv_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32] + [ctypes.c_int64] * 5 + [
            ctypes.c_void_p, ctypes.c_double, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
        L.synth_uniform_i32.restype = None
        L.synth_uniform_i32.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        _lib = L
    return _lib


def nthreads():
    return max(1, min(64, os.cpu_count() or 1))


def splitmix64(x):
    return int(lib().synth_splitmix64(ctypes.c_uint64(x & 0xFFFFFFFFFFFFFFFF)))


def normal(seed, tid, i):
    return float(lib().synth_normal(seed, tid, i))


def normal_bf16(seed, tid, shape, mean=0.0, std=1.0):
    """bf16 bit patterns (uint16) of N(mean, std) samples, C order."""
    out = np.empty(shape, dtype=np.uint16)
    lib().synth_normal_bf16(seed, tid, out.size, mean, std, out.ctypes.data, nthreads())
    return out


def kv_bf16(seed, tid, L, B, nkv, max_ctx, d, ctx, mean=0.0, std=1.0):
    """[L][B][nkv][max_ctx][d] bf16 bits: N(mean,std) at positions < ctx[b], zero beyond."""
    ctx = np.ascontiguousarray(np.asarray(ctx, dtype=np.int32))
    assert ctx.shape == (B,)
    out = np.empty((L, B, nkv, max_ctx, d), dtype=np.uint16)
    lib().synth_kv_bf16(seed, tid, L, B, nkv, max_ctx, d, ctx.ctypes.data, mean, std,
                        out.ctypes.data, nthreads())
    return out


def uniform_i32(seed, tid, n, lo, hi):
    """n integers uniform in the inclusive range [lo, hi]."""
    out = np.empty(n, dtype=np.int32)
    lib().synth_uniform_i32(seed, tid, n, lo, hi, out.ctypes.data)
    return out


def bf16_to_f32(a):
    """Exact widening of bf16 bit patterns to float32 (test/bench convenience)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a):
    """Round-to-nearest-even narrowing of float32 to bf16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
