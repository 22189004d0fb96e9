"""GB300-native persistent decode megakernel: one launch per decoder forward
pass, one resident block per SM interpreting a host-built instruction list.

The compute path is libmk.so (hand-written CUDA for sm_103a behind the C ABI
in include/mk.h); `mk` is its ctypes binding with the same names.
"""
from . import mk  # noqa: F401
from ._build import LIB, build  # noqa: F401
