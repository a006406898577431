"""GB300-native W4A16 INT4 MoE expert GEMM pair (gate_up, then down).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/w4a16moe.h``); ``ops`` is a thin
ctypes binding with the same names. The library is loaded lazily, on first
use, and a missing library is an error: there is no CPU fallback.
"""

__all__ = ["ops", "workloads", "build"]
