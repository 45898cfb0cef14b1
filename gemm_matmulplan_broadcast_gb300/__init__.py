"""GB300-native ONNX MatMul: a C-ABI CUDA library (``libolc_matmul.so``,
declared in ``include/olc_matmul.h``) and a thin ctypes binding over it.

    from gemm_matmulplan_broadcast_gb300 import Plan, matmul

The library is loaded on first use; if it has not been built, that use
raises (build with ``python -m gemm_matmulplan_broadcast_gb300.build``).
"""

from .binding import ALGORITHMS, GemmPlan, GroupedPlan, OlcError, Plan, gemm, load, matmul  # noqa: F401

__all__ = ["Plan", "GemmPlan", "GroupedPlan", "matmul", "gemm", "load", "OlcError", "ALGORITHMS"]
