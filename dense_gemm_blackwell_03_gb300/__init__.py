"""bwgemm: dense ``C = A @ B.T`` (bf16 / fp16, K-major operands) on one GB300.

The arithmetic runs only in the hand-written sm_103a kernels of
``libbwgemm.so`` (built from ``csrc/``).  The Python side is argument
marshalling over the library's C ABI (``include/bwgemm.h``); importing this
package loads nothing, the first call into the binding loads the library, and
it raises if the library is missing rather than computing anything on the host.
"""
import importlib

__all__ = ["BF16", "FP16", "BwgemmError", "Plan", "PlanOptions", "gemm",
           "library_path", "load_library", "select_config", "check_args"]


def __getattr__(name):
    if name in __all__:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
