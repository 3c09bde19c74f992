"""B300-native packed low-bit (1-bit / ternary, group 128) GEMV and GEMM.

The compute path is liblb.so (CUDA for sm_103a, C ABI in include/lb.h); ``lb`` is its ctypes
binding and ``tensors`` adds torch allocation helpers.  ``synth`` holds the seeded input
generators.  Import ``gemm_lb_gemv_02_b300.lb`` to load the library (it raises ImportError if the
library has not been built).
"""

__all__ = ["lb", "tensors", "synth", "build"]
