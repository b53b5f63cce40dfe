"""accelerator_gb300 -- libgemm, dense C = A*B on one GB300 (sm_103a).

The compute lives in the CUDA library built from ``csrc/`` (see ``build.py``);
``binding.py`` is the thin ctypes layer over its C ABI.  Importing the package
loads nothing: the library is opened at the first call, and a missing library
is an error, never a fallback.
"""

FP32, TF32, BF16, FP16, FP32_VIA_BF16 = 0, 1, 2, 3, 4

__all__ = ["gemm", "gemm_ex", "GemmError", "FP32", "TF32", "BF16", "FP16", "FP32_VIA_BF16"]


def __getattr__(name):
    if name in ("gemm", "gemm_ex", "GemmError"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
