"""ctypes binding over libgemm's C ABI (include/gemm.h).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built this raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FP32, TF32, BF16, FP16, FP32_VIA_BF16, TF32_RN = 0, 1, 2, 3, 4, 5
MODES = {"fp32": FP32, "tf32": TF32, "bf16": BF16, "fp16": FP16, "fp32_via_bf16": FP32_VIA_BF16,
         "tf32_rn": TF32_RN}

OK = 0
ERR_INVALID_ARG = 1
ERR_MISALIGNED = 2
ERR_CUDA = 3
ERR_NO_MEMORY = 4
ERR_UNSUPPORTED_DEVICE = 5
ERR_TIMEOUT = 6
ERR_SCRATCH_LIMIT = 7
ERR_BOUNDS = 8          # debug build only: an out-of-buffer access was caught and skipped

# Every entry point include/gemm.h declares, with its ctypes signature.
_i64, _vp, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "gemm": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "gemm_ex": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float, ctypes.c_float, _int,
                       _vp]),
    "gemm_status_string": (ctypes.c_char_p, [_int]),
    "gemm_debug_status": (_int, [_vp]),
    "gemm_version": (_int, []),
    "gemm_debug_build": (_int, []),
    "gemm_launch_count": (_i64, []),
    "gemm_selftest_bounded_wait": (_int, [_i64, _vp]),
    "gemm_tf32_noalloc": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp]),
}

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = "gemm"):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libgemm.so.  Raises if it has not been built.

    With LIBGEMM_DEBUG=1 in the environment (read at the first call) the debug
    build is loaded instead: kernels with device-side bounds checks, built by
    ``python -m accelerator_gb300.build --debug``.
    """
    global _lib
    if _lib is not None:          # loaded: no lock needed to read it
        return _lib
    with _lock:
        if _lib is None:
            debug = os.environ.get("LIBGEMM_DEBUG", "") not in ("", "0")
            path = _build.LIB_DEBUG if debug else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgemm is not built ({path} missing); run "
                    "`python -m accelerator_gb300.build" + (" --debug" if debug else "")
                    + "` (or __graft_entry__.build())")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(handle, name)
                f.restype = res
                f.argtypes = args
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


def gemm_raw(a_ptr: int, b_ptr: int, c_ptr: int, M: int, K: int, N: int, mode: int,
             stream_ptr: int = 0) -> int:
    """Direct call of the C entry point with raw addresses; returns the status."""
    return int(lib().gemm(a_ptr or None, b_ptr or None, c_ptr or None, M, K, N, mode,
                          stream_ptr or None))


def gemm_ex_raw(a_ptr: int, b_ptr: int, c_ptr: int, M: int, K: int, N: int, alpha: float,
                beta: float, mode: int, stream_ptr: int = 0) -> int:
    """Direct call of gemm_ex with raw addresses; returns the status."""
    return int(lib().gemm_ex(a_ptr or None, b_ptr or None, c_ptr or None, M, K, N, float(alpha),
                             float(beta), mode, stream_ptr or None))


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def gemm(A, B, C=None, mode=FP32, stream=None):
    """C = A @ B on the current CUDA device with libgemm.

    A (M x K) and B (K x N): contiguous CUDA tensors, float32 for FP32/TF32,
    bfloat16 for BF16, float16 for FP16.  C: a contiguous float32 (M x N) CUDA tensor to
    overwrite, or None to allocate one.  Returns C.  Asynchronous on `stream`
    (default: torch's current stream).
    """
    mode, C = _operands(A, B, C, mode)
    rc = gemm_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), A.shape[0], A.shape[1], B.shape[1],
                  mode, _stream_ptr(stream))
    if rc != OK:
        raise GemmError(rc)
    return C


def gemm_ex(A, B, C=None, alpha=1.0, beta=0.0, mode=FP32, stream=None):
    """C = alpha * A @ B + beta * C with libgemm (operands as for gemm()).

    C is read when beta != 0; with C None, beta must be 0.  Returns C.
    """
    if C is None and beta != 0:
        raise ValueError("beta != 0 needs an input C")
    mode, C = _operands(A, B, C, mode)
    rc = gemm_ex_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), A.shape[0], A.shape[1],
                     B.shape[1], alpha, beta, mode, _stream_ptr(stream))
    if rc != OK:
        raise GemmError(rc, "gemm_ex")
    return C


_WANT = {}   # mode -> the operand dtype, filled at the first call


def _operands(A, B, C, mode):
    """Checks the tensors of a call; returns (mode number, C or a new C)."""
    import torch
    if isinstance(mode, str):
        mode = MODES[mode.lower()]
    if not _WANT:
        _WANT.update({FP32: torch.float32, TF32: torch.float32, BF16: torch.bfloat16,
                      FP16: torch.float16, FP32_VIA_BF16: torch.float32, TF32_RN: torch.float32})
    want = _WANT.get(mode, torch.float32)
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes {tuple(A.shape)} and {tuple(B.shape)} do not chain")
    for name, t in (("A", A), ("B", B)):
        if t.dtype != want or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {want} tensor")
    M, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif (C.dtype != torch.float32 or not C.is_cuda or not C.is_contiguous()
          or tuple(C.shape) != (M, N)):
        raise TypeError("C must be a contiguous CUDA float32 tensor of shape (M, N)")
    return mode, C


def debug_status(stream=None) -> int:
    return int(lib().gemm_debug_status(_stream_ptr(stream) or None))


def debug_build() -> bool:
    """True when the loaded library carries the device-side bounds checks."""
    return bool(lib().gemm_debug_build())


def launch_count() -> int:
    return int(lib().gemm_launch_count())


def version() -> int:
    return int(lib().gemm_version())


def selftest_bounded_wait(timeout_ns: int, stream=None) -> int:
    return int(lib().gemm_selftest_bounded_wait(int(timeout_ns), _stream_ptr(stream) or None))
