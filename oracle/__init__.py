"""fp64 CPU oracle for C = A*B -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import this package.
The product library never does, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain triple loop in double, k
ascending); this module only compiles it with gcc and marshals numpy arrays.
The definition it follows is the opening formula of "Shared Memory Tiling for
Matrix Multiplication": C_ij = sum_k A_ik * B_kj, with the row-major indexing
of "Matrix Multiplication -- Naive to Tiled", section 02.

Input formats (``fmt``):
  "f32"   float32 values, widened exactly;
  "bf16"  uint16 bfloat16 bit patterns, widened exactly;
  "tf32"  float32 with the low 13 fraction bits cleared, then widened
          (a diagnostic for the TF32 tensor path);
  "f64"   float64 values as given;
  "f16"   uint16 IEEE binary16 bit patterns, widened exactly;
  "tf32rna"  float32 rounded to the nearest TF32 value (10 fraction bits),
          ties away from zero, then widened.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

_FMT = {"f32": 0, "bf16": 1, "tf32": 2, "f64": 3, "f16": 4, "tf32rna": 5}
_DTYPE = {"f32": np.float32, "bf16": np.uint16, "tf32": np.float32, "f64": np.float64,
          "f16": np.uint16, "tf32rna": np.float32}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, no fp contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [ip, vp, vp, i64, i64, i64, dp, dp, ip]
            lib.oracle_dot.argtypes = [ip, vp, vp, i64, i64, i64, vp, vp, i64, dp, dp, ip]
            lib.oracle_sum.argtypes = [ip, vp, vp, i64, i64, i64, dp, dp]
            lib.oracle_widen.argtypes = [ip, vp, i64, dp]
            lib.oracle_threads.argtypes = [ip]
            lib.oracle_gemm_f32_chain.argtypes = [vp, vp, i64, i64, i64, vp, ip]
            lib.oracle_gemm_f32_chain.restype = ctypes.c_int
            lib.oracle_update.argtypes = [vp, vp, i64, ctypes.c_double, ctypes.c_double, vp]
            lib.oracle_update.restype = ctypes.c_int
            lib.oracle_update_f32.argtypes = [vp, vp, i64, ctypes.c_float, ctypes.c_float, vp]
            lib.oracle_update_f32.restype = ctypes.c_int
            for f in (lib.oracle_gemm, lib.oracle_dot, lib.oracle_sum,
                      lib.oracle_widen, lib.oracle_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_input(x: np.ndarray, fmt: str) -> np.ndarray:
    if fmt not in _FMT:
        raise ValueError(f"unknown oracle format {fmt!r}")
    x = np.asarray(x)
    if x.ndim != 2:
        raise ValueError("oracle inputs are 2-D matrices")
    if x.dtype != _DTYPE[fmt]:
        raise TypeError(f"format {fmt!r} wants dtype {np.dtype(_DTYPE[fmt])}, got {x.dtype}")
    return np.ascontiguousarray(x)


def _ptr(x: np.ndarray):
    return x.ctypes.data_as(ctypes.c_void_p)


def _dims(A: np.ndarray, B: np.ndarray):
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    return M, K, N


def threads(nthreads: int = 0) -> int:
    """Threads the oracle's parallel loops use (0 = OpenMP's default)."""
    return int(_load().oracle_threads(int(nthreads)))


def gemm(A: np.ndarray, B: np.ndarray, fmt: str = "f32", nthreads: int = 0):
    """Full product. Returns (C, S): C_ij = sum_k A_ik B_kj, S_ij = sum_k |A_ik B_kj|."""
    A, B = _as_input(A, fmt), _as_input(B, fmt)
    M, K, N = _dims(A, B)
    C = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    rc = _load().oracle_gemm(_FMT[fmt], _ptr(A), _ptr(B), M, K, N, _ptr(C), _ptr(S), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm failed")
    return C, S


def fma_chain(A: np.ndarray, B: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """float32 C with C_ij = the binary32 chain acc = fma(A_ik, B_kj, acc), k ascending."""
    A, B = _as_input(A, "f32"), _as_input(B, "f32")
    M, K, N = _dims(A, B)
    C = np.empty((M, N), np.float32)
    if _load().oracle_gemm_f32_chain(_ptr(A), _ptr(B), M, K, N, _ptr(C), int(nthreads)) != 0:
        raise RuntimeError("oracle_gemm_f32_chain failed")
    return C


def dot(A: np.ndarray, B: np.ndarray, rows, cols, fmt: str = "f32", nthreads: int = 0):
    """Chosen entries only. Returns (C[t], S[t]) for t-th pair (rows[t], cols[t])."""
    A, B = _as_input(A, fmt), _as_input(B, fmt)
    M, K, N = _dims(A, B)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    n = rows.shape[0]
    C = np.empty(n, np.float64)
    S = np.empty(n, np.float64)
    rc = _load().oracle_dot(_FMT[fmt], _ptr(A), _ptr(B), M, K, N, _ptr(rows), _ptr(cols), n,
                            _ptr(C), _ptr(S), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_dot failed (bad index or argument)")
    return C, S


def total(A: np.ndarray, B: np.ndarray, fmt: str = "f32"):
    """(sum of all C_ij, sum of all S_ij) computed as sum_k colsum(A)_k * rowsum(B)_k."""
    A, B = _as_input(A, fmt), _as_input(B, fmt)
    M, K, N = _dims(A, B)
    t = ctypes.c_double()
    ta = ctypes.c_double()
    rc = _load().oracle_sum(_FMT[fmt], _ptr(A), _ptr(B), M, K, N,
                            ctypes.byref(t), ctypes.byref(ta))
    if rc != 0:
        raise RuntimeError("oracle_sum failed")
    return t.value, ta.value


def widen(x: np.ndarray, fmt: str) -> np.ndarray:
    """Exact double value of each input element under format fmt."""
    x = np.ascontiguousarray(x, dtype=_DTYPE[fmt])
    out = np.empty(x.shape, np.float64)
    rc = _load().oracle_widen(_FMT[fmt], _ptr(x), x.size, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_widen failed")
    return out


def update(P, C_in, alpha: float, beta: float) -> np.ndarray:
    """alpha * P + beta * C_in in double (P the product, C_in the old C).

    beta == 0 reads no C_in and alpha == 0 reads no P: pass None there.
    """
    ref = P if P is not None else C_in
    shape = np.shape(ref)
    n = int(np.prod(shape))
    Pd = None if P is None else np.ascontiguousarray(P, dtype=np.float64)
    Cf = None if C_in is None else np.ascontiguousarray(C_in, dtype=np.float32)
    out = np.empty(shape, np.float64)
    rc = _load().oracle_update(None if Pd is None else _ptr(Pd), None if Cf is None else _ptr(Cf),
                               n, float(alpha), float(beta), _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_update failed")
    return out


def update_f32(P, C_in, alpha: float, beta: float) -> np.ndarray:
    """The binary32 update fmaf(beta, C_in, alpha * P) (see oracle_update_f32)."""
    ref = P if P is not None else C_in
    shape = np.shape(ref)
    n = int(np.prod(shape))
    Pf = None if P is None else np.ascontiguousarray(P, dtype=np.float32)
    Cf = None if C_in is None else np.ascontiguousarray(C_in, dtype=np.float32)
    out = np.empty(shape, np.float32)
    rc = _load().oracle_update_f32(None if Pf is None else _ptr(Pf),
                                   None if Cf is None else _ptr(Cf), n, float(alpha), float(beta),
                                   _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_update_f32 failed")
    return out
