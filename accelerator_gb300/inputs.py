"""Seeded synthetic inputs for the GEMM workloads.

This module serves both sides of every parity check -- the CUDA library and
the fp64 oracle -- so it holds no arithmetic of the product itself: it only
draws random matrices, encodes them in the input formats, and picks which
entries of C a sampled check looks at.  It depends on numpy alone.

Workload shapes follow the pages' studies: square N = 128 .. 4096 ("From 306 ms
to 86 ms"; "Matrix Multiplication -- Naive to Tiled", section 06), the
non-square exercise of that page's section 08 (512 x 768 times 768 x 1024),
and a ragged 1000 x 777 x 1500 shape that is a multiple of no tile size.
Base seed 42, as in the first page's host program; A and B come from
independent child streams of one numpy SeedSequence.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 42

DISTRIBUTIONS = ("u01", "pm1", "int4")


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(n)]


def _draw(rng: np.random.Generator, shape, dist: str) -> np.ndarray:
    if dist == "u01":
        # uniform on [0, 1): numpy's float32 draw never returns 1.0
        return rng.random(shape, dtype=np.float32)
    if dist == "pm1":
        # uniform on [-1, 1): 2u - 1 is exact in float32 for u = m * 2**-24
        u = rng.random(shape, dtype=np.float32)
        return (np.float32(2.0) * u - np.float32(1.0)).astype(np.float32)
    if dist == "int4":
        # integers -4 .. 4, exactly representable in fp32, tf32 and bf16
        return rng.integers(-4, 5, size=shape, dtype=np.int32).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}; expected one of {DISTRIBUTIONS}")


def matrices(M: int, K: int, N: int, dist: str = "u01", seed: int = BASE_SEED):
    """A (M x K) and B (K x N), row-major float32, from independent sub-streams."""
    ra, rb = _streams(seed, 2)
    return _draw(ra, (M, K), dist), _draw(rb, (K, N), dist)


def matrix_c(M: int, N: int, dist: str = "pm1", seed: int = BASE_SEED):
    """An input C (M x N, row-major float32) for C = alpha*A*B + beta*C, from a
    stream of its own (independent of the A and B of the same seed)."""
    (rc,) = _streams(seed + 0x5EED, 1)
    return _draw(rc, (M, N), dist)


def int_pattern(row0: int, rows: int, cols: int, a: int = 7, b: int = 3) -> np.ndarray:
    """Rows row0 .. row0 + rows - 1 of a deterministic integer matrix with
    entries ((a * i + b * k + 1) mod 9) - 4 in [-4, 4], as float32: cheap to
    make block by block for operands too large to draw at once, and exact in
    binary32, TF32, bfloat16 and binary16."""
    i = (np.arange(row0, row0 + rows, dtype=np.int64) * a) % 9
    k = (np.arange(cols, dtype=np.int64) * b + 1) % 9
    return (((i[:, None] + k[None, :]) % 9) - 4).astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (to nearest, ties to even); uint16 patterns.

    The inputs are finite, so no NaN handling is needed.  This is the input
    recipe for the BF16-input mode: both the library and the oracle receive
    the same patterns.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def sample_indices(M: int, N: int, n: int = 4096, seed: int = BASE_SEED):
    """Entries of C for a sampled check: n uniform (i, j) pairs with replacement,
    from a stream independent of the inputs' (seed + 1), plus the four corners
    and 32 evenly spaced entries each of the last row and the last column, so
    the edge tiles are always looked at.  Returns (rows, cols) as int64 arrays.
    """
    if M <= 0 or N <= 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    rows = rng.integers(0, M, size=n, dtype=np.int64)
    cols = rng.integers(0, N, size=n, dtype=np.int64)
    er = [0, 0, M - 1, M - 1]
    ec = [0, N - 1, 0, N - 1]
    for c in np.linspace(0, N - 1, num=min(32, N)).astype(np.int64):
        er.append(M - 1)
        ec.append(int(c))
    for r in np.linspace(0, M - 1, num=min(32, M)).astype(np.int64):
        er.append(int(r))
        ec.append(N - 1)
    rows = np.concatenate([rows, np.asarray(er, np.int64)])
    cols = np.concatenate([cols, np.asarray(ec, np.int64)])
    return rows, cols


def fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE binary16 (numpy's conversion: to nearest,
    ties to even); uint16 patterns.  The input recipe of the FP16-input mode:
    the library and the oracle receive the same patterns.  Values must lie
    within binary16's range (the workloads' do: |x| <= 4)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def tf32_rna(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to TF32 (10 fraction bits) to nearest, ties away
    from zero: half a TF32 unit (bit 12) added to the pattern, then the 13 low
    bits cleared (a carry moves into the exponent).  Finite inputs only.  The
    input recipe for feeding GEMM_TF32 operands rounded the way GEMM_TF32_RN
    rounds them."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x1000)) & np.uint64(0xFFFFE000)).astype(np.uint32)
    return r.view(np.float32)


def tf32_exact(x: np.ndarray) -> np.ndarray:
    """float32 values with the low 13 fraction bits cleared, so every value is
    exactly representable in TF32 and the tensor cores read it unchanged."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return u.view(np.float32)
