"""GPU edge cases: ragged sizes around every tile boundary, odd alignments,
empty dimensions and out-of-bounds writes.  Full oracle on every case.

Missing guards or barriers show up "only at certain matrix sizes" (second
page, "Shared Memory Tiling for Matrix Multiplication", list of traps), so
sizes straddle the kernels' tile edges: 16 (FP32 K slab), 32/64 (tensor-core
K slabs), 128 (M tiles, FP32 N tile) and 256 (tensor-core N tile).
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_exact, assert_within
from gpu_util import device_operands, run

pytestmark = pytest.mark.gpu

MODES = ["fp32", "tf32", "bf16", "fp16", "tf32_rn"]
DIMS = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 63, 65, 127, 129, 255, 257]


def _shapes(count=40, seed=5):
    rng = np.random.default_rng(seed)
    shapes = [(d, d, d) for d in DIMS]
    shapes += [tuple(int(x) for x in rng.choice(DIMS, 3)) for _ in range(count)]
    shapes += [(300, 1, 7), (1, 513, 1), (129, 2, 257), (257, 300, 1)]
    return shapes


@pytest.mark.parametrize("mode", MODES)
def test_ragged_sweep(libgemm, mode):
    for (M, K, N) in _shapes():
        A, B = inputs.matrices(M, K, N, "pm1", seed=M * 7919 + K * 31 + N)
        C = run(libgemm, A, B, mode)
        Cref, S = oracle.gemm(A, B)
        assert_within(C, Cref, S, TOL[mode], f"{mode} {M}x{K}x{N}")


@pytest.mark.parametrize("mode", MODES)
def test_ragged_sweep_integers_exact(libgemm, mode):
    for (M, K, N) in _shapes(count=15, seed=6):
        A, B = inputs.matrices(M, K, N, "int4", seed=M + 100 * K + 10000 * N)
        C = run(libgemm, A, B, mode)
        Cref, _ = oracle.gemm(A, B)
        assert_exact(C, Cref, f"{mode} {M}x{K}x{N} integers")


def _offset_view(t, shape, offset_elems):
    """A contiguous view of `shape` starting offset_elems into a fresh buffer."""
    import torch
    n = int(np.prod(shape))
    buf = torch.empty(n + offset_elems + 8, dtype=t.dtype, device=t.device)
    v = buf[offset_elems:offset_elems + n].view(*shape)
    v.copy_(t)
    return v, buf


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("which", ["A", "B", "C", "ABC"])
@pytest.mark.parametrize("M,K,N", [(200, 136, 264), (256, 8192, 200)])
def test_unaligned_bases(libgemm, mode, which, M, K, N):
    """Bases aligned to the element size only (not to 16 bytes); the long-K
    shape is split in K in every mode (workspaces and fix-up kernels)."""
    import torch
    A, B = inputs.matrices(M, K, N, "pm1", seed=21)
    a, b = device_operands(A, B, mode)
    if "A" in which:
        a, _ka = _offset_view(a, (M, K), 1)
    if "B" in which:
        b, _kb = _offset_view(b, (K, N), 1)
    c = torch.full((M, N), float("nan"), device="cuda")
    if "C" in which:
        c, _kc = _offset_view(c, (M, N), 1)
    libgemm.gemm(a, b, c, mode=libgemm.MODES[mode])
    torch.cuda.synchronize()
    Cref, S = oracle.gemm(A, B)
    assert_within(c.cpu().numpy(), Cref, S, TOL[mode], f"{mode} unaligned {which}")


@pytest.mark.parametrize("mode", MODES)
def test_no_writes_outside_c(libgemm, mode):
    """Canary bands on both sides of C stay untouched (a bounds check that
    needs no sanitizer)."""
    import torch
    for (M, K, N) in [(1000, 777, 1500), (129, 65, 257), (1, 1, 1), (255, 33, 3), (300, 9001, 203)]:
        A, B = inputs.matrices(M, K, N, "pm1", seed=3)
        a, b = device_operands(A, B, mode)
        guard = 4096
        buf = torch.full((M * N + 2 * guard,), 12345.0, device="cuda")
        c = buf[guard:guard + M * N].view(M, N)
        c.fill_(float("nan"))
        libgemm.gemm(a, b, c, mode=libgemm.MODES[mode])
        torch.cuda.synchronize()
        host = buf.cpu().numpy()
        assert np.all(host[:guard] == 12345.0), f"{mode} {M}x{K}x{N}: write before C"
        assert np.all(host[guard + M * N:] == 12345.0), f"{mode} {M}x{K}x{N}: write after C"
        Cref, S = oracle.gemm(A, B)
        assert_within(host[guard:guard + M * N].reshape(M, N), Cref, S, TOL[mode])


@pytest.mark.parametrize("mode", MODES)
def test_k_zero_is_empty_sum(libgemm, mode):
    import torch
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}.get(mode, torch.float32)
    a = torch.empty((37, 0), dtype=dt, device="cuda")
    b = torch.empty((0, 53), dtype=dt, device="cuda")
    c = torch.full((37, 53), float("nan"), device="cuda")
    libgemm.gemm(a, b, c, mode=libgemm.MODES[mode])
    torch.cuda.synchronize()
    assert torch.all(c == 0).item()


@pytest.mark.parametrize("mode", MODES)
def test_empty_m_or_n_is_noop(libgemm, mode):
    import torch
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}.get(mode, torch.float32)
    before = libgemm.launch_count()
    for (M, K, N) in [(0, 5, 7), (5, 7, 0), (0, 0, 0)]:
        a = torch.ones((M, K), dtype=dt, device="cuda")
        b = torch.ones((K, N), dtype=dt, device="cuda")
        c = torch.empty((M, N), device="cuda")
        libgemm.gemm(a, b, c, mode=libgemm.MODES[mode])
    assert libgemm.launch_count() == before


def test_identity_and_permutation_exact(libgemm):
    """Identity / permutation inputs with values exact in TF32 and BF16 give
    exact results in every mode."""
    import torch
    rng = np.random.default_rng(31)
    M = K = N = 300
    A = inputs.matrices(M, K, N, "int4", seed=8)[0] * np.float32(0.25)
    P = np.zeros((K, N), np.float32)
    P[np.arange(K), rng.permutation(N)] = 1.0
    for mode in MODES:
        C = run(libgemm, A, P, mode)
        Cref, _ = oracle.gemm(A, P)
        assert_exact(C, Cref, f"{mode} permutation")
        C = run(libgemm, np.eye(M, dtype=np.float32), A, mode)
        assert_exact(C, A.astype(np.float64), f"{mode} identity")
    del torch
