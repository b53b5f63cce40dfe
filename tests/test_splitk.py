"""GPU parity of the tensor-core K split (shapes with too few output tiles to
fill the GPU and a long K), through the C ABI against the oracle.

Such products run as (tile, K range) units whose partial sums the library
adds in a fixed order in a second kernel, which also applies the update of
gemm_ex.  Covered here: square-ish small-MN/large-K shapes, a single-tile
shape split dozens of ways, ragged M, N and K (a partial last K slab, N not
a multiple of 4: the element-wise fix-up), run-to-run determinism, and that
the split really is taken (two kernels for an aligned BF16 product).  The
FP32 (FFMA) path splits shapes with very few tiles the same way ("wide"
split: every tile cut into up to 256 K ranges, partials added by the same
second kernel); it is covered by the same checks.

Each check can see a split piece dropped or added twice: where the oracle
is given the values the tensor cores read (TF32-truncated, bfloat16,
binary16), only the binary32 accumulation may differ, so the same-inputs
tolerance (1e-4 S) applies, well below one piece's share at any K here; and
integer inputs in [-4, 4] (every partial an integer below 2**24, exact in
any order) are compared bit for bit, in every mode, at the three split
regimes: one pair tile in 74 pieces (256 x 65536 x 256), four pair tiles
(1024 x 16384 x 1024), and the last partial round of 4096^3.
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, TOL_SAME_INPUTS, assert_exact, assert_within
from gpu_util import device_operands, oracle_inputs, run

pytestmark = pytest.mark.gpu

TC_MODES = ["tf32", "bf16", "fp16"]


def _same_inputs(A, B, mode):
    """(A, B, fmt, tol): the oracle's operands as the kernels read them, and
    the tolerance of the binary32 accumulation alone."""
    Ao, Bo, fmt = oracle_inputs(A, B, "bf16" if mode == "fp32_via_bf16" else mode)
    return Ao, Bo, fmt, min(TOL[mode], TOL_SAME_INPUTS)


def _sampled(libgemm, M, K, N, mode, dist="pm1", n=2048):
    A, B = inputs.matrices(M, K, N, dist, seed=M + K + N)
    C = run(libgemm, A, B, mode)
    Ao, Bo, fmt, tol = _same_inputs(A, B, mode)
    rows, cols = inputs.sample_indices(M, N, n)
    Cref, S = oracle.dot(Ao, Bo, rows, cols, fmt)
    assert_within(C[rows, cols], Cref, S, tol, f"{mode} {M}x{K}x{N}")
    tot, atot = oracle.total(Ao, Bo, fmt)
    got = float(np.sum(C.astype(np.float64)))
    assert abs(got - tot) <= tol * atot, (got, tot)
    return A, B, C


@pytest.mark.parametrize("mode", TC_MODES)
@pytest.mark.parametrize("M,K,N", [(1024, 16384, 1024), (256, 65536, 256), (128, 8192, 128)])
def test_small_mn_large_k(libgemm, mode, M, K, N):
    _sampled(libgemm, M, K, N, mode)


@pytest.mark.parametrize("M,K,N", [(256, 65536, 256), (128, 8192, 128)])
def test_fp32_wide_split(libgemm, M, K, N):
    _sampled(libgemm, M, K, N, "fp32")


@pytest.mark.parametrize("mode", TC_MODES + ["fp32_via_bf16", "tf32_rn", "fp32"])
@pytest.mark.parametrize("M,K,N", [(300, 9001, 203), (257, 4100, 130), (100, 5000, 77)])
def test_ragged_split_full(libgemm, mode, M, K, N):
    A, B = inputs.matrices(M, K, N, "pm1", seed=M * 3 + N)
    C = run(libgemm, A, B, mode)
    Ao, Bo, fmt, tol = _same_inputs(A, B, mode)
    Cref, S = oracle.gemm(Ao, Bo, fmt)
    assert_within(C, Cref, S, tol, f"{mode} {M}x{K}x{N}")
    # and against the original float32 values at the mode's own tolerance
    Cref, S = oracle.gemm(A, B)
    assert_within(C, Cref, S, TOL[mode], f"{mode} {M}x{K}x{N} (f32 inputs)")


ALL_MODES = ["tf32", "bf16", "fp16", "fp32", "fp32_via_bf16", "tf32_rn"]


@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("M,K,N", [(256, 65536, 256), (1024, 16384, 1024), (4096, 4096, 4096)])
def test_integers_bit_exact_at_each_split_regime(libgemm, mode, M, K, N):
    """|C| <= 16 K <= 2**20: every partial is an integer, exact in any order,
    so the split result must equal the oracle's bit for bit.  Full C for the
    single-tile split; sampled entries plus the exact sum of all entries for
    the larger shapes (a missing or doubled piece moves the sum)."""
    A, B = inputs.matrices(M, K, N, "int4", seed=M + K + N)
    C = run(libgemm, A, B, mode)
    what = f"{mode} int {M}x{K}x{N}"
    if M * N <= 256 * 256:
        Cref, _ = oracle.gemm(A, B)
        assert_exact(C, Cref, what)
    else:
        rows, cols = inputs.sample_indices(M, N, 4096)
        Cref, _ = oracle.dot(A, B, rows, cols)
        assert_exact(C[rows, cols], Cref, what + " sampled")
    tot, _ = oracle.total(A, B)
    assert float(np.sum(C.astype(np.float64))) == tot, what + " sum of all entries"


@pytest.mark.parametrize("mode", ["bf16", "tf32", "fp32"])
def test_integers_bit_exact_when_split(libgemm, mode):
    # |C| <= 16 * 8192 < 2**24 and every partial is an integer: exact in any order
    A, B = inputs.matrices(192, 8192, 320, "int4", seed=4)
    C = run(libgemm, A, B, mode)
    Cref, _ = oracle.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("mode", ["bf16", "tf32", "fp32"])
def test_split_is_deterministic(libgemm, mode):
    A, B = inputs.matrices(512, 12288, 384, "pm1", seed=9) if mode != "fp32" else \
        inputs.matrices(128, 12288, 256, "pm1", seed=9)
    first = run(libgemm, A, B, mode)
    for _ in range(2):
        np.testing.assert_array_equal(run(libgemm, A, B, mode), first)


def test_split_is_taken(libgemm):
    import torch
    A, B = inputs.matrices(256, 16384, 256, "pm1", seed=2)
    a, b = device_operands(A, B, "bf16")
    c = torch.empty((256, 256), device="cuda")
    n0 = libgemm.launch_count()
    libgemm.gemm(a, b, c, mode=libgemm.BF16)      # split MMA kernel + fix-up kernel
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n0 == 2
    n1 = libgemm.launch_count()
    A2, B2 = inputs.matrices(4096, 512, 4096, "pm1", seed=2)
    a2, b2 = device_operands(A2, B2, "bf16")
    c2 = torch.empty((4096, 4096), device="cuda")
    libgemm.gemm(a2, b2, c2, mode=libgemm.BF16)   # 256 tiles fill the GPU: no split
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n1 == 1
    a3, b3 = device_operands(A, B, "fp32")
    n2 = libgemm.launch_count()
    libgemm.gemm(a3, b3, c, mode=libgemm.FP32)    # 4 FFMA tiles: wide split + fix-up kernel
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n2 == 2


@pytest.mark.parametrize("mode", ["bf16", "tf32", "fp32"])
@pytest.mark.parametrize("N", [256, 203])
def test_split_with_update(libgemm, mode, N):
    """gemm_ex on a split product: the update is applied once, after the sum."""
    import torch
    M, K = 256, 16384
    A, B = inputs.matrices(M, K, N, "pm1", seed=N)
    C_in = inputs.matrix_c(M, N, "pm1", seed=N)
    a, b = device_operands(A, B, mode)
    c = torch.from_numpy(C_in.copy()).cuda()
    libgemm.gemm_ex(a, b, c, alpha=0.5, beta=-2.0, mode=libgemm.MODES[mode])
    torch.cuda.synchronize()
    assert libgemm.debug_status() == libgemm.OK
    out = c.cpu().numpy().astype(np.float64)
    Ao, Bo, fmt = oracle_inputs(A, B, mode)
    P, S = oracle.gemm(Ao, Bo, fmt)
    ref = oracle.update(P, C_in, 0.5, -2.0)
    lim = 0.5 * TOL[mode] * S + 2 * 2.0 ** -24 * (0.5 * S + 2 * np.abs(C_in))
    assert np.all(np.abs(out - ref) <= lim)
