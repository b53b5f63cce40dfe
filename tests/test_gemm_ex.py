"""GPU parity of gemm_ex, C = alpha*A*B + beta*C, through the C ABI against
the oracle's update (oracle.update in fp64, oracle.update_f32 for the exact
binary32 reading) on seeded inputs.

The generalised product is the one of the cuBLAS call in "Matrix
Multiplication -- Naive to Tiled", section 07.  Every mode is covered on a
shape of several tiles with a ragged tail (vector epilogue) and on one whose
N is odd (scalar epilogue), for the kinds of update the library
distinguishes: alpha only, alpha and beta, beta only (alpha == 0), and the
plain product (alpha == 1, beta == 0), which must equal gemm() bit for bit.
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_update_within
from gpu_util import device_operands, oracle_inputs, run

pytestmark = pytest.mark.gpu

MODES = ["fp32", "tf32", "bf16", "fp16", "fp32_via_bf16", "tf32_rn"]
# (520, 96, 1027): K too short to split, so the tensor kernel itself writes
# C, whose rows (N % 4 = 3) take the row-by-row staged stores
SHAPES = [(300, 200, 520), (257, 130, 261), (520, 96, 1027)]
SCALARS = [(1.0, 0.0), (2.5, 0.0), (-0.75, 1.5), (1.0, 1.0), (0.0, -2.0), (0.0, 0.0), (0.0, 1.0)]


def run_ex(binding, A, B, C_in, alpha, beta, mode):
    """gemm_ex on cuda:0 with C starting as C_in; returns the new C on the host."""
    import torch
    a, b = device_operands(A, B, "fp32" if mode == "fp32_via_bf16" else mode)
    c = torch.from_numpy(np.ascontiguousarray(C_in, np.float32)).cuda()
    binding.gemm_ex(a, b, c, alpha=alpha, beta=beta, mode=binding.MODES[mode])
    torch.cuda.synchronize()
    assert binding.debug_status() == binding.OK
    return c.cpu().numpy()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("alpha,beta", SCALARS)
def test_gemm_ex_against_oracle(libgemm, mode, M, K, N, alpha, beta):
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + K + N)
    C_in = inputs.matrix_c(M, N, "pm1", seed=M + K + N)
    out = run_ex(libgemm, A, B, C_in, alpha, beta, mode)
    if mode == "fp32_via_bf16":
        Ao, Bo, fmt = A, B, "f32"
    else:
        Ao, Bo, fmt = oracle_inputs(A, B, mode)
    P, S = oracle.gemm(Ao, Bo, fmt)
    assert_update_within(out, P, S, C_in, alpha, beta, TOL[mode], f"{mode} a={alpha} b={beta}")
    if alpha == 1.0 and beta == 0.0:
        np.testing.assert_array_equal(out, run(libgemm, A, B, mode))


@pytest.mark.parametrize("M,K,N", [(300, 100, 520), (257, 112, 261), (3, 1, 5)])
@pytest.mark.parametrize("alpha,beta", [(2.5, 0.0), (-0.75, 1.5), (3.0, -1.0)])
def test_fp32_update_is_the_binary32_reading(libgemm, M, K, N, alpha, beta):
    """FP32 mode, bit for bit: fma(beta, C, alpha * acc) with acc the binary32
    FMA chain (K < 128 keeps every tile's K range whole)."""
    A, B = inputs.matrices(M, K, N, "pm1", seed=3 * M + K)
    C_in = inputs.matrix_c(M, N, "pm1", seed=3 * M + K)
    out = run_ex(libgemm, A, B, C_in, alpha, beta, "fp32")
    want = oracle.update_f32(oracle.fma_chain(A, B), C_in, alpha, beta)
    np.testing.assert_array_equal(out, want)


@pytest.mark.parametrize("mode", ["fp32", "bf16", "tf32"])
def test_beta_zero_reads_no_c(libgemm, mode):
    A, B = inputs.matrices(200, 96, 264, "pm1", seed=5)
    C_in = np.full((200, 264), np.nan, np.float32)
    out = run_ex(libgemm, A, B, C_in, -1.25, 0.0, mode)
    Ao, Bo, fmt = oracle_inputs(A, B, mode)
    P, S = oracle.gemm(Ao, Bo, fmt)
    assert_update_within(out, P, S, None, -1.25, 0.0, TOL[mode], f"{mode} beta=0 over NaN C")


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_alpha_zero_reads_no_operands(libgemm, mode):
    A, B = inputs.matrices(64, 32, 96, "pm1", seed=6)
    A[:] = np.nan
    C_in = inputs.matrix_c(64, 96, "pm1", seed=6)
    out = run_ex(libgemm, A, B, C_in, 0.0, -3.0, mode)
    np.testing.assert_array_equal(out, oracle.update_f32(None, C_in, 0.0, -3.0))


@pytest.mark.parametrize("alpha,beta", [(2.0, 0.5), (0.0, 0.0), (1.0, 1.0)])
def test_k_zero_is_beta_c(libgemm, alpha, beta):
    import torch
    C_in = inputs.matrix_c(33, 45, "pm1", seed=8)
    c = torch.from_numpy(C_in.copy()).cuda()
    a = torch.empty((33, 0), dtype=torch.float32, device="cuda")
    b = torch.empty((0, 45), dtype=torch.float32, device="cuda")
    libgemm.gemm_ex(a, b, c, alpha=alpha, beta=beta, mode=libgemm.FP32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(c.cpu().numpy(), oracle.update_f32(None, C_in, 0.0, beta))


@pytest.mark.parametrize("mode", ["fp32", "bf16", "tf32"])
def test_split_and_large_shapes(libgemm, mode):
    """Shapes whose tiles are all split in K (640 x 2048 x 640), none
    (2048^3), and only the last wave's or round's (4096^3: the whole tiles
    apply the update in the GEMM kernel, the split ones after the partials
    are added), checked on sampled entries, corners and last row and column
    included."""
    for (M, K, N) in [(640, 2048, 640), (2048, 2048, 2048), (4096, 4096, 4096)]:
        A, B = inputs.matrices(M, K, N, "pm1", seed=K + 1)
        C_in = inputs.matrix_c(M, N, "pm1", seed=K + 1)
        out = run_ex(libgemm, A, B, C_in, 0.5, -2.0, mode)
        Ao, Bo, fmt = oracle_inputs(A, B, mode)
        rows, cols = inputs.sample_indices(M, N, 2048)
        P, S = oracle.dot(Ao, Bo, rows, cols, fmt)
        assert_update_within(out[rows, cols], P, S, C_in[rows, cols], 0.5, -2.0, TOL[mode],
                             f"{mode} {M}x{K}x{N}")
