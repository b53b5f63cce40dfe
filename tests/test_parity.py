"""GPU parity: libgemm through its C ABI against the fp64 oracle.

Workloads are the seeded synthetic inputs of the pages' studies:
  * 256^3 and 1024^3 with entries uniform on [0, 1);
  * the ragged 1000 x 777 x 1500 shape with entries uniform on [-1, 1), and
    the same shape with integers in [-4, 4] (exact in every mode: bit-exact);
  * the square sweep N = 128 .. 4096 (full oracle up to 1024, then 4096+
    sampled entries and the sum-of-all-elements identity);
  * 8192^3 on the tensor-core modes, uniform on [-1, 1).
FP16 (binary16 inputs, the tolerance of TF32) and TF32_RN (inputs rounded to
TF32 to nearest) ride along in every mode list.
Every element must satisfy |C - Cref| <= tol * S_ij; C is poisoned with NaN
before each launch so an unwritten element fails.
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, TOL_SAME_INPUTS, assert_exact, assert_sum, assert_within
from gpu_util import oracle_inputs, run

pytestmark = pytest.mark.gpu

MODES = ["fp32", "tf32", "bf16", "fp16", "tf32_rn"]


def _full_case(libgemm, oracle_cache, M, K, N, dist, mode):
    A, B = inputs.matrices(M, K, N, dist)
    C = run(libgemm, A, B, mode)
    Cref, S = oracle_cache.full((M, K, N, dist), A, B)
    worst = assert_within(C, Cref, S, TOL[mode], f"{mode} {M}x{K}x{N} {dist}")
    return A, B, C, worst


@pytest.mark.parametrize("mode", MODES)
def test_square_256_u01(libgemm, oracle_cache, mode):
    _full_case(libgemm, oracle_cache, 256, 256, 256, "u01", mode)


@pytest.mark.parametrize("mode", MODES)
def test_square_1024_u01(libgemm, oracle_cache, mode):
    _full_case(libgemm, oracle_cache, 1024, 1024, 1024, "u01", mode)


@pytest.mark.parametrize("mode", MODES)
def test_ragged_1000x777x1500_pm1(libgemm, oracle_cache, mode):
    _full_case(libgemm, oracle_cache, 1000, 777, 1500, "pm1", mode)


@pytest.mark.parametrize("mode", MODES + ["fp32_via_bf16"])
def test_pages_non_square_exercise(libgemm, oracle_cache, mode):
    # "Matrix Multiplication -- Naive to Tiled", section 08, exercise 1: A of
    # 512 x 768 times B of 768 x 1024, entries uniform on [0, 1)
    if mode == "fp32_via_bf16":
        A, B = inputs.matrices(512, 768, 1024, "u01")
        C = run(libgemm, A, B, mode)
        Cref, S = oracle_cache.full((512, 768, 1024, "u01"), A, B)
        assert_within(C, Cref, S, TOL[mode], "fp32_via_bf16 512x768x1024")
    else:
        _full_case(libgemm, oracle_cache, 512, 768, 1024, "u01", mode)


@pytest.mark.parametrize("mode", MODES)
def test_ragged_integers_bit_exact(libgemm, oracle_cache, mode):
    # |C| <= 777 * 16 < 2**24 and every partial sum is an integer: exact in binary32
    A, B = inputs.matrices(1000, 777, 1500, "int4")
    C = run(libgemm, A, B, mode)
    Cref, _ = oracle_cache.full((1000, 777, 1500, "int4"), A, B)
    assert_exact(C, Cref, f"{mode} integers")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [128, 512])
def test_sweep_small_full(libgemm, oracle_cache, mode, n):
    _full_case(libgemm, oracle_cache, n, n, n, "u01", mode)


@pytest.mark.parametrize("mode", ["tf32", "bf16", "fp16", "tf32_rn"])
def test_same_inputs_diagnostic(libgemm, mode):
    """Tensor path against the oracle fed the very values the tensor cores
    read (TF32-exact or BF16 values): only binary32 accumulation differs."""
    A, B = inputs.matrices(512, 1000, 384, "pm1", seed=77)
    if mode == "tf32":
        A, B = inputs.tf32_exact(A), inputs.tf32_exact(B)
    C = run(libgemm, A, B, mode)
    a, b, fmt = oracle_inputs(A, B, mode)
    Cref, S = oracle.gemm(a, b, fmt=fmt)
    assert_within(C, Cref, S, TOL_SAME_INPUTS, f"{mode} same-inputs")


def _sampled_case(libgemm, M, K, N, dist, mode, n=4096):
    A, B = inputs.matrices(M, K, N, dist)
    C = run(libgemm, A, B, mode)
    rows, cols = inputs.sample_indices(M, N, n=n)
    cref, s = oracle.dot(A, B, rows, cols)
    assert_within(C[rows, cols], cref, s, TOL[mode], f"{mode} {M}x{K}x{N} sampled")
    total, abs_total = oracle.total(A, B)
    assert_sum(C, total, abs_total, TOL[mode], f"{mode} {M}x{K}x{N} sum")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [2048, 4096])
def test_sweep_large_sampled(libgemm, mode, n):
    _sampled_case(libgemm, n, n, n, "u01", mode)


@pytest.mark.parametrize("mode", ["tf32", "bf16", "fp16", "tf32_rn"])
def test_large_8192_sampled(libgemm, mode):
    _sampled_case(libgemm, 8192, 8192, 8192, "pm1", mode)


@pytest.mark.parametrize("M,K,N", [(1000, 112, 1500), (257, 100, 383), (128, 16, 128),
                                   (4096, 64, 4096), (3, 1, 5), (2048, 240, 2048)])
def test_fp32_is_the_binary32_fma_chain(libgemm, M, K, N):
    """FP32 mode, bit for bit: each C_ij is acc = fma(A_ik, B_kj, acc), k
    ascending, wherever the library keeps a tile's K range whole: K < 128
    (under 8 slabs of 16), or a tile count between half a wave and two waves
    with fewer than 32 slabs per CTA of the stream-K form (2048 x 240 x 2048:
    256 tiles of 128 x 128, 15 slabs each)."""
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + 7 * K + 13 * N)
    C = run(libgemm, A, B, "fp32")
    np.testing.assert_array_equal(C, oracle.fma_chain(A, B))


def test_fp32_fma_chain_hand_cases(libgemm):
    from test_oracle import _chain_cases
    for case in _chain_cases():
        A = case["A"].astype(np.float32).reshape(1, -1)
        B = case["B"].astype(np.float32).reshape(-1, 1)
        C = run(libgemm, A, B, "fp32")
        assert float(C[0, 0]) == float(case["C"][0]), case["name"]


# the one-launch conversion (rows of whole 16-byte chunks) and the
# element-wise one, with whole tiles, the last round split (4096^3), all
# tiles split (256 x 16384 x 256), partial tiles and long K
VIA_BF16_SHAPES = [(1000, 777, 1500), (4096, 4096, 4096), (129, 65, 257), (1, 1, 1),
                   (640, 96, 1028), (3, 4, 4), (256, 16384, 256), (3000, 2000, 1000),
                   (8192, 512, 256), (256, 512, 8192), (2048, 8192, 2048), (1000, 4100, 1500)]


@pytest.mark.parametrize("M,K,N", VIA_BF16_SHAPES)
def test_fp32_via_bf16_equals_bf16_on_rounded_operands(libgemm, M, K, N):
    """GEMM_FP32_VIA_BF16 rounds float operands to bfloat16 on the GPU (to
    nearest, ties to even) and multiplies as GEMM_BF16: bit for bit the same
    as GEMM_BF16 on operands rounded on the host, and within the BF16
    tolerance of the oracle on the original floats (sampled entries above
    2^31 multiply-adds)."""
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + K + N)
    C = run(libgemm, A, B, "fp32_via_bf16")
    np.testing.assert_array_equal(C, run(libgemm, A, B, "bf16"))
    if M * N * K <= 2 ** 31:
        Cref, S = oracle.gemm(A, B)
        assert_within(C, Cref, S, TOL["fp32_via_bf16"], "fp32 via bf16")
    else:
        rows, cols = inputs.sample_indices(M, N, 4096)
        Cref, S = oracle.dot(A, B, rows, cols)
        assert_within(C[rows, cols], Cref, S, TOL["fp32_via_bf16"], "fp32 via bf16 sampled")



@pytest.mark.parametrize("M,K,N", [(1000, 777, 1500), (4096, 4096, 4096), (256, 16384, 256),
                                   (129, 65, 257), (640, 96, 1028)])
def test_tf32_rn_equals_tf32_on_rounded_operands(libgemm, M, K, N):
    """GEMM_TF32_RN rounds float operands to TF32 to nearest (ties away from
    zero) on the GPU and multiplies as GEMM_TF32: bit for bit GEMM_TF32 on
    operands rounded on the host the same way (one conversion launch for
    aligned rows, element-wise launches otherwise)."""
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + 3 * K + N)
    C = run(libgemm, A, B, "tf32_rn")
    np.testing.assert_array_equal(C, run(libgemm, inputs.tf32_rna(A), inputs.tf32_rna(B), "tf32"))


def test_tf32_rn_removes_the_truncation_bias(libgemm):
    """On inputs uniform on [0, 1) every truncated operand is too small, so
    GEMM_TF32's C sits below the exact product on average; rounding to
    nearest has no such bias.  Mean signed error relative to S, full C."""
    A, B = inputs.matrices(512, 2048, 512, "u01", seed=21)
    Cref, S = oracle.gemm(A, B)
    bias = {m: float(np.mean((run(libgemm, A, B, m).astype(np.float64) - Cref) / S))
            for m in ("tf32", "tf32_rn")}
    assert bias["tf32"] < -2e-4, bias            # about -2^-11 per operand, both operands
    assert abs(bias["tf32_rn"]) < 0.1 * abs(bias["tf32"]), bias
