"""Pins for the fp64 oracle, against facts that do not come from the oracle.

Each test is chosen so that a plausible slip in oracle.c -- a transposed
operand, a swapped index, a dropped or doubled term, a wrong sign, a wrong
widening of a format -- fails at least one of them:

  * hand-worked products (tests/golden/hand_products.txt), non-square, signed;
  * identity and permutation matrices (exact);
  * rank-1 closed forms and all-ones inputs (exact on small integers);
  * the sum identity sum_ij C_ij = sum_k colsum(A)_k rowsum(B)_k;
  * S == C on non-negative inputs, S invariant under sign flips;
  * known bit patterns of the BF16 and TF32 formats;
  * agreement with numpy's float64 matmul (a library routine) on small inputs,
    within the float64 summation bound.
CPU only.
"""
import math

import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from golden_io import hand_products, update_hand


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


@pytest.mark.parametrize("case", hand_products(), ids=lambda c: c["name"])
def test_hand_worked_products(case):
    C, S = oracle.gemm(case["A"], case["B"], fmt="f64")
    np.testing.assert_array_equal(C, case["C"])
    if "S" in case:
        np.testing.assert_array_equal(S, case["S"])
    # the same values given as float32 (all are exact in binary32)
    C32, _ = oracle.gemm(_f32(case["A"]), _f32(case["B"]), fmt="f32")
    np.testing.assert_array_equal(C32, case["C"])


@pytest.mark.parametrize("M,K,N", [(5, 7, 3), (1, 9, 4), (6, 1, 6)])
def test_identity(M, K, N):
    A, B = inputs.matrices(M, K, N, "pm1", seed=3)
    C, _ = oracle.gemm(A, np.eye(K, dtype=np.float32))
    np.testing.assert_array_equal(C, A.astype(np.float64))      # A * I = A
    C, _ = oracle.gemm(np.eye(K, dtype=np.float32), B)
    np.testing.assert_array_equal(C, B.astype(np.float64))      # I * B = B


def test_permutation():
    rng = np.random.default_rng(7)
    M, K, N = 6, 5, 8
    A, B = inputs.matrices(M, K, N, "pm1", seed=4)
    pi = rng.permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), pi] = 1.0           # (A P)[:, pi[k]] = A[:, k]
    C, _ = oracle.gemm(A, P)
    expect = np.empty((M, K))
    expect[:, pi] = A
    np.testing.assert_array_equal(C, expect)
    Q = np.zeros((K, K), np.float32)
    Q[np.arange(K), pi] = 1.0           # (Q B)[k, :] = B[pi[k], :]
    C, _ = oracle.gemm(Q, B)
    np.testing.assert_array_equal(C, B[pi].astype(np.float64))


def test_rank_one_closed_forms():
    rng = np.random.default_rng(11)
    M, K, N = 7, 13, 5
    u = rng.integers(-5, 6, M).astype(np.float32)
    v = rng.integers(-5, 6, N).astype(np.float32)
    # A = u 1^T, B = 1 v^T  ->  C_ij = K u_i v_j
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    C, _ = oracle.gemm(A, B)
    np.testing.assert_array_equal(C, K * np.outer(u, v).astype(np.float64))
    # A = u a^T, B = b v^T  ->  C = (a . b) u v^T
    a = rng.integers(-3, 4, K).astype(np.float32)
    b = rng.integers(-3, 4, K).astype(np.float32)
    C, _ = oracle.gemm(np.outer(u, a).astype(np.float32), np.outer(b, v).astype(np.float32))
    ab = float(sum(int(x) * int(y) for x, y in zip(a, b)))
    np.testing.assert_array_equal(C, ab * np.outer(u, v).astype(np.float64))


@pytest.mark.parametrize("K", [0, 1, 2, 777])
def test_all_ones(K):
    C, S = oracle.gemm(np.ones((3, K), np.float32), np.ones((K, 4), np.float32))
    np.testing.assert_array_equal(C, np.full((3, 4), float(K)))
    np.testing.assert_array_equal(S, np.full((3, 4), float(K)))


def test_empty_dims():
    C, S = oracle.gemm(np.ones((0, 3), np.float32), np.ones((3, 4), np.float32))
    assert C.shape == (0, 4) and S.shape == (0, 4)
    C, S = oracle.gemm(np.ones((2, 3), np.float32), np.ones((3, 0), np.float32))
    assert C.shape == (2, 0)
    C, S = oracle.gemm(np.ones((2, 0), np.float32), np.ones((0, 3), np.float32))
    np.testing.assert_array_equal(C, np.zeros((2, 3)))          # the empty sum
    assert oracle.total(np.ones((2, 0), np.float32), np.ones((0, 3), np.float32)) == (0.0, 0.0)


def test_sum_identity_integers():
    A, B = inputs.matrices(37, 29, 41, "int4", seed=5)
    C, S = oracle.gemm(A, B)
    t, ta = oracle.total(A, B)
    # every partial sum here is an integer below 2**53: both sides are exact
    assert t == float(np.sum(C)) and ta == float(np.sum(S))
    assert t == float(np.sum(A.astype(np.int64) @ B.astype(np.int64)))


@pytest.mark.parametrize("fmt", ["f32", "bf16", "tf32"])
def test_sum_identity_random(fmt):
    A, B = inputs.matrices(33, 65, 47, "pm1", seed=6)
    if fmt == "bf16":
        A, B = inputs.bf16_bits(A), inputs.bf16_bits(B)
    C, S = oracle.gemm(A, B, fmt=fmt)
    t, ta = oracle.total(A, B, fmt=fmt)
    assert math.isclose(t, math.fsum(C.ravel()), rel_tol=1e-12, abs_tol=1e-12 * ta)
    assert math.isclose(ta, math.fsum(S.ravel()), rel_tol=1e-12)


def test_scale_against_value():
    A, B = inputs.matrices(19, 23, 17, "u01", seed=8)
    C, S = oracle.gemm(A, B)
    np.testing.assert_array_equal(S, C)                  # all terms >= 0
    A2, B2 = inputs.matrices(19, 23, 17, "pm1", seed=8)
    C2, S2 = oracle.gemm(A2, B2)
    assert np.all(S2 >= np.abs(C2))
    Cn, Sn = oracle.gemm(-A2, B2)
    np.testing.assert_array_equal(Cn, -C2)
    np.testing.assert_array_equal(Sn, S2)
    Ca, _ = oracle.gemm(np.abs(A2), np.abs(B2))
    np.testing.assert_array_equal(Ca, S2)


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (16, 64, 16), (33, 17, 64), (64, 64, 64)])
@pytest.mark.parametrize("dist", ["u01", "pm1"])
def test_against_numpy_float64(M, K, N, dist):
    A, B = inputs.matrices(M, K, N, dist, seed=M * 1000 + N)
    C, S = oracle.gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    # two float64 sums of the same K exact products differ by at most
    # 2 * gamma_K * S with gamma_K = K u / (1 - K u), u = 2**-53
    g = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
    assert np.all(np.abs(C - ref) <= 2 * g * S + 1e-300)


def test_dot_matches_full():
    A, B = inputs.matrices(40, 50, 60, "pm1", seed=9)
    C, S = oracle.gemm(A, B)
    rows, cols = inputs.sample_indices(40, 60, n=300, seed=9)
    c, s = oracle.dot(A, B, rows, cols)
    np.testing.assert_array_equal(c, C[rows, cols])     # same k order: bit-identical
    np.testing.assert_array_equal(s, S[rows, cols])


def test_dot_rejects_bad_index():
    A, B = inputs.matrices(4, 5, 6, "u01")
    with pytest.raises(RuntimeError):
        oracle.dot(A, B, [4], [0])
    with pytest.raises(RuntimeError):
        oracle.dot(A, B, [0], [-1])


def test_thread_count_does_not_change_results():
    A, B = inputs.matrices(31, 200, 29, "pm1", seed=10)
    C1, S1 = oracle.gemm(A, B, nthreads=1)
    C4, S4 = oracle.gemm(A, B, nthreads=4)
    np.testing.assert_array_equal(C1, C4)
    np.testing.assert_array_equal(S1, S4)


def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x4049],
                    np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, (2 - 2.0 ** -7) * 2.0 ** 127,
            2.0 ** -133, 3.140625]
    got = oracle.widen(bits, "bf16")
    assert list(got) == want


def test_f16_widening_known_patterns():
    bits = np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x0400, 0x3555, 0x8000, 0x3BFF], np.uint16)
    want = [1.0, -2.0, 65504.0, 2.0 ** -24, 2.0 ** -14, 1365 / 4096, -0.0, 1 - 2.0 ** -11]
    assert list(oracle.widen(bits, "f16")) == want


def test_f16_agrees_with_numpy_half():
    # numpy's binary16 decoding is an independent implementation of the format
    bits = np.arange(0, 0x7C00, 7, dtype=np.uint16)          # finite, non-negative
    bits = np.concatenate([bits, bits | 0x8000])
    np.testing.assert_array_equal(oracle.widen(bits, "f16"),
                                  bits.view(np.float16).astype(np.float64))


def test_tf32_truncation_known_values():
    x = np.array([1.0, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -11, 1.0 + 2.0 ** -23,
                  -(1.0 + 2.0 ** -10 + 2.0 ** -11), 3.0, 2.0 ** -126 * (1 + 2.0 ** -12)],
                 np.float32)
    want = [1.0, 1.0 + 2.0 ** -10, 1.0, 1.0, -(1.0 + 2.0 ** -10), 3.0, 2.0 ** -126]
    assert list(oracle.widen(x, "tf32")) == want
    # f32 format widens unchanged
    assert list(oracle.widen(x, "f32")) == [float(v) for v in x]


def test_tf32_rna_hand_worked_patterns():
    """tests/golden/tf32_rna.txt: ties, carries into the exponent, subnormals,
    overflow to infinity, signed zeros."""
    from golden_io import tf32_rna
    rows = tf32_rna()
    x = np.array([a for a, _ in rows], np.uint32).view(np.float32)
    want = np.array([b for _, b in rows], np.uint32).view(np.float32).astype(np.float64)
    got = oracle.widen(x, "tf32rna")
    np.testing.assert_array_equal(got, want)
    assert list(np.signbit(got)) == list(np.signbit(want))


def test_tf32_rna_is_the_nearest_tf32_value():
    """For many finite binary32 values: the result is a TF32 value (no bits
    below the top 10 fraction bits), no TF32 value is nearer -- the two
    candidates are the value with the 13 low bits cleared and the next one
    up in magnitude -- and of two equally near ones the larger magnitude is
    taken."""
    rng = np.random.default_rng(7)
    u = rng.integers(0, 0x7F7FF000, size=200000, dtype=np.uint64).astype(np.uint32)
    u = np.concatenate([u, (u & np.uint32(0xFFFFE000)) | np.uint32(0x1000)])   # ties
    u = np.concatenate([u, u | np.uint32(0x80000000)])                          # negatives
    x = u.view(np.float32)
    got = oracle.widen(x, "tf32rna")
    assert np.all(np.isfinite(got))
    g32 = got.astype(np.float32)
    assert np.array_equal(g32.astype(np.float64), got)            # exact in binary32
    assert not np.any(g32.view(np.uint32) & np.uint32(0x1FFF))    # and a TF32 value
    down = (u & np.uint32(0xFFFFE000)).view(np.float32).astype(np.float64)
    up = ((u & np.uint32(0xFFFFE000)) + np.uint32(0x2000)).view(np.float32).astype(np.float64)
    xd = x.astype(np.float64)
    dd, du = np.abs(xd - down), np.abs(up - xd)
    want = np.where(du <= dd, up, down)
    np.testing.assert_array_equal(got, want)


def test_formats_agree_on_exact_inputs():
    # integers -4..4 are exact in every format, so every format gives one C
    A, B = inputs.matrices(9, 31, 11, "int4", seed=12)
    ref, _ = oracle.gemm(A, B, fmt="f32")
    for fmt, (a, b) in {"tf32": (A, B), "tf32rna": (A, B),
                        "bf16": (inputs.bf16_bits(A), inputs.bf16_bits(B)),
                        "f16": (inputs.fp16_bits(A), inputs.fp16_bits(B)),
                        "f64": (A.astype(np.float64), B.astype(np.float64))}.items():
        C, _ = oracle.gemm(a, b, fmt=fmt)
        np.testing.assert_array_equal(C, ref)


def test_rejects_bad_arguments():
    A = np.ones((2, 3), np.float32)
    with pytest.raises(ValueError):
        oracle.gemm(A, np.ones((4, 2), np.float32))
    with pytest.raises(TypeError):
        oracle.gemm(A, np.ones((3, 2), np.float64))
    with pytest.raises(ValueError):
        oracle.gemm(A, np.ones((3, 2), np.float32), fmt="fp8")


def _chain_cases():
    import os
    from golden_io import GOLDEN
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "f32_chain.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            else:
                cur[key] = np.asarray([float(v) for v in vals])
    return cases


@pytest.mark.parametrize("case", _chain_cases(), ids=lambda c: c["name"])
def test_f32_chain_hand_cases(case):
    A = case["A"].astype(np.float32).reshape(1, -1)
    B = case["B"].astype(np.float32).reshape(-1, 1)
    assert A.astype(np.float64).tolist()[0] == case["A"].tolist()      # exact in binary32
    C = oracle.fma_chain(A, B)
    assert float(C[0, 0]) == float(case["C"][0])


def test_f32_chain_exact_on_integers():
    A, B = inputs.matrices(23, 200, 17, "int4", seed=13)
    C = oracle.fma_chain(A, B)
    ref, _ = oracle.gemm(A, B)
    np.testing.assert_array_equal(C.astype(np.float64), ref)


def test_f32_chain_within_binary32_bound():
    A, B = inputs.matrices(31, 300, 29, "pm1", seed=14)
    C = oracle.fma_chain(A, B).astype(np.float64)
    ref, S = oracle.gemm(A, B)
    u = 2.0 ** -24
    g = 300 * u / (1 - 300 * u)
    assert np.all(np.abs(C - ref) <= g * S)
    assert np.any(C != ref)            # it really is binary32 arithmetic


# ---- the update C := alpha * A*B + beta * C_in (generalised product) ----

@pytest.mark.parametrize("case", update_hand(), ids=lambda c: c["name"])
def test_update_hand_cases(case):
    P, _ = oracle.gemm(case["A"], case["B"], "f64")
    out = oracle.update(P, case["C_in"], case["alpha"], case["beta"])
    np.testing.assert_array_equal(out, case["OUT"])
    P32 = P.astype(np.float32)
    out32 = oracle.update_f32(P32, case["C_in"], case["alpha"], case["beta"])
    np.testing.assert_array_equal(out32.astype(np.float64), case["OUT"])   # exact in binary32


def test_update_identity_and_empty():
    P = np.arange(12, dtype=np.float64).reshape(3, 4) - 5.5
    np.testing.assert_array_equal(oracle.update(P, None, 1.0, 0.0), P)
    np.testing.assert_array_equal(oracle.update_f32(P, None, 1.0, 0.0), P.astype(np.float32))
    assert oracle.update(np.zeros((0, 3)), None, 2.0, 0.0).shape == (0, 3)


def test_update_beta_zero_reads_no_c():
    P = np.array([[1.0, -2.0], [3.0, 0.5]])
    nan_c = np.full((2, 2), np.nan, np.float32)
    out = oracle.update(P, nan_c, 3.0, 0.0)
    np.testing.assert_array_equal(out, 3.0 * P)
    out32 = oracle.update_f32(P, nan_c, 3.0, 0.0)
    np.testing.assert_array_equal(out32, (3.0 * P).astype(np.float32))


def test_update_alpha_zero_reads_no_product():
    C_in = np.array([[1.5, -2.0, np.inf]], np.float32)
    P = np.full((1, 3), np.nan)
    np.testing.assert_array_equal(oracle.update(P, C_in, 0.0, -2.0), [[-3.0, 4.0, -np.inf]])
    np.testing.assert_array_equal(oracle.update_f32(P, C_in, 0.0, -2.0), [[-3.0, 4.0, -np.inf]])
    np.testing.assert_array_equal(oracle.update(None, C_in, 0.0, 0.0), np.zeros((1, 3)))


def test_update_f32_rounds_alpha_product_once():
    # alpha * P = 3 * (1 + 2^-23) = 3 + 1.5 * 2^-22 lies halfway between the
    # binary32 neighbours 3 + 2^-22 (odd) and 3 + 2^-21 (even): ties to even.
    P = np.array([1.0 + 2.0 ** -23], np.float32)
    out = oracle.update_f32(P, None, 3.0, 0.0)
    assert float(out[0]) == 3.0 + 2.0 ** -21
    C_in = P.copy()                       # alpha = 0: beta * C_in, the same rounding
    assert float(oracle.update_f32(None, C_in, 0.0, 3.0)[0]) == 3.0 + 2.0 ** -21


def test_update_f32_is_fused():
    # beta * C_in = (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 exactly; with t = -1 the
    # fused result is 2^-11 + 2^-24.  Rounding beta * C_in first (a tie, to
    # the even 1 + 2^-11) would give 2^-11.
    b = 1.0 + 2.0 ** -12
    out = oracle.update_f32(np.array([-1.0], np.float32), np.array([b], np.float32), 1.0, b)
    assert float(out[0]) == 2.0 ** -11 + 2.0 ** -24


def test_update_f32_within_two_roundings_of_exact():
    rng = np.random.default_rng(21)
    P = rng.standard_normal(1000).astype(np.float32)
    C_in = rng.standard_normal(1000).astype(np.float32)
    alpha, beta = np.float32(0.7), np.float32(-1.3)
    out = oracle.update_f32(P, C_in, alpha, beta).astype(np.float64)
    exact = oracle.update(P.astype(np.float64), C_in, float(alpha), float(beta))
    u = 2.0 ** -24
    bound = 2 * u * (np.abs(float(alpha) * P.astype(np.float64)) + np.abs(exact)) + 1e-45
    assert np.all(np.abs(out - exact) <= bound)


def test_update_rejects_missing_operands():
    with pytest.raises(RuntimeError):
        oracle.update(None, np.ones((2, 2), np.float32), 1.0, 1.0)
    with pytest.raises(RuntimeError):
        oracle.update_f32(np.ones((2, 2), np.float32), None, 1.0, 1.0)
