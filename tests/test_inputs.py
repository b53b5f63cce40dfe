"""The seeded input generators: determinism, ranges and the BF16 encoding. CPU only."""
import numpy as np
import pytest

from accelerator_gb300 import inputs


def test_deterministic_and_independent():
    A1, B1 = inputs.matrices(64, 32, 48, "u01")
    A2, B2 = inputs.matrices(64, 32, 48, "u01")
    np.testing.assert_array_equal(A1, A2)
    np.testing.assert_array_equal(B1, B2)
    A3, _ = inputs.matrices(64, 32, 48, "u01", seed=43)
    assert not np.array_equal(A1, A3)
    # A and B come from different streams
    assert not np.array_equal(A1[:32, :32], B1[:32, :32])


@pytest.mark.parametrize("dist,lo,hi", [("u01", 0.0, 1.0), ("pm1", -1.0, 1.0)])
def test_uniform_ranges(dist, lo, hi):
    A, B = inputs.matrices(300, 400, 500, dist)
    for X in (A, B):
        assert X.dtype == np.float32 and X.flags.c_contiguous
        assert X.min() >= lo and X.max() < hi
        assert abs(float(X.mean()) - (lo + hi) / 2) < 0.01


def test_int4_values():
    A, B = inputs.matrices(100, 777, 150, "int4")
    vals = np.unique(np.concatenate([A.ravel(), B.ravel()]))
    np.testing.assert_array_equal(vals, np.arange(-4, 5, dtype=np.float32))


def test_bf16_round_to_nearest_even():
    x = np.array([
        1.0,                       # exact
        1.0 + 2.0 ** -8,           # halfway between 1 and 1+2^-7: ties to even -> 1
        1.0 + 3 * 2.0 ** -8,       # halfway, odd below -> up to 1 + 2^-6
        1.0 + 2.0 ** -8 + 2.0 ** -20,  # just above halfway -> up
        -1.0 - 2.0 ** -9,          # below halfway -> -1
        3.0e38,                    # large, finite
    ], np.float32)
    got = inputs.bf16_bits(x)
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xBF80]
    assert [int(v) for v in got[:5]] == want
    # round trip of the large value: relative error below 2^-8
    back = (got[5:].astype(np.uint32) << 16).view(np.float32)
    assert abs(float(back[0]) / 3.0e38 - 1) < 2.0 ** -8


def _bf16_nearest_even_by_definition(x):
    """The bfloat16 value nearest to each float32 x, ties to the even
    significand, found from the two neighbouring bfloat16 values (the
    truncation and the next one up in magnitude) compared in float64, where
    both distances are exact: no rounding trick on the bit pattern."""
    u = x.view(np.uint32)
    lo = (u & np.uint32(0xFFFF0000))                     # toward zero
    hi = lo + np.uint32(0x10000)                         # next in magnitude
    flo = lo.view(np.float32).astype(np.float64)
    fhi = hi.view(np.float32).astype(np.float64)
    fx = x.astype(np.float64)
    dlo, dhi = np.abs(fx - flo), np.abs(fhi - fx)
    even_lo = ((lo >> np.uint32(16)) & np.uint32(1)) == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ~even_lo)
    return np.where(pick_hi, hi, lo) >> np.uint32(16)


def test_bf16_matches_nearest_even_definition():
    rng = np.random.default_rng(11)
    # finite patterns whose next bfloat16 up is still finite
    u = rng.integers(0, 0x7F7F0000, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (u & np.uint32(0xFFFF0000)) | np.uint32(0x8000)          # exactly halfway
    carries = np.uint32(0x3F80FFFF) + np.zeros(1, np.uint32)        # rounds into the next binade
    subnormal = rng.integers(1, 0x007FFFFF, size=2000, dtype=np.uint64).astype(np.uint32)
    u = np.concatenate([u, ties, carries, subnormal, np.array([0x3FFF8000, 0x3FFFFFFF], np.uint32)])
    u = np.concatenate([u, u | np.uint32(0x80000000)])              # and the negatives
    x = u.view(np.float32)
    got = inputs.bf16_bits(x).astype(np.uint32)
    np.testing.assert_array_equal(got, _bf16_nearest_even_by_definition(x))


def test_tf32_rna_recipe_matches_the_oracle_format():
    """The host-side TF32 rounding recipe (a bit trick) and the oracle's
    format (the grid definition) agree on finite values, ties included."""
    import oracle
    rng = np.random.default_rng(3)
    u = rng.integers(0, 0x7F7FE000, size=100000, dtype=np.uint64).astype(np.uint32)
    u = np.concatenate([u, (u & np.uint32(0xFFFFE000)) | np.uint32(0x1000)])
    u = np.concatenate([u, u | np.uint32(0x80000000)])
    x = u.view(np.float32).reshape(1, -1)
    np.testing.assert_array_equal(inputs.tf32_rna(x).astype(np.float64), oracle.widen(x, "tf32rna"))


def test_sample_indices_cover_edges():
    rows, cols = inputs.sample_indices(1000, 1500, n=4096)
    assert rows.dtype == np.int64 and rows.shape == cols.shape
    assert rows.min() >= 0 and rows.max() == 999 and cols.min() >= 0 and cols.max() == 1499
    pairs = set(zip(rows.tolist(), cols.tolist()))
    for corner in [(0, 0), (0, 1499), (999, 0), (999, 1499)]:
        assert corner in pairs
    r2, c2 = inputs.sample_indices(1000, 1500, n=4096)
    np.testing.assert_array_equal(rows, r2)
    np.testing.assert_array_equal(cols, c2)
    r0, c0 = inputs.sample_indices(0, 5)
    assert r0.size == 0 and c0.size == 0
