"""Comparison helpers shared by the GPU parity tests.

Tolerances (relative to the scale S_ij = sum_k |A_ik B_kj| the oracle returns):
FP32 1e-5, TF32 2e-3, BF16 1e-2 against the oracle on the original float32
values; integer-valued inputs small enough to stay exact must match bit for
bit in every mode.
"""
from __future__ import annotations

import numpy as np

TOL = {"fp32": 1e-5, "tf32": 2e-3, "bf16": 1e-2, "fp16": 2e-3, "fp32_via_bf16": 1e-2,
       "tf32_rn": 2e-3}

# Diagnostic tolerances when the oracle sees the same rounded inputs as the
# tensor cores (TF32-truncated or BF16 values): only the binary32
# accumulation differs, bounded by about K * 2**-24 relative to S; 1e-4
# leaves room for K up to ~1600 in the worst case and far more on average.
TOL_SAME_INPUTS = 1e-4


def assert_within(C, Cref, S, tol, what=""):
    C = np.asarray(C, dtype=np.float64)
    assert C.shape == Cref.shape, (C.shape, Cref.shape)
    finite = np.isfinite(C)
    if not finite.all():
        idx = np.argwhere(~finite)[:5]
        raise AssertionError(f"{what}: {int((~finite).sum())} non-finite entries, e.g. at {idx.tolist()}")
    err = np.abs(C - Cref)
    lim = tol * S
    bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)[:5]
        rows = [(tuple(i), C[tuple(i)], Cref[tuple(i)], S[tuple(i)]) for i in idx]
        worst = float(np.max(err / np.where(S > 0, S, 1)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries off by more than "
                             f"{tol}*S (worst |dC|/S = {worst:.3e}); e.g. (idx, got, want, S): {rows}")
    return float(np.max(err / np.where(S > 0, S, 1))) if err.size else 0.0


def assert_sum(C, total, abs_total, tol, what=""):
    """Sum of all entries of C (fp64) against the oracle's sum identity."""
    got = float(np.sum(np.asarray(C, dtype=np.float64)))
    assert abs(got - total) <= tol * abs_total, (
        f"{what}: sum of C = {got!r}, oracle {total!r}, allowed {tol * abs_total!r}")


def assert_exact(C, Cref, what=""):
    C = np.asarray(C, dtype=np.float64)
    if not np.array_equal(C, Cref):
        bad = np.argwhere(C != Cref)[:5]
        raise AssertionError(f"{what}: {int((C != Cref).sum())} entries differ, e.g. "
                             f"{[(tuple(i), C[tuple(i)], Cref[tuple(i)]) for i in bad]}")


U = 2.0 ** -24   # unit roundoff of binary32


def assert_update_within(out, P, S, C_in, alpha, beta, tol, what):
    """|out - (alpha P + beta C_in)| <= |alpha| tol S plus the epilogue's own
    two roundings, 2u (|alpha| S + |beta C_in|) (|P| <= S)."""
    import oracle
    ref = oracle.update(P, C_in, alpha, beta)
    out = np.asarray(out, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite entries"
    c_abs = 0.0 if C_in is None else np.abs(C_in)
    lim = abs(alpha) * tol * S + 2 * U * (abs(alpha) * S + abs(beta) * c_abs) + 1e-30
    err = np.abs(out - ref)
    bad = err > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} entries off, e.g. "
                           f"{[(tuple(i), out[tuple(i)], ref[tuple(i)]) for i in np.argwhere(bad)[:4]]}")
