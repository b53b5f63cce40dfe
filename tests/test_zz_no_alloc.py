"""gemm_tf32_noalloc: the TF32 product for callers that cannot allocate
device memory (an application whose memory is all reserved for its own pool,
or a loop where an allocation must not stall or fail).  Its scratch -- the
re-strided operands and the K-split workspace gemm() would allocate -- is one
static device buffer inside the library.

Each case calls the entry point through the C ABI and checks its C against
the oracle (within the TF32 tolerance of the parity tests, 2e-3 times the
oracle's scale S_ij, or bit for bit on integer inputs) and against gemm()'s
C in GEMM_TF32 on the same inputs, bit for bit: both plan the product the
same way.  Calls follow one another on one stream, so later calls run on a
buffer that still holds an earlier call's data.  Kept in a file of its own
that pytest collects last.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_exact, assert_within

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(libgemm, a, b, c, M, K, N):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    return libgemm.lib().gemm_tf32_noalloc(
        ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
        ctypes.c_void_p(c.data_ptr()), M, K, N, ctypes.c_void_p(stream) if stream else None)


def _both(libgemm, A, B):
    """(C of gemm_tf32_noalloc, C of gemm() in TF32) on NaN-poisoned C."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c_gemm = torch.full((M, N), float("nan"), device="cuda")
    libgemm.gemm(a, b, c_gemm, mode=libgemm.TF32)
    c = torch.full((M, N), float("nan"), device="cuda")
    rc = _noalloc(libgemm, a, b, c, M, K, N)
    assert rc == libgemm.OK, libgemm.status_string(rc)
    torch.cuda.synchronize()
    assert libgemm.debug_status() == libgemm.OK
    return c.cpu().numpy(), c_gemm.cpu().numpy()


# (M, K, N, values): aligned; A and B re-strided (K, N not multiples of 4);
# one pair tile with K split in many pieces; ragged integers (bit-exact)
CASES = [(1024, 1024, 1536, "u01"), (700, 777, 902, "pm1"), (256, 16384, 256, "pm1"),
         (1000, 777, 1500, "int4")]


def test_noalloc_matches_oracle_and_gemm(libgemm):
    for (M, K, N, dist) in CASES:
        A, B = inputs.matrices(M, K, N, dist, seed=M + K + N)
        got, via_gemm = _both(libgemm, A, B)
        what = f"noalloc {M}x{K}x{N} {dist}"
        assert_exact(got, via_gemm.astype(np.float64), what + " vs gemm()")
        Cref, S = oracle.gemm(A, B)
        if dist == "int4":
            assert_exact(got, Cref, what + " vs oracle")
        else:
            assert_within(got, Cref, S, TOL["tf32"], what + " vs oracle")


def test_noalloc_4096_cube_equals_gemm(libgemm):
    """The bench size, whose last round of tiles gemm() splits in K: the same
    split, the same bits; integers in [-4, 4] checked against the oracle on
    sampled entries and the exact sum of all entries."""
    import torch
    n = 4096
    A, B = inputs.matrices(n, n, n, "int4", seed=5)
    got, via_gemm = _both(libgemm, A, B)
    assert_exact(got, via_gemm.astype(np.float64), "noalloc 4096^3 vs gemm()")
    rows, cols = inputs.sample_indices(n, n, 4096)
    Cref, _ = oracle.dot(A, B, rows, cols)
    assert_exact(got[rows, cols], Cref, "noalloc 4096^3 sampled vs oracle")
    tot, _ = oracle.total(A, B)
    assert float(np.sum(got.astype(np.float64))) == tot
    # time both entry points on the same operands (reported, not asserted)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.empty((n, n), device="cuda")
    ms = {}
    for name, call in (("gemm", lambda: libgemm.gemm(a, b, c, mode=libgemm.TF32)),
                       ("noalloc", lambda: _noalloc(libgemm, a, b, c, n, n, n))):
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            call()
        e1.record()
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / 10
    print(f"TF32 4096^3 back to back: gemm {ms['gemm']:.4f} ms, noalloc {ms['noalloc']:.4f} ms")


def test_noalloc_k_zero_writes_zeros(libgemm):
    import torch
    M, N = 96, 130
    a = torch.zeros((M, 0), device="cuda")
    b = torch.zeros((0, N), device="cuda")
    c = torch.full((M, N), float("nan"), device="cuda")
    rc = _noalloc(libgemm, a, b, c, M, 0, N)
    assert rc == libgemm.OK
    torch.cuda.synchronize()
    assert torch.all(c == 0).item()


def test_noalloc_rejects_products_beyond_its_buffer(libgemm):
    import torch
    # a re-strided B of 4096 x roundup(4097, 32) floats is just over 64 MiB
    M, K, N = 16, 4096, 4097
    a = torch.zeros((M, K), device="cuda")
    b = torch.zeros((K, N), device="cuda")
    c = torch.full((M, N), 7.0, device="cuda")
    n0 = libgemm.launch_count()
    rc = _noalloc(libgemm, a, b, c, M, K, N)
    assert rc == libgemm.ERR_SCRATCH_LIMIT
    assert libgemm.launch_count() == n0
    torch.cuda.synchronize()
    assert torch.all(c == 7.0).item()


CHILD = r'''
import ctypes, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from accelerator_gb300 import binding, inputs
for (M, K, N) in [(1000, 777, 1500), (300, 4100, 260)]:
    A, B = inputs.matrices(M, K, N, "int4", seed=M + N)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.lib().gemm_tf32_noalloc(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                         ctypes.c_void_p(c.data_ptr()), M, K, N,
                                         ctypes.c_void_p(s) if s else None)
    assert rc == 0, binding.status_string(rc)
    torch.cuda.synchronize()
    assert binding.debug_status() == 0
    Cref, _ = oracle.gemm(A, B)
    assert np.array_equal(c.cpu().numpy().astype(np.float64), Cref), (M, K, N)
    print("ok", M, K, N)
'''


def test_noalloc_single_cta_kernel():
    """The 1-SM fallback kernel (forced in a child process) through the
    no-allocation entry point, bit for bit on integer inputs."""
    env = dict(os.environ, GEMM_FORCE_CONFIG="single_cta")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok") == 2
