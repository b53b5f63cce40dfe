"""gemm_tf32_noalloc: the TF32 product for callers that cannot allocate
device memory (an application whose memory is all reserved for its own pool,
or a loop where an allocation must not stall or fail).  Its scratch is one
static device buffer inside the library instead of stream-ordered
allocations.

The entry point is called through the C ABI and its output compared with
gemm()'s in GEMM_TF32 on the same inputs, within the TF32 tolerance of the
parity tests (2e-3 times the oracle's scale S_ij), on two calls in a row of
different shapes -- the second call runs on a buffer that still holds the
first call's data.  Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_within

pytestmark = pytest.mark.gpu


def _noalloc(libgemm, a, b, c, M, K, N):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    return libgemm.lib().gemm_tf32_noalloc(
        ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
        ctypes.c_void_p(c.data_ptr()), M, K, N, ctypes.c_void_p(stream) if stream else None)


def test_noalloc_matches_gemm_twice(libgemm):
    import torch
    # the second shape is smaller in K and N, with a K that makes A re-strided too
    for (M, K, N, dist) in [(1024, 1024, 1536, "u01"), (700, 777, 900, "pm1")]:
        A, B = inputs.matrices(M, K, N, dist, seed=M + K + N)
        a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        c_gemm = torch.full((M, N), float("nan"), device="cuda")
        libgemm.gemm(a, b, c_gemm, mode=libgemm.TF32)
        c = torch.full((M, N), float("nan"), device="cuda")
        rc = _noalloc(libgemm, a, b, c, M, K, N)
        assert rc == libgemm.OK, libgemm.status_string(rc)
        torch.cuda.synchronize()
        assert libgemm.debug_status() == libgemm.OK
        _, S = oracle.gemm(A, B)
        got, want = c.cpu().numpy(), c_gemm.cpu().numpy().astype(np.float64)
        assert_within(got, want, S, TOL["tf32"], f"noalloc vs gemm {M}x{K}x{N}")


def test_noalloc_rejects_products_beyond_its_buffer(libgemm):
    import torch
    # B^T of 4097 x 4096 floats is just over 64 MiB
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
