"""The stream-K form of the FP32 (FFMA) path, against the oracle.

Products whose 128 x 128 tiles fill between half a wave and two waves of CTA
slots (456 on a GB300), with K long enough (at least 32 slabs of 16 per
CTA), run as one persistent CTA per slot, each taking an equal share of the
tile x K-slab units; the CTA that stores a split tile's last piece adds the
pieces in K order.  Covered: a 0.56-wave square, a 1.26-wave shape, ragged M, N
and K (a partial last slab), integer inputs bit for bit, the update of
gemm_ex, run-to-run determinism, and that the two launches are taken.
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_exact, assert_update_within, assert_within
from gpu_util import device_operands, run

pytestmark = pytest.mark.gpu

# (M, K, N): 256 tiles x 128 slabs; 576 tiles x 64 slabs; 272 ragged tiles
# x 101 slabs (K = 1601: the last slab partial)
# the last: a quarter to half a wave of tiles with long K, where a tile has
# up to five pieces (those past the third added one by one)
SHAPES = [(2048, 2048, 2048), (3072, 1024, 3072), (2000, 1601, 2100), (1000, 3000, 1900)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_stream_integers_exact(libgemm, M, K, N):
    A, B = inputs.matrices(M, K, N, "int4", seed=M + K + N)
    C = run(libgemm, A, B, "fp32")
    rows, cols = inputs.sample_indices(M, N, 4096)
    Cref, _ = oracle.dot(A, B, rows, cols)
    assert_exact(C[rows, cols], Cref, f"stream-K integers {M}x{K}x{N}")
    tot, _ = oracle.total(A, B)
    assert float(np.sum(C.astype(np.float64))) == tot


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_stream_full_oracle(libgemm, M, K, N):
    A, B = inputs.matrices(M, K, N, "pm1", seed=3 * M + K)
    C = run(libgemm, A, B, "fp32")
    Cref, S = oracle.gemm(A, B)
    assert_within(C, Cref, S, TOL["fp32"], f"stream-K {M}x{K}x{N}")


def test_stream_update_and_determinism(libgemm):
    import torch
    M, K, N = 2000, 1601, 2100
    A, B = inputs.matrices(M, K, N, "pm1", seed=77)
    C_in = inputs.matrix_c(M, N, "pm1", seed=77)
    a, b = device_operands(A, B, "fp32")
    outs = []
    for _ in range(2):
        c = torch.from_numpy(C_in.copy()).cuda()
        libgemm.gemm_ex(a, b, c, alpha=0.5, beta=-1.5, mode=libgemm.FP32)
        torch.cuda.synchronize()
        assert libgemm.debug_status() == libgemm.OK
        outs.append(c.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    P, S = oracle.gemm(A, B)
    assert_update_within(outs[0], P, S, C_in, 0.5, -1.5, TOL["fp32"], "stream-K gemm_ex")


def test_stream_launches(libgemm):
    import torch
    A, B = inputs.matrices(2048, 2048, 2048, "pm1", seed=1)
    a, b = device_operands(A, B, "fp32")
    c = torch.empty((2048, 2048), device="cuda")
    n0 = libgemm.launch_count()
    libgemm.gemm(a, b, c, mode=libgemm.FP32)   # the counters' zero fill and the stream-K kernel
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n0 == 2
