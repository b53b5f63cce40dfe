"""Both FP32 kernels on every shape class.  The library sends small products
(at most 384^2 outputs, K <= 512) to the 32 x 32-tile kernel and the rest to
the 128 x 128-tile kernel with its K splits, so each is forced in a child
process (GEMM_FORCE_CONFIG, read once per process) and run on the ragged
sweep's shapes and on shapes the other would take, each result compared bit
for bit with the oracle's binary32 FMA chain (k ascending) wherever the
kernel keeps a tile's K range whole -- always for the 32 x 32 kernel -- and
within tolerance otherwise, with alpha / beta and C's NaN guard checked too."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import os, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from accelerator_gb300 import binding, inputs
from checks import TOL, assert_within, assert_update_within
from test_edges import _shapes

force = os.environ["GEMM_FORCE_CONFIG"]
torch.cuda.init()

def product(M, K, N, dist="pm1", alpha=1.0, beta=0.0):
    A, B = inputs.matrices(M, K, N, dist, seed=M * 7919 + K * 31 + N)
    C_in = inputs.matrix_c(M, N, seed=M + N) if beta != 0.0 else None
    buf = torch.full((M * N + 8,), float("nan"), device="cuda")
    c = buf[4:4 + M * N].view(M, N)
    if C_in is not None:
        c.copy_(torch.from_numpy(C_in).cuda())
    binding.gemm_ex(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), c, alpha=alpha,
                    beta=beta, mode=binding.FP32)
    torch.cuda.synchronize()
    assert binding.debug_status() == binding.OK
    around = torch.cat([buf[:4], buf[4 + M * N:]]).cpu().numpy()
    assert np.isnan(around).all(), f"wrote outside C {M}x{K}x{N}"
    return A, B, C_in, c.cpu().numpy()

n = 0
# the ragged sweep (K < 600): both kernels keep K whole there except the
# 128 x 128 kernel's splits of few-tile shapes, so compare within tolerance
# and, for the 32 x 32 kernel, bit for bit with the chain
for (M, K, N) in _shapes():
    A, B, _, C = product(M, K, N)
    Cref, S = oracle.gemm(A, B)
    assert_within(C, Cref, S, TOL["fp32"], f"{force} {M}x{K}x{N}")
    if force == "ffma_small":
        np.testing.assert_array_equal(C, oracle.fma_chain(A, B))
    n += 1
# shapes of the other kernel's range
big = [(1000, 777, 1500), (300, 700, 201), (513, 1025, 257), (31, 2000, 33), (1025, 96, 1031)]
small = [(128, 128, 128), (64, 500, 96), (1, 300, 1), (384, 512, 384), (200, 37, 130)]
for (M, K, N) in (big if force == "ffma_small" else small):
    A, B, _, C = product(M, K, N)
    if force == "ffma_small" or K < 128:
        np.testing.assert_array_equal(C, oracle.fma_chain(A, B), err_msg=f"{force} {M}x{K}x{N}")
    else:
        Cref, S = oracle.gemm(A, B)
        assert_within(C, Cref, S, TOL["fp32"], f"{force} {M}x{K}x{N}")
    n += 1
# alpha / beta
for (M, K, N) in [(200, 37, 130), (1000, 777, 150)]:
    A, B, C_in, C = product(M, K, N, alpha=-0.5, beta=1.5)
    P, S = oracle.gemm(A, B)
    assert_update_within(C, P, S, C_in, -0.5, 1.5, TOL["fp32"], f"{force} ex {M}x{K}x{N}")
    n += 1
print("ok", n, flush=True)
'''


@pytest.mark.parametrize("force", ["ffma_small", "ffma_tiles128"])
def test_each_fp32_kernel_on_all_shape_classes(force):
    env = dict(os.environ, GEMM_FORCE_CONFIG=force)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "ok " in r.stdout
