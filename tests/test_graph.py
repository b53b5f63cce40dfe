"""gemm() under CUDA stream capture: captured into a graph and replayed, every
mode gives the same C, bit for bit, as the same call made eagerly.

The library's per-device set-up happens at the first call on a device, so
each test makes one eager call before capturing.  Captured shapes include
ones that take scratch from the library's stream-ordered pool inside the
capture (the re-strided A of K = 777, the BF16 rounding pass, the K-split
workspaces, the FFMA stream-K form's partial tiles and counters, whose zero
fill the stream-K kernel follows by programmatic dependent launch) and so
become graph memory nodes.
"""
import numpy as np
import pytest

from accelerator_gb300 import inputs
from gpu_util import device_operands

pytestmark = pytest.mark.gpu

CASES = [("fp32", 1000, 777, 1500), ("tf32", 1000, 777, 1500), ("bf16", 1000, 777, 1500),
         ("fp16", 1000, 777, 1500), ("fp32_via_bf16", 1000, 777, 1500),
         ("tf32_rn", 1000, 777, 1500),
         ("bf16", 256, 16384, 256), ("tf32", 4096, 512, 4096), ("fp32", 256, 4096, 256),
         ("fp32", 4096, 256, 4096), ("fp32", 2048, 1024, 2048)]


@pytest.mark.parametrize("mode,M,K,N", CASES, ids=lambda v: str(v))
def test_capture_and_replay(libgemm, mode, M, K, N):
    import torch
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + N)
    a, b = device_operands(A, B, mode)
    m = libgemm.MODES[mode]
    eager = torch.empty((M, N), dtype=torch.float32, device="cuda")
    libgemm.gemm(a, b, eager, mode=m)
    torch.cuda.synchronize()
    assert libgemm.debug_status() == libgemm.OK

    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        libgemm.gemm(a, b, c, mode=m)        # on the capture stream (torch's current)
    for _ in range(2):
        c.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert libgemm.debug_status() == libgemm.OK
        np.testing.assert_array_equal(c.cpu().numpy(), eager.cpu().numpy())


def test_capture_gemm_ex(libgemm):
    import torch
    A, B = inputs.matrices(300, 9001, 203, "pm1", seed=11)
    C_in = inputs.matrix_c(300, 203, "pm1", seed=11)
    a, b = device_operands(A, B, "bf16")
    eager = torch.from_numpy(C_in.copy()).cuda()
    libgemm.gemm_ex(a, b, eager, alpha=0.5, beta=-1.5, mode=libgemm.BF16)
    torch.cuda.synchronize()
    c = torch.from_numpy(C_in.copy()).cuda()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        libgemm.gemm_ex(a, b, c, alpha=0.5, beta=-1.5, mode=libgemm.BF16)
    c.copy_(torch.from_numpy(C_in))
    graph.replay()
    torch.cuda.synchronize()
    assert libgemm.debug_status() == libgemm.OK
    np.testing.assert_array_equal(c.cpu().numpy(), eager.cpu().numpy())
