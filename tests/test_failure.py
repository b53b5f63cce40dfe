"""Failure detection without faulting the GPU.

The tensor-core pipeline waits on mbarriers.  Every such wait is bounded: when
it expires the kernel records a timeout in the device error word and returns,
and gemm_debug_status() reports it.  Here one block waits on a barrier that
nothing completes (a flag nothing sets); the wait must give up, report
GEMM_ERR_TIMEOUT, and leave the context usable for the next product.
"""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_within
from gpu_util import run

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports(libgemm):
    import torch
    import time
    t0 = time.perf_counter()
    rc = libgemm.selftest_bounded_wait(20_000_000)   # 20 ms
    dt = time.perf_counter() - t0
    assert rc == libgemm.ERR_TIMEOUT, libgemm.status_string(rc)
    assert dt < 10.0
    assert libgemm.debug_status() == libgemm.OK     # the word was cleared
    # the context is still good: a normal product runs and is right
    A, B = inputs.matrices(130, 70, 260, "pm1", seed=1)
    for mode in ("fp32", "tf32", "bf16"):
        C = run(libgemm, A, B, mode)
        Cref, S = oracle.gemm(A, B)
        assert_within(C, Cref, S, TOL[mode])
    torch.cuda.synchronize()


def test_launch_count_counts_kernels(libgemm):
    import torch
    A, B = inputs.matrices(256, 256, 256, "u01")
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.empty((256, 256), device="cuda")
    n0 = libgemm.launch_count()
    # 256^3 is a small product: one launch of the 32 x 32-tile FFMA kernel
    libgemm.gemm(a, b, c, mode=libgemm.FP32)
    assert libgemm.launch_count() - n0 == 1
    libgemm.gemm(a, b, c, mode=libgemm.TF32)                 # the MMA kernel alone (B read as stored)
    assert libgemm.launch_count() - n0 == 2
    # a K that is not a multiple of 4 floats makes the tensor path re-stride A first
    a2 = torch.from_numpy(np.ascontiguousarray(A[:, :255])).cuda()
    b2 = torch.from_numpy(np.ascontiguousarray(B[:255])).cuda()
    n1 = libgemm.launch_count()
    libgemm.gemm(a2, b2, c, mode=libgemm.TF32)
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n1 == 2
    # an N that is not a multiple of 4 floats re-strides B as well
    b3 = torch.from_numpy(np.ascontiguousarray(B[:255, :254])).cuda()
    c3 = torch.empty((256, 254), device="cuda")
    n3 = libgemm.launch_count()
    libgemm.gemm(a2, b3, c3, mode=libgemm.TF32)
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n3 == 3
    # FP32_VIA_BF16: one conversion kernel for both operands + MMA kernel when
    # their rows are whole 16-byte chunks; two conversion kernels otherwise
    n2 = libgemm.launch_count()
    libgemm.gemm(a, b, c, mode=libgemm.FP32_VIA_BF16)
    assert libgemm.launch_count() - n2 == 2
    libgemm.gemm(a2, b2, c, mode=libgemm.FP32_VIA_BF16)
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n2 == 5
    # TF32_RN: the same shape of launches with the TF32 rounding pass
    n4 = libgemm.launch_count()
    libgemm.gemm(a, b, c, mode=libgemm.TF32_RN)
    assert libgemm.launch_count() - n4 == 2
    libgemm.gemm(a2, b2, c, mode=libgemm.TF32_RN)
    torch.cuda.synchronize()
    assert libgemm.launch_count() - n4 == 5
