"""The 1-SM tensor-core kernel, the fallback for devices that cannot hold
clusters of two CTAs, checked against the oracle on a GB300 by forcing it
with GEMM_FORCE_CONFIG=single_cta in a child process (the choice is made once
per process, at the first call on a device)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from accelerator_gb300 import binding, inputs
from checks import TOL, assert_within
from gpu_util import run, oracle_inputs
for (M, K, N) in [(1000, 777, 1500), (256, 8192, 256), (2048, 512, 2048)]:
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + N)
    for mode in ("tf32", "bf16", "fp16"):
        n0 = binding.launch_count()
        C = run(binding, A, B, mode)
        Ao, Bo, fmt = oracle_inputs(A, B, mode)
        Cref, S = oracle.gemm(Ao, Bo, fmt)
        assert_within(C, Cref, S, TOL[mode], f"1-SM {mode} {M}x{K}x{N}")
        print("ok", mode, M, K, N, binding.launch_count() - n0)
'''


def test_single_cta_kernel_parity():
    env = dict(os.environ, GEMM_FORCE_CONFIG="single_cta")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok") == 9
