"""Concurrent callers: in a fresh process, 8 host threads make their first
library calls at the same moment (racing the per-device set-up), each on its
own CUDA stream, in mixed modes and shapes (some taking scratch from the
library's pool, some split in K), then call again; every result must match
the oracle.  ctypes releases the GIL during the calls, so they really
overlap on the host, and the streams let the kernels overlap on the GPU."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from accelerator_gb300 import binding, inputs
from checks import TOL, assert_within
from gpu_util import device_operands, oracle_inputs

torch.cuda.init()
jobs = [("fp32", 300, 700, 200), ("tf32", 257, 130, 261), ("bf16", 1000, 777, 1500),
        ("fp16", 256, 8192, 256), ("fp32_via_bf16", 640, 96, 1028), ("tf32", 256, 16384, 256),
        ("fp32", 128, 4096, 128), ("bf16", 512, 768, 1024), ("tf32_rn", 700, 512, 900),
        ("fp32", 2048, 1024, 2048)]
prepared = []
for i, (mode, M, K, N) in enumerate(jobs):
    A, B = inputs.matrices(M, K, N, "pm1", seed=100 + i)
    a, b = device_operands(A, B, "fp32" if mode == "fp32_via_bf16" else mode)
    prepared.append((mode, A, B, a, b, torch.cuda.Stream()))
torch.cuda.synchronize()
barrier = threading.Barrier(len(jobs))
results, errors = [None] * len(jobs), []

def work(i):
    mode, A, B, a, b, s = prepared[i]
    try:
        barrier.wait()
        outs = []
        for _ in range(2):
            c = torch.full((A.shape[0], B.shape[1]), float("nan"), device="cuda")
            with torch.cuda.stream(s):
                binding.gemm(a, b, c, mode=binding.MODES[mode], stream=s)
            outs.append(c)
        s.synchronize()
        results[i] = [o.cpu().numpy() for o in outs]
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
for t in threads: t.start()
for t in threads: t.join()
assert not errors, errors
assert binding.debug_status() == binding.OK
for i, (mode, A, B, a, b, s) in enumerate(prepared):
    Ao, Bo, fmt = (A, B, "f32") if mode == "fp32_via_bf16" else oracle_inputs(A, B, mode)
    Cref, S = oracle.gemm(Ao, Bo, fmt)
    for C in results[i]:
        assert_within(C, Cref, S, TOL[mode], f"thread {i} {mode}")
    np.testing.assert_array_equal(results[i][0], results[i][1])
print("ok", len(jobs))
'''


def test_concurrent_first_calls_and_streams():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "ok 10" in r.stdout
