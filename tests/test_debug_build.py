"""The debug build (GEMM_DEBUG): the same kernels with every global access
checked against the buffer it belongs to, an out-of-buffer access skipped and
reported as GEMM_ERR_BOUNDS instead of touching memory.  It stands in for a
memory checker, which cannot run where these tests run.

CPU: both variants build and say which they are.  GPU: a child process loads
the debug build and runs products along every kernel path -- FFMA interior
and edge tiles, the in-kernel split of a partial last wave and the workspace
split, the tensor kernels whole, with the last round split and all split,
the 1-SM fallback, the small-product FFMA kernel, the FFMA stream-K form, the re-stride and the
bfloat16 and TF32 rounding passes, the alpha / beta update and K = 0 -- each checked
against the oracle, with no bounds report after any of them."""
import ctypes
import os
import subprocess
import sys

import pytest

from accelerator_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_variants_report_their_kind():
    rel = ctypes.CDLL(build.build())
    dbg = ctypes.CDLL(build.build(debug=True))
    assert rel.gemm_debug_build() == 0
    assert dbg.gemm_debug_build() == 1
    for lib in (rel, dbg):
        lib.gemm_status_string.restype = ctypes.c_char_p
        assert b"debug build" in lib.gemm_status_string(8)


CHILD = r'''
import os, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np, torch
import oracle
from accelerator_gb300 import binding, inputs
from checks import TOL, assert_update_within
from gpu_util import device_operands, oracle_inputs

assert binding.debug_build(), "the debug build was not loaded"
torch.cuda.init()
single = os.environ.get("GEMM_FORCE_CONFIG") == "single_cta"

def check(mode, M, K, N, alpha=1.0, beta=0.0, sampled=False):
    A, B = inputs.matrices(M, K, N, "pm1", seed=M * 7 + K * 3 + N)
    a, b = device_operands(A, B, "fp32" if mode == "fp32_via_bf16" else mode)
    C_in = inputs.matrix_c(M, N, seed=M + N) if beta != 0.0 else None
    c = (torch.from_numpy(C_in).cuda() if C_in is not None
         else torch.full((M, N), float("nan"), device="cuda"))
    binding.gemm_ex(a, b, c, alpha=alpha, beta=beta, mode=binding.MODES[mode])
    torch.cuda.synchronize()
    st = binding.debug_status()
    assert st == binding.OK, (mode, M, K, N, binding.status_string(st))
    if mode == "fp32_via_bf16":   # the oracle sees the bfloat16 roundings
        Ao, Bo, fmt = inputs.bf16_bits(A), inputs.bf16_bits(B), "bf16"
    else:
        Ao, Bo, fmt = oracle_inputs(A, B, mode)
    C = c.cpu().numpy()
    if sampled:
        rows, cols = inputs.sample_indices(M, N, 2048)
        P, S = oracle.dot(Ao, Bo, rows, cols, fmt)
        got = C[rows, cols]
    else:
        P, S = oracle.gemm(Ao, Bo, fmt)
        got = C
    cin = None if C_in is None else (C_in[rows, cols] if sampled else C_in)
    assert_update_within(got, P, S, cin, alpha, beta, TOL[mode],
                         f"debug {mode} {M}x{K}x{N} a={alpha} b={beta}")
    print("ok", mode, M, K, N, alpha, beta, flush=True)

tc_modes = ("tf32", "bf16", "fp16")
if single:
    for mode in tc_modes:
        check(mode, 1000, 777, 1500)
        check(mode, 256, 8192, 256)
else:
    # FFMA: workspace split (few tiles), scalar B and C (N % 4 != 0), interior
    # tiles only, a partial last wave split in the kernel, alpha / beta; the
    # 32 x 32-tile kernel of small products (vector and scalar forms)
    for shp in [(1000, 777, 1500), (300, 700, 201), (2048, 64, 2048), (200, 136, 264),
                (31, 500, 33), (1030, 300, 517)]:   # the last: B re-strided, 16-byte copies
        check("fp32", *shp)
    check("fp32", 2816, 256, 2816, sampled=True)
    check("fp32", 1000, 777, 1500, alpha=0.5, beta=-1.25)
    # FFMA stream-K (a persistent CTA per slot, a split tile's pieces added
    # by the CTA of its last piece): vector and scalar B and C
    check("fp32", 2000, 1601, 2100, sampled=True)
    check("fp32", 1990, 1601, 2102, sampled=True, alpha=0.5, beta=-1.25)
    check("fp32", 1000, 3000, 1900, sampled=True)   # up to five pieces a tile
    # tensor kernels: re-strided A (K % 4 != 0), re-strided B and scalar
    # stores (N % 4 != 0),
    # all tiles split (one pair tile, long K), the last round split
    for mode in tc_modes:
        for shp in [(1000, 777, 1500), (300, 700, 201), (256, 8192, 256)]:
            check(mode, *shp)
        check(mode, 4096, 4096, 4096, sampled=True)
        check(mode, 1000, 777, 1500, alpha=2.0, beta=0.75)
    # conversion passes: vector and element-wise forms
    check("fp32_via_bf16", 640, 96, 1028)
    check("fp32_via_bf16", 300, 700, 201)
    check("tf32_rn", 640, 96, 1028)
    check("tf32_rn", 300, 700, 201)
    # K = 0: fill and scale
    for mode in ("fp32", "bf16"):
        check(mode, 64, 0, 96)
        check(mode, 64, 0, 96, alpha=1.0, beta=3.0)
print("done", flush=True)
'''


def _child(env_extra):
    env = dict(os.environ, LIBGEMM_DEBUG="1", **env_extra)
    build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-4000:]
    assert "done" in r.stdout
    return r.stdout


@pytest.mark.gpu
def test_debug_build_all_paths_in_bounds():
    out = _child({})
    assert out.count("ok ") == 34


@pytest.mark.gpu
def test_debug_build_single_cta_in_bounds():
    out = _child({"GEMM_FORCE_CONFIG": "single_cta"})
    assert out.count("ok ") == 6
