"""The two shared-memory forms of the tensor kernels' B operand give the same
C, bit for bit.  Where N is a multiple of a B box's width (32 TF32 / 64
BF16 and FP16 columns) and K of a swizzle atom's height (4 / 8 rows), B is
loaded by one 4-D TMA box per stage into atoms ordered [k group][column
block]; elsewhere, and everywhere under GEMM_FORCE_CONFIG=b_boxes_2d (read
at a process's first call on a device, so set in a child process), by 2-D
boxes per column block.  Same products, same order of summation: the child's
C must equal this process's, and both the oracle's within tolerance."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_exact, assert_within
from gpu_util import oracle_inputs, run

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# aligned for the 4-D form: whole tiles with the last round split, one tile
# split in K, a partial last tile in M and N, a short K
SHAPES = [(4096, 4096, 4096), (256, 16384, 256), (1000, 512, 1088), (640, 96, 1024)]
MODES = ["tf32", "bf16", "fp16", "tf32_rn"]

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np
from accelerator_gb300 import binding, inputs
from gpu_util import run
out = {}
for i, (M, K, N) in enumerate(%r):
    A, B = inputs.matrices(M, K, N, "pm1", seed=M + 3 * K + N)
    for mode in %r:
        out[f"{i}_{mode}"] = run(binding, A, B, mode)
np.savez(sys.argv[2], **out)
print("done")
'''


def test_b_layouts_agree(libgemm, tmp_path):
    path = str(tmp_path / "boxes2d.npz")
    env = dict(os.environ, GEMM_FORCE_CONFIG="b_boxes_2d")
    r = subprocess.run([sys.executable, "-c", CHILD % (SHAPES, MODES), ROOT, path], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    boxes2d = np.load(path)
    for i, (M, K, N) in enumerate(SHAPES):
        A, B = inputs.matrices(M, K, N, "pm1", seed=M + 3 * K + N)
        for mode in MODES:
            C = run(libgemm, A, B, mode)
            np.testing.assert_array_equal(C, boxes2d[f"{i}_{mode}"], err_msg=f"{mode} {M}x{K}x{N}")
            Ao, Bo, fmt = oracle_inputs(A, B, mode)
            if M * N * K <= 2 ** 31:
                Cref, S = oracle.gemm(Ao, Bo, fmt)
                assert_within(C, Cref, S, TOL[mode], f"{mode} {M}x{K}x{N}")
            else:
                rows, cols = inputs.sample_indices(M, N, 2048)
                Cref, S = oracle.dot(Ao, Bo, rows, cols, fmt)
                assert_within(C[rows, cols], Cref, S, TOL[mode], f"{mode} {M}x{K}x{N} sampled")


@pytest.mark.parametrize("mode", MODES)
def test_atom_layout_integers_exact(libgemm, mode):
    A, B = inputs.matrices(1000, 768, 1024, "int4", seed=8)
    C = run(libgemm, A, B, mode)
    Cref, _ = oracle.gemm(A, B)
    assert_exact(C, Cref, f"{mode} integers, atom-ordered B")
