"""An operand of more than 2^31 elements: A of 65600 x 32800 (2.15e9 floats,
8.6 GB in FP32), so element offsets into A only fit 64-bit arithmetic, with
B of 32800 x 72.  Entries are integers in [-4, 4] (|C| <= 16 * 32800 < 2^24),
exact in every mode, so whole rows of C are compared bit for bit with the
oracle: the first rows, rows around the 2^31-element boundary of A, and the
last rows (M is not a multiple of any tile height)."""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs

pytestmark = pytest.mark.gpu

M, K, N = 65600, 32800, 72
# row 65472 straddles element 2^31 of A (offsets 2147481600 .. 2147514399);
# rows from 65473 on lie wholly beyond it
ROWS = [0, 1, 127, 128, 65471, 65472, 65473, 65536, 65598, 65599]


@pytest.fixture(scope="module")
def large_case():
    import torch
    free, _ = torch.cuda.mem_get_info()
    if free < 16 * 2 ** 30:
        pytest.skip("needs 16 GiB of free device memory")
    a32 = torch.empty((M, K), dtype=torch.float32, device="cuda")
    block = 4096
    for r0 in range(0, M, block):
        rows = min(block, M - r0)
        a32[r0:r0 + rows].copy_(torch.from_numpy(inputs.int_pattern(r0, rows, K)))
    Bh = inputs.int_pattern(0, K, N, a=5, b=2)
    b32 = torch.from_numpy(Bh).cuda()
    A_rows = np.concatenate([inputs.int_pattern(r, 1, K) for r in ROWS])
    Cref, _ = oracle.gemm(A_rows, Bh)
    yield a32, b32, Cref
    del a32, b32
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16", "fp16", "tf32_rn"])
def test_operand_beyond_2_31_elements(libgemm, large_case, mode):
    import torch
    a32, b32, Cref = large_case
    assert a32.numel() > 2 ** 31
    if mode in ("bf16", "fp16"):
        dt = torch.bfloat16 if mode == "bf16" else torch.float16
        a, b = a32.to(dt), b32.to(dt)          # integers in [-4, 4]: exact
    else:
        a, b = a32, b32
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    libgemm.gemm(a, b, c, mode=libgemm.MODES[mode])
    torch.cuda.synchronize()
    assert libgemm.debug_status() == libgemm.OK
    got = c[ROWS].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, Cref)
    assert not torch.isnan(c).any().item()
    del a, b, c
