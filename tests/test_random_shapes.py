"""Seeded random products: shapes up to 3000 (K up to 6000 when M*N is
small), all six modes, random alpha and beta, and operands and C placed at
element offsets 0..2 inside larger buffers, so bases that are aligned to the
element but not to 16 bytes are covered along with every split and edge
path the shapes happen to take.  Each result is compared with the oracle
(sampled entries above 3e8 multiply-adds) and the elements around C must keep
their NaN poison."""
import numpy as np
import pytest

import oracle
from accelerator_gb300 import inputs
from checks import TOL, assert_update_within

pytestmark = pytest.mark.gpu

MODES = ("fp32", "tf32", "bf16", "fp16", "fp32_via_bf16", "tf32_rn")


def _cases(seed, n, p_big):
    rng = np.random.default_rng(seed)
    for case in range(n):
        big = rng.random() < p_big
        M = int(rng.integers(1, 3000 if big else 600))
        N = int(rng.integers(1, 3000 if big else 600))
        long_k = M * N < 40000 and rng.random() < 0.5
        K = int(rng.integers(0, 6000 if long_k else 900))
        mode = MODES[int(rng.integers(0, len(MODES)))]
        alpha = float(rng.choice([1.0, 0.5, -2.0, 0.0])) if rng.random() < 0.3 else 1.0
        beta = float(rng.choice([0.0, 1.0, -0.75])) if rng.random() < 0.3 else 0.0
        offs = tuple(int(rng.integers(0, 3)) for _ in range(3))
        yield case, M, K, N, mode, alpha, beta, offs


def _operands(A, B, mode):
    import torch
    if mode == "bf16":
        return (torch.from_numpy(inputs.bf16_bits(A).view(np.int16)).view(torch.bfloat16),
                torch.from_numpy(inputs.bf16_bits(B).view(np.int16)).view(torch.bfloat16),
                inputs.bf16_bits(A), inputs.bf16_bits(B), "bf16")
    if mode == "fp16":
        return (torch.from_numpy(inputs.fp16_bits(A).view(np.int16)).view(torch.float16),
                torch.from_numpy(inputs.fp16_bits(B).view(np.int16)).view(torch.float16),
                inputs.fp16_bits(A), inputs.fp16_bits(B), "f16")
    if mode == "fp32_via_bf16":   # the oracle sees the bfloat16 roundings
        return (torch.from_numpy(A), torch.from_numpy(B), inputs.bf16_bits(A),
                inputs.bf16_bits(B), "bf16")
    fmt = {"tf32": "tf32", "tf32_rn": "tf32rna"}.get(mode, "f32")
    return torch.from_numpy(A), torch.from_numpy(B), A, B, fmt


def _placed(host, offset, shape):
    """A CUDA view of `shape` starting `offset` elements into a larger buffer."""
    import torch
    n = int(np.prod(shape))
    buf = torch.empty(n + offset + 1, dtype=host.dtype, device="cuda")
    view = buf[offset:offset + n].view(*shape)
    view.copy_(host.reshape(shape).cuda())
    return view


@pytest.mark.parametrize("seed,n,p_big", [(7, 150, 0.15), (11, 150, 0.4)])
def test_random_products(libgemm, seed, n, p_big):
    import torch
    for case, M, K, N, mode, alpha, beta, offs in _cases(seed, n, p_big):
        what = f"case {case} {mode} {M}x{K}x{N} alpha={alpha} beta={beta} offsets={offs}"
        A, B = inputs.matrices(M, K, N, "pm1", seed=case + 1000 * seed)
        ah, bh, Ao, Bo, fmt = _operands(A, B, mode)
        a, b = _placed(ah, offs[0], (M, K)), _placed(bh, offs[1], (K, N))
        C_in = inputs.matrix_c(M, N, seed=case) if beta != 0.0 else None
        cbuf = torch.full((M * N + offs[2] + 8,), float("nan"), device="cuda")
        c = cbuf[offs[2]:offs[2] + M * N].view(M, N)
        if C_in is not None:
            c.copy_(torch.from_numpy(C_in).cuda())
        libgemm.gemm_ex(a, b, c, alpha=alpha, beta=beta, mode=libgemm.MODES[mode])
        torch.cuda.synchronize()
        assert libgemm.debug_status() == libgemm.OK, what
        around = torch.cat([cbuf[:offs[2]], cbuf[offs[2] + M * N:]]).cpu().numpy()
        assert np.isnan(around).all(), f"{what}: wrote outside C"
        got = c.cpu().numpy()
        if M * N * K > 3e8:
            rows, cols = inputs.sample_indices(M, N, 1024, seed=case)
            P, S = oracle.dot(Ao, Bo, rows, cols, fmt)
            got, cin = got[rows, cols], None if C_in is None else C_in[rows, cols]
        else:
            P, S = oracle.gemm(Ao, Bo, fmt)
            cin = C_in
        assert_update_within(got, P, S, cin, alpha, beta, TOL[mode], what)
