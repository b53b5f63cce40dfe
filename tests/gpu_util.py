"""Moving seeded numpy inputs onto the GPU and running libgemm on them."""
from __future__ import annotations

import numpy as np

from accelerator_gb300 import inputs


def device_operands(A: np.ndarray, B: np.ndarray, mode: str):
    """Torch CUDA tensors for mode: float32, or the bf16 rounding of A and B."""
    import torch
    if mode == "bf16":
        a = torch.from_numpy(inputs.bf16_bits(A).view(np.int16)).view(torch.bfloat16)
        b = torch.from_numpy(inputs.bf16_bits(B).view(np.int16)).view(torch.bfloat16)
    elif mode == "fp16":
        a = torch.from_numpy(inputs.fp16_bits(A).view(np.int16)).view(torch.float16)
        b = torch.from_numpy(inputs.fp16_bits(B).view(np.int16)).view(torch.float16)
    else:
        a, b = torch.from_numpy(A), torch.from_numpy(B)
    return a.cuda(), b.cuda()


def run(binding, A: np.ndarray, B: np.ndarray, mode: str, poison: bool = True) -> np.ndarray:
    """C = A*B through the C ABI on cuda:0, C pre-filled with NaN; returns C on the host."""
    import torch
    a, b = device_operands(A, B, mode)
    M, N = A.shape[0], B.shape[1]
    c = torch.full((M, N), float("nan") if poison else 0.0, dtype=torch.float32, device="cuda")
    binding.gemm(a, b, c, mode=binding.MODES[mode])
    torch.cuda.synchronize()
    assert binding.debug_status() == binding.OK
    return c.cpu().numpy()


def oracle_inputs(A: np.ndarray, B: np.ndarray, mode: str):
    """(A, B, fmt) for the oracle seeing exactly the values the tensor cores see."""
    if mode == "bf16":
        return inputs.bf16_bits(A), inputs.bf16_bits(B), "bf16"
    if mode == "fp16":
        return inputs.fp16_bits(A), inputs.fp16_bits(B), "f16"
    if mode == "tf32":
        return A, B, "tf32"
    if mode == "tf32_rn":
        return A, B, "tf32rna"
    return A, B, "f32"
