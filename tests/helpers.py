"""Shared helpers for the GPU tests: moving seeded host arrays to the device and
back, and the seeded input mixes used by the parity tests."""
from __future__ import annotations

import numpy as np

import oracle as O

DT_NP = {O.F32: np.float32, O.F16: np.float16, O.BF16: np.uint16}


def to_dev(x: np.ndarray, dtype: int):
    """Host array (float32 / float16 / uint16 bf16 bits) -> CUDA tensor of that type."""
    import torch

    x = np.ascontiguousarray(x)
    if dtype == O.BF16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    if dtype == O.F16:
        return torch.from_numpy(x.view(np.float16)).cuda()
    return torch.from_numpy(x.astype(np.float32, copy=False)).cuda()


def bytes_dev(a: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t) -> np.ndarray:
    """CUDA tensor -> host numpy (bf16 and fp16 as uint16 bit patterns)."""
    import torch

    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def mixed_input(n: int, dtype: int, seed: int, G: int = 32) -> np.ndarray:
    """A seeded mix that exercises every path: normal weights, Laplace tails,
    x50 outliers, an all-zero block, a block of exact half-steps (ties) and a
    block of tiny values. Returned in the storage type (bf16 as uint16 bits)."""
    from blockwise_quantized_zero_gb300 import inputs

    x = inputs.normal_f32(n, 0.02, seed)
    if n > 8:
        x[::7] = inputs.laplace_f32(len(x[::7]), 0.01, seed, stream=1)
        x[::997] *= 50
    nb = n // G
    if nb >= 4:
        x[G:2 * G] = 0.0                                   # zero block
        k = np.arange(G, dtype=np.float32) - G // 2
        x[2 * G:3 * G] = (k + 0.5) * np.float32(2.0 ** -7)  # exact ties for every width
        x[2 * G] = np.float32(127 * 2.0 ** -7)
        x[3 * G:4 * G] *= np.float32(1e-6)                  # tiny block
    if dtype == O.BF16:
        from blockwise_quantized_zero_gb300.inputs import to_bf16_bits

        return to_bf16_bits(x)
    if dtype == O.F16:
        return x.astype(np.float16)
    return x


def oracle_quantize(x: np.ndarray, dtype: int, fmt: int, G: int):
    return O.quantize(x, fmt, G, dtype=dtype if dtype == O.BF16 else None)
