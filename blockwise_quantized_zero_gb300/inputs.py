"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the quantization method. It draws random
values from a counter-based generator (Philox-4x64 from numpy, keyed by
``(seed, stream, chunk)`` so any chunk can be regenerated on its own) and
rounds them to the storage type with library routines (numpy for fp16, torch
CPU for bf16; both round to nearest even). Both the CUDA path and the oracle
receive the same bytes from here.

Workload recipes (shapes, distributions and seeds of the five synthetic
workloads the method is measured on):

* ``weights_fp16_outliers``: 1,048,576 fp16 ~ N(0, 0.02), with
  round(0.001 n) elements chosen without replacement and multiplied by 50
  before rounding (qwZ-style weights with outliers), seed 0;
* ``weight_shard_bf16``: one 8192 x 8192 bf16 shard ~ N(0, 0.02), seed 2;
* ``gradient_shard_f32``: 134,217,728 fp32 ~ Laplace(0, 1e-4) per shard,
  seed 3, stream = shard index;
* ``gradient_bf16``: 268,435,456 bf16 ~ N(0, 1e-3) per micro-batch step,
  seed 4, stream = step (and 100 + shard for the reduce's peer shards);
* ``llama70b_layer_bf16``: the seven matrices of one Llama-3-70B decoder
  layer (q, o 8192x8192; k, v 8192x1024; gate, up 8192x28672; down
  28672x8192) ~ N(0, 0.02), seed 5, stream = matrix index.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

CHUNK = 1 << 24  # elements per independently keyed chunk

LLAMA70B_LAYER = (
    ("q", 8192, 8192),
    ("k", 8192, 1024),
    ("v", 8192, 1024),
    ("o", 8192, 8192),
    ("gate", 8192, 28672),
    ("up", 8192, 28672),
    ("down", 28672, 8192),
)


def _gen(seed: int, stream: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, chunk])))


def _threads() -> int:
    return max(1, min(8, os.cpu_count() or 1))


def _fill(n: int, seed: int, stream: int, draw) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        out[lo:hi] = draw(_gen(seed, stream, c), hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal_f32(n: int, sigma: float, seed: int, stream: int = 0) -> np.ndarray:
    """n float32 samples of N(0, sigma^2)."""
    return _fill(n, seed, stream,
                 lambda g, m: g.standard_normal(m, dtype=np.float32) * np.float32(sigma))


def laplace_f32(n: int, beta: float, seed: int, stream: int = 0) -> np.ndarray:
    """n float32 samples of Laplace(0, beta)."""
    return _fill(n, seed, stream, lambda g, m: g.laplace(0.0, beta, m).astype(np.float32))


def uniform_f32(n: int, lo: float, hi: float, seed: int, stream: int = 0) -> np.ndarray:
    return _fill(n, seed, stream, lambda g, m: g.uniform(lo, hi, m).astype(np.float32))


def to_f16(x: np.ndarray) -> np.ndarray:
    """Round float32 to fp16 (numpy, nearest-even); returned as np.float16."""
    return x.astype(np.float16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (torch CPU, nearest-even); returned as uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def outlier_indices(n: int, frac: float, seed: int) -> np.ndarray:
    k = int(round(frac * n))
    return np.sort(_gen(seed, 1 << 20, 0).choice(n, size=k, replace=False))


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

def weights_fp16_outliers(n: int = 1 << 20, sigma: float = 0.02, frac: float = 0.001,
                          factor: float = 50.0, seed: int = 0) -> np.ndarray:
    x = normal_f32(n, sigma, seed)
    idx = outlier_indices(n, frac, seed)
    x[idx] *= np.float32(factor)
    return to_f16(x)


def weight_shard_bf16(rows: int = 8192, cols: int = 8192, sigma: float = 0.02,
                      seed: int = 2) -> np.ndarray:
    return to_bf16_bits(normal_f32(rows * cols, sigma, seed))


def gradient_shard_f32(n: int = 1 << 27, beta: float = 1e-4, seed: int = 3,
                       shard: int = 0) -> np.ndarray:
    return laplace_f32(n, beta, seed, stream=shard)


def gradient_bf16(n: int = 1 << 28, sigma: float = 1e-3, seed: int = 4,
                  step: int = 0) -> np.ndarray:
    return to_bf16_bits(normal_f32(n, sigma, seed, stream=step))


def llama70b_layer_bf16(sigma: float = 0.02, seed: int = 5, scale_rows: int = 1):
    """Yield (name, rows, cols, uint16 bf16 bits) for each matrix of the layer.

    ``scale_rows`` divides every row count (1 = the full layer), for small
    versions of the same shapes in tests.
    """
    for i, (name, r, c) in enumerate(LLAMA70B_LAYER):
        r = r // scale_rows
        yield name, r, c, to_bf16_bits(normal_f32(r * c, sigma, seed, stream=i))
