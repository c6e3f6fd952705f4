"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
GEMM's or the quantisers' arithmetic.  Both the CUDA path and the CPU oracle
consume what it returns.

Recipe: i.i.d. N(0,1) FP32 values from ``torch.Generator('cpu')`` seeded with
``seed`` (the workloads use seed = 1000 + workload index), A drawn before B.
BF16 operands are those values cast to bfloat16 by torch (round to nearest
even).  The draws are bit-identical on every machine, so every GPU run sees the
same bytes.
"""
from __future__ import annotations

import numpy as np
import torch


def normal_f32(rows: int, cols: int, gen: torch.Generator) -> np.ndarray:
    return torch.randn(rows, cols, generator=gen, dtype=torch.float32).numpy()


def gemm_inputs_f32(m: int, n: int, k: int, seed: int):
    """(A, B) FP32 N(0,1), shapes (m, k) and (n, k)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    a = normal_f32(m, k, g)
    b = normal_f32(n, k, g)
    return a, b


def bf16_codes(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of x cast to bfloat16 (torch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def random_codes(shape, n_codes: int, seed: int, exclude=()) -> np.ndarray:
    """Uniform random codes in [0, n_codes) avoiding the listed codes (e.g. NaN codes)."""
    rng = np.random.default_rng(seed)
    allowed = np.array([c for c in range(n_codes) if c not in set(exclude)], dtype=np.int64)
    idx = rng.integers(0, allowed.size, size=shape)
    return allowed[idx]
