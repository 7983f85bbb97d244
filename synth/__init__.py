"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

Holds no arithmetic of the FP8 method: it only draws random numbers and
stores them as bf16 bit patterns (uint16), so both sides receive the same bytes.

Every tensor comes from its own numpy PCG64 stream keyed by (seed, tensor id,
step).  ``N(mu, sigma)`` means sigma is the standard deviation.  Values are
drawn in fp64, rounded to fp32 and then to bf16 with round-to-nearest-even
(finite values only: the normal draws never overflow).
"""
from __future__ import annotations

import numpy as np

TENSOR_IDS = {"x": 1, "w": 2, "g": 3, "bias": 4, "lengths": 5, "outlier": 6}


def _rng(seed: int, tensor: str | int, step: int = 0) -> np.random.Generator:
    tid = TENSOR_IDS[tensor] if isinstance(tensor, str) else int(tensor)
    return np.random.Generator(np.random.PCG64([int(seed), tid, int(step)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, sigma: float, seed: int, tensor, step: int = 0,
                mu: float = 0.0, chunk: int = 1 << 24) -> np.ndarray:
    """N(mu, sigma) samples as bf16 bit patterns of the given shape."""
    rng = _rng(seed, tensor, step)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s) * sigma + mu
        out[s:e] = f32_to_bf16_bits(v.astype(np.float32))
    return out.reshape(shape)


def normal_with_outliers_bf16(shape, sigma: float, seed: int, tensor, step: int = 0,
                              p: float = 0.01, factor: float = 50.0,
                              chunk: int = 1 << 24) -> np.ndarray:
    """N(0, sigma) where each element independently, with probability p
    (a seeded Bernoulli draw), is multiplied by ``factor`` before the bf16
    rounding: the "1% outliers x50" input of the block-scaled workload."""
    rng = _rng(seed, tensor, step)
    orng = _rng(seed, "outlier", step * 16 + (TENSOR_IDS[tensor] if isinstance(tensor, str) else int(tensor)))
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s) * sigma
        hit = orng.random(e - s) < p
        v[hit] *= factor
        out[s:e] = f32_to_bf16_bits(v.astype(np.float32))
    return out.reshape(shape)


def thd_lengths(seed: int, n_seq: int = 64, lo: int = 128, hi: int = 4096) -> np.ndarray:
    """Sequence lengths of a packed THD batch, uniform integers in [lo, hi]."""
    return _rng(seed, "lengths").integers(lo, hi + 1, size=n_seq, dtype=np.int64)


# Workload recipes (shapes and distributions of the pages' workloads).
CONFIG1 = dict(M=64, K=256, N=256, x_sigma=1.0, w_sigma=0.02, seed=0)
CONFIG2 = dict(M=4096, K=4096, N=4096, x_sigma=1.0, w_sigma=0.02, g_sigma=1e-3,
               steps=20, seed=0)
CONFIG3 = dict(M=16384, hidden=4096, ffn=14336, w_sigma=0.02, x_sigma=1.0, g_sigma=1e-3, seed=0)
CONFIG4 = dict(n_seq=64, lo=128, hi=4096, K=4096, N=4096, x_sigma=1.0, w_sigma=0.02,
               g_sigma=1e-3, multiple=16, seed=0)
CONFIG5 = dict(M=32768, K=8192, N=8192, sigma=1.0, p=0.01, factor=50.0, seed=0)
