"""Seeded synthetic inputs for the emulated all-reduce (shared by tests and bench).

This module holds no arithmetic of the all-reduce itself: it only turns
(seed, rank, element index) into input values, the same way on the host
(numpy) and on a device (plain PyTorch ops), so that a full-size input made on
the GPU and a sampled column of it recomputed on the host agree bit for bit.

Counter-based generator: splitmix64 as published by S. Vigna (the finaliser of
Steele, Lea and Flood's SplitMix, 2014): for a 64-bit counter x,
    z = x + 0x9E3779B97F4A7C15
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    z = z ^ (z >> 31)
all modulo 2^64.  Draw j of element e on rank r:
    u32(seed, r, e, j) = splitmix64(seed ^ (r << 40) ^ (16 e + j)) >> 32.

Distributions (all exact or rounded once, so host and device agree):
  uniform[-1, 1]   : ((u >> 8) - 2^23) * 2^-23                       (exact in fp32)
  normal(0, sigma) : Irwin-Hall with 12 draws: K = sum_j (u_j >> 8) as an integer,
                     fp32(K - 6 * 2^24) * 2^-24 * fp32(sigma)       (sigma = std dev)
  int uniform      : (u mod (hi - lo + 1)) + lo                      (int32)
  bf16             : round-to-nearest-even of the fp32 value ('normal_bf16',
                     'uniform_bf16')
"""
from __future__ import annotations

import numpy as np

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1
DRAWS_PER_ELEMENT = 16   # counter stride per element; the normal uses 12 of them


def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


# ---------------------------------------------------------------- host (numpy)

def splitmix64_np(x: np.ndarray) -> np.ndarray:
    z = x.astype(np.uint64) + np.uint64(_GOLDEN)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def u32_np(seed: int, rank: int, idx, draw: int = 0) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.uint64)
    key = np.uint64((seed ^ (rank << 40)) & _MASK64)
    ctr = key ^ (idx * np.uint64(DRAWS_PER_ELEMENT) + np.uint64(draw))
    return (splitmix64_np(ctr) >> np.uint64(32)).astype(np.uint64)


def uniform_np(seed: int, rank: int, idx) -> np.ndarray:
    k = (u32_np(seed, rank, idx) >> np.uint64(8)).astype(np.int64) - (1 << 23)
    return k.astype(np.float32) * np.float32(2.0 ** -23)


def normal_np(seed: int, rank: int, idx, sigma: float) -> np.ndarray:
    K = np.zeros(np.shape(idx), dtype=np.int64)
    for j in range(12):
        K += (u32_np(seed, rank, idx, j) >> np.uint64(8)).astype(np.int64)
    x = (K - 6 * (1 << 24)).astype(np.float32) * np.float32(2.0 ** -24)
    return x * np.float32(sigma)


def int_uniform_np(seed: int, rank: int, idx) -> np.ndarray:
    lo, hi = -(1 << 20), 1 << 20
    u = u32_np(seed, rank, idx)
    return ((u % np.uint64(hi - lo + 1)).astype(np.int64) + lo).astype(np.int32)


def bf16_bits_np(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def values_np(kind: str, seed: int, rank: int, idx, sigma: float = 1.0) -> np.ndarray:
    """kind: 'uniform' / 'normal' (fp32), 'uniform_bf16' / 'normal_bf16' (uint16 bits), 'int'."""
    if kind == "uniform":
        return uniform_np(seed, rank, idx)
    if kind == "uniform_bf16":
        return bf16_bits_np(uniform_np(seed, rank, idx))
    if kind == "normal":
        return normal_np(seed, rank, idx, sigma)
    if kind == "normal_bf16":
        return bf16_bits_np(normal_np(seed, rank, idx, sigma))
    if kind == "int":
        return int_uniform_np(seed, rank, idx)
    raise ValueError(kind)


# ------------------------------------------------------------- device (torch)

def _lsr(z, k: int):
    # logical shift right on int64 tensors
    return (z >> k) & ((1 << (64 - k)) - 1)


def splitmix64_torch(x):
    z = x + _signed(_GOLDEN)
    z = (z ^ _lsr(z, 30)) * _signed(_M1)
    z = (z ^ _lsr(z, 27)) * _signed(_M2)
    return z ^ _lsr(z, 31)


def u32_torch(seed: int, rank: int, idx, draw: int = 0):
    key = _signed((seed ^ (rank << 40)) & _MASK64)
    ctr = (idx * DRAWS_PER_ELEMENT + draw) ^ key
    return _lsr(splitmix64_torch(ctr), 32)


def values_torch(kind: str, seed: int, rank: int, start: int, n: int, device, sigma: float = 1.0):
    """Elements [start, start + n) of rank `rank`, generated on `device`."""
    import torch

    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    if kind in ("uniform", "uniform_bf16"):
        k = (u32_torch(seed, rank, idx) >> 8) - (1 << 23)
        x = k.to(torch.float32) * (2.0 ** -23)
        return x.to(torch.bfloat16) if kind == "uniform_bf16" else x
    if kind in ("normal", "normal_bf16"):
        K = torch.zeros_like(idx)
        for j in range(12):
            K += u32_torch(seed, rank, idx, j) >> 8
        del idx
        x = (K - 6 * (1 << 24)).to(torch.float32)
        del K
        x.mul_(2.0 ** -24).mul_(float(np.float32(sigma)))
        if kind == "normal_bf16":
            return x.to(torch.bfloat16)
        return x
    if kind == "int":
        lo, hi = -(1 << 20), 1 << 20
        u = u32_torch(seed, rank, idx)
        return (torch.remainder(u, hi - lo + 1) + lo).to(torch.int32)
    raise ValueError(kind)
