"""Helpers for the GPU parity tests (inputs, sampling, comparisons)."""
from __future__ import annotations

import numpy as np
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import synthetic

VEC = {ar.AR_FLOAT32: 4, ar.AR_BFLOAT16: 8, ar.AR_INT32: 4}
TORCH = {ar.AR_FLOAT32: torch.float32, ar.AR_BFLOAT16: torch.bfloat16, ar.AR_INT32: torch.int32}
KIND_DTYPE = {"uniform": ar.AR_FLOAT32, "normal": ar.AR_FLOAT32, "normal_bf16": ar.AR_BFLOAT16,
              "uniform_bf16": ar.AR_BFLOAT16,
              "int": ar.AR_INT32}
GUARD = 64          # bytes of guard words on each side of a guarded buffer
GUARD_BYTE = 0x5A


def to_device(a: np.ndarray, dtype: int, device) -> torch.Tensor:
    if dtype == ar.AR_BFLOAT16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class Guarded:
    """A device buffer with guard bytes on both sides (checks stray writes)."""

    def __init__(self, count: int, dtype: int, device):
        esize = 2 if dtype == ar.AR_BFLOAT16 else 4
        self.nbytes = count * esize
        self.raw = torch.full((GUARD * 2 + self.nbytes,), GUARD_BYTE, dtype=torch.uint8, device=device)
        self.tensor = self.raw[GUARD:GUARD + self.nbytes].view(TORCH[dtype])

    def guards_intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == GUARD_BYTE).all() and (tail == GUARD_BYTE).all())


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def sample_indices(count: int, P: int, dtype: int, n_random: int = 1024, seed: int = 0) -> np.ndarray:
    """Random indices plus every ring-chunk edge, the tree split and the tail."""
    V = VEC[dtype]
    L = ceil_div(ceil_div(count, P), V) * V
    H = min(count, ceil_div(ceil_div(count, 2), V) * V)
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, count, size=min(n_random, count)).tolist())
    idx |= {0, count - 1}
    for c in range(1, P + 1):
        for d in (-1, 0, 1):
            idx.add(c * L + d)
    for d in (-1, 0, 1):
        idx.add(H + d)
    for d in range(1, 2 * V + 1):
        idx.add(count - d)
    return np.array(sorted(i for i in idx if 0 <= i < count), dtype=np.int64)


def device_inputs(kind: str, seed: int, P: int, count: int, device, sigma: float = 1.0,
                  start: int = 0):
    return [synthetic.values_torch(kind, seed, r, start, count, device, sigma) for r in range(P)]


def host_columns(kind: str, seed: int, P: int, idx: np.ndarray, sigma: float = 1.0,
                 start: int = 0) -> np.ndarray:
    return np.stack([synthetic.values_np(kind, seed, r, idx + start, sigma) for r in range(P)])


def check_sampled(recvs, sends, kind: str, seed: int, count: int, dtype: int, op: int, algo: int,
                  scale: float, sigma: float = 1.0, start: int = 0, n_random: int = 1024):
    """Sampled outputs of a full-size call against the oracle, bit for bit.

    The oracle's inputs come from the host generator; the device inputs at
    the same indices are checked to be the same values.
    """
    P = len(recvs)
    idx = sample_indices(count, P, dtype, n_random=n_random, seed=seed + 1)
    cols = host_columns(kind, seed, P, idx, sigma, start)
    it = torch.from_numpy(idx).to(recvs[0].device)
    dev_cols = np.stack([to_host(s.index_select(0, it)) for s in sends])
    assert np.array_equal(dev_cols.view(np.uint8), cols.view(np.uint8)), "device / host inputs differ"
    oalgo = oracle.TREE if algo == ar.AR_ALGO_TREE else oracle.RING
    want = oracle.allreduce_sampled(cols, idx, count, dtype, op, oalgo, scale)
    for r in range(P):
        got = to_host(recvs[r].index_select(0, it))
        if not np.array_equal(got.view(np.uint8), want.view(np.uint8)):
            bad = np.nonzero(got != want)[0][:5]
            raise AssertionError(f"rank {r}: sampled outputs differ at {idx[bad].tolist()}: "
                                 f"{got[bad]} vs {want[bad]}")


def all_ranks_identical(recvs) -> bool:
    a = recvs[0].view(torch.uint8) if recvs[0].dtype != torch.bfloat16 else recvs[0].view(torch.int16)
    for t in recvs[1:]:
        b = t.view(torch.uint8) if t.dtype != torch.bfloat16 else t.view(torch.int16)
        if not torch.equal(a, b):
            return False
    return True
