"""Helpers for the GPU parity tests (inputs, sampling, comparisons)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

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


# ------------------------------------------------------ whole-array parity

ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))


def oracle_full(host_sends, dtype: int, op: int, algo: int, scale: float = 1.0,
                group: int | None = None) -> np.ndarray:
    """The oracle's all-reduce result for every element (one array: every
    rank receives the same).  The elements are cut into ranges that run as
    separate single-threaded oracle calls on a thread pool (ctypes releases
    the GIL); each call folds its elements in the order the full count
    defines, so the ranges change nothing but the wall time.  group: the
    hierarchical order with groups of that many ranks."""
    P, count = len(host_sends), int(host_sends[0].shape[0])
    out = np.empty(count, dtype=oracle.NP_DTYPE[dtype])
    if count == 0:
        return out
    step = max(1 << 16, -(-count // (4 * ORACLE_THREADS)))
    ranges = [(b, min(count, b + step)) for b in range(0, count, step)]
    outs = [out] * P

    def run(be):
        b, e = be
        if group is not None:
            oracle.allreduce_hier(host_sends, group, dtype, op, scale, b, e, recvs=outs)
        else:
            oracle.allreduce(host_sends, dtype, op, algo, scale, b, e, recvs=outs)

    if len(ranges) == 1:
        run(ranges[0])
    else:
        with ThreadPoolExecutor(ORACLE_THREADS) as ex:
            list(ex.map(run, ranges))
    return out


def assert_equal_every_element(got, want: np.ndarray, what: str):
    """A device (or host) result against the oracle's, bit for bit, over the
    whole array; names the first differing indices."""
    g = to_host(got) if isinstance(got, torch.Tensor) else got
    if g.shape != want.shape:
        raise AssertionError(f"{what}: shape {g.shape} vs {want.shape}")
    bits = {2: np.uint16, 4: np.uint32}[want.dtype.itemsize]
    gi, wi = np.ascontiguousarray(g).view(bits), want.view(bits)
    if np.array_equal(gi, wi):
        return
    bad = np.nonzero(gi != wi)[0]
    raise AssertionError(f"{what}: {bad.size} of {want.size} elements differ, first at "
                         f"{bad[:5].tolist()}: {g[bad[:5]]} vs {want[bad[:5]]}")


def host_inputs(sends, kind: str, seed: int, sigma: float = 1.0, start: int = 0,
                n_check: int = 256) -> list:
    """Host copies of the device inputs, checked against the host generator
    at sampled indices (the oracle's inputs are the generator's values)."""
    host = [to_host(s) for s in sends]
    count = int(host[0].shape[0])
    rng = np.random.default_rng(seed + 7)
    idx = np.unique(np.concatenate([rng.integers(0, count, size=min(n_check, count)), [0, count - 1]]))
    cols = host_columns(kind, seed, len(host), idx, sigma, start)
    for r, h in enumerate(host):
        if not np.array_equal(h[idx].view(np.uint8), cols[r].view(np.uint8)):
            raise AssertionError(f"rank {r}: device inputs differ from the host generator")
    return host


def init_comm(P: int, capped_kernel: str | None = None) -> int:
    """ar_init with AR_CAPPED_KERNEL set to `capped_kernel` ("wide" or "tma":
    the kernel that P <= 8 all-reduces and reduce-scatters capped below the SM
    count run) while the communicator is created; None leaves the default."""
    if capped_kernel is None:
        return ar.ar_init(P)
    old = os.environ.get("AR_CAPPED_KERNEL")
    os.environ["AR_CAPPED_KERNEL"] = capped_kernel
    try:
        return ar.ar_init(P)
    finally:
        if old is None:
            os.environ.pop("AR_CAPPED_KERNEL", None)
        else:
            os.environ["AR_CAPPED_KERNEL"] = old
