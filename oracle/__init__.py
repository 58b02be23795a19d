"""CPU oracle for the emulated all-reduce -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library ``libar.so`` and its binding) never imports it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, compiled with
gcc); this module only builds it and marshals numpy arrays through ctypes.
Data types: fp32 as ``np.float32``, bf16 as raw ``np.uint16`` bit patterns,
int32 as ``np.int32``.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(worked example, literal ring message-passing simulation, hand-derived tree
expressions, order-independence of integer / min / max folds, the recursive
summation error bound, exact power-of-two scaling, RNE against PyTorch's
bf16 cast) and ``tests/test_oracle_mutants.py`` shows that planted mistakes
in ``oracle.c`` fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, I32 = 0, 1, 2
SUM, MIN, MAX = 0, 1, 2
RING, TREE, LL = 1, 2, 3

NP_DTYPE = {F32: np.float32, BF16: np.uint16, I32: np.int32}

CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
          "-ffp-contract=off", "-fno-fast-math"]


def compile_source(src: str, out: str) -> str:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc; no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


class OracleError(ValueError):
    pass


def _check(rc: int):
    if rc == -2:
        raise OracleError("scale != 1 is defined only for floating-point sum")
    if rc != 0:
        raise OracleError(f"invalid oracle arguments (rc={rc})")


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        L.oracle_allreduce.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), sz,
                                       sz, sz, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_float]
        L.oracle_allreduce.restype = ctypes.c_int
        L.oracle_allreduce_sampled.argtypes = [ctypes.c_int, vp, vp, sz, sz, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_float, vp]
        L.oracle_allreduce_sampled.restype = ctypes.c_int
        L.oracle_tree_expr.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_char_p, sz]
        L.oracle_tree_expr.restype = ctypes.c_int
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_ring_chunk_len.argtypes = [sz, ctypes.c_int, ctypes.c_int]
        L.oracle_ring_chunk_len.restype = sz
        L.oracle_tree_split.argtypes = [sz, ctypes.c_int]
        L.oracle_tree_split.restype = sz
        L.oracle_reduce_scatter.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), sz,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_float]
        L.oracle_reduce_scatter.restype = ctypes.c_int
        L.oracle_all_gather.argtypes = [ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp), sz,
                                        ctypes.c_int]
        L.oracle_all_gather.restype = ctypes.c_int
        L.oracle_allreduce_hier.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp),
                                            ctypes.POINTER(vp), sz, sz, sz, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_float]
        L.oracle_allreduce_hier.restype = ctypes.c_int
        L.oracle_allreduce_hier_sampled.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, sz, sz,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_float, vp]
        L.oracle_allreduce_hier_sampled.restype = ctypes.c_int
        self.lib = L
        self.path = path

    def allreduce(self, sends, dtype: int, op: int = SUM, algo: int = RING, scale: float = 1.0,
                  begin: int = 0, end: int | None = None, recvs=None):
        """All-reduce of the P host arrays in ``sends``; returns the P outputs.

        Only elements [begin, end) of each output are computed (the rest stay
        as allocated, or as passed in ``recvs``); the combination order always
        follows the full ``count`` = len(sends[0]).
        """
        P = len(sends)
        count = int(sends[0].shape[0])
        want = NP_DTYPE[dtype]
        sends = [np.ascontiguousarray(s) for s in sends]
        for s in sends:
            if s.dtype != want or s.shape != (count,):
                raise OracleError("all send arrays must share dtype and length")
        if recvs is None:
            recvs = [np.zeros(count, dtype=want) for _ in range(P)]
        end = count if end is None else end
        sp = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sends])
        rp = (ctypes.c_void_p * P)(*[r.ctypes.data for r in recvs])
        _check(self.lib.oracle_allreduce(P, sp, rp, count, begin, end, dtype, op, algo, scale))
        return recvs

    def allreduce_sampled(self, vals: np.ndarray, idx, count: int, dtype: int, op: int = SUM,
                          algo: int = RING, scale: float = 1.0) -> np.ndarray:
        """vals[r, i] = rank r's input at element idx[i]; returns y[idx[i]]."""
        vals = np.ascontiguousarray(vals, dtype=NP_DTYPE[dtype])
        idx = np.ascontiguousarray(idx, dtype=np.uint64)
        P, m = vals.shape
        if idx.shape != (m,):
            raise OracleError("idx must have one entry per column of vals")
        out = np.zeros(m, dtype=NP_DTYPE[dtype])
        _check(self.lib.oracle_allreduce_sampled(P, vals.ctypes.data, idx.ctypes.data, m, count,
                                                 dtype, op, algo, scale, out.ctypes.data))
        return out

    def allreduce_hier(self, sends, group: int, dtype: int, op: int = SUM, scale: float = 1.0,
                       begin: int = 0, end: int | None = None, recvs=None):
        """Hierarchical all-reduce, groups of `group` consecutive ranks (output
        elements [begin, end) only, as for allreduce)."""
        P = len(sends)
        count = int(sends[0].shape[0])
        want = NP_DTYPE[dtype]
        sends = [np.ascontiguousarray(s) for s in sends]
        for s in sends:
            if s.dtype != want or s.shape != (count,):
                raise OracleError("all send arrays must share dtype and length")
        if recvs is None:
            recvs = [np.zeros(count, dtype=want) for _ in range(P)]
        end = count if end is None else end
        sp = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sends])
        rp = (ctypes.c_void_p * P)(*[r.ctypes.data for r in recvs])
        _check(self.lib.oracle_allreduce_hier(P, group, sp, rp, count, begin, end, dtype, op, scale))
        return recvs

    def allreduce_hier_sampled(self, vals: np.ndarray, idx, count: int, group: int, dtype: int,
                               op: int = SUM, scale: float = 1.0) -> np.ndarray:
        vals = np.ascontiguousarray(vals, dtype=NP_DTYPE[dtype])
        idx = np.ascontiguousarray(idx, dtype=np.uint64)
        P, m = vals.shape
        out = np.zeros(m, dtype=NP_DTYPE[dtype])
        _check(self.lib.oracle_allreduce_hier_sampled(P, group, vals.ctypes.data, idx.ctypes.data, m,
                                                      count, dtype, op, scale, out.ctypes.data))
        return out

    def reduce_scatter(self, sends, dtype: int, op: int = SUM, scale: float = 1.0):
        """sends: P arrays of P * recvcount elements; returns P shards."""
        P = len(sends)
        total = int(sends[0].shape[0])
        if total % P:
            raise OracleError("reduce-scatter input length must be P * recvcount")
        rc = total // P
        want = NP_DTYPE[dtype]
        sends = [np.ascontiguousarray(s) for s in sends]
        for s in sends:
            if s.dtype != want or s.shape != (total,):
                raise OracleError("all send arrays must share dtype and length")
        recvs = [np.zeros(rc, dtype=want) for _ in range(P)]
        sp = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sends])
        rp = (ctypes.c_void_p * P)(*[r.ctypes.data for r in recvs])
        _check(self.lib.oracle_reduce_scatter(P, sp, rp, rc, dtype, op, scale))
        return recvs

    def all_gather(self, sends, dtype: int):
        """sends: P arrays of sendcount elements; returns P arrays of P * sendcount."""
        P = len(sends)
        sc = int(sends[0].shape[0])
        want = NP_DTYPE[dtype]
        sends = [np.ascontiguousarray(s) for s in sends]
        for s in sends:
            if s.dtype != want or s.shape != (sc,):
                raise OracleError("all send arrays must share dtype and length")
        recvs = [np.zeros(P * sc, dtype=want) for _ in range(P)]
        sp = (ctypes.c_void_p * P)(*[s.ctypes.data for s in sends])
        rp = (ctypes.c_void_p * P)(*[r.ctypes.data for r in recvs])
        _check(self.lib.oracle_all_gather(P, sp, rp, sc, dtype))
        return recvs

    def tree_expr(self, P: int, tree: int) -> str:
        buf = ctypes.create_string_buffer(64 * 1024)
        _check(self.lib.oracle_tree_expr(P, tree, buf, len(buf)))
        return buf.value.decode()

    def f32_to_bf16(self, x: float) -> int:
        return int(self.lib.oracle_f32_to_bf16(float(x)))

    def bf16_to_f32(self, h: int) -> float:
        return float(self.lib.oracle_bf16_to_f32(int(h)))

    def ring_chunk_len(self, count: int, P: int, dtype: int) -> int:
        return int(self.lib.oracle_ring_chunk_len(count, P, dtype))

    def tree_split(self, count: int, dtype: int) -> int:
        return int(self.lib.oracle_tree_split(count, dtype))


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def allreduce(*a, **k):
    return default().allreduce(*a, **k)


def allreduce_sampled(*a, **k):
    return default().allreduce_sampled(*a, **k)


def tree_expr(P: int, tree: int) -> str:
    return default().tree_expr(P, tree)


def reduce_scatter(*a, **k):
    return default().reduce_scatter(*a, **k)


def allreduce_hier(*a, **k):
    return default().allreduce_hier(*a, **k)


def allreduce_hier_sampled(*a, **k):
    return default().allreduce_hier_sampled(*a, **k)


def all_gather(*a, **k):
    return default().all_gather(*a, **k)


def f32_to_bf16(x: float) -> int:
    return default().f32_to_bf16(x)


def ring_chunk_len(count: int, P: int, dtype: int) -> int:
    return default().ring_chunk_len(count, P, dtype)


def tree_split(count: int, dtype: int) -> int:
    return default().tree_split(count, dtype)
