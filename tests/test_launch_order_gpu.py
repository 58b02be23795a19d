"""Calls that depend on one another, issued back to back with no host wait.

A call that has the whole GPU is launched so that its kernel may become
resident while the kernel before it on the stream drains, and waits on the
device for that kernel's completion before it touches memory (programmatic
dependent launch); a call capped with AR_OPT_MAX_BLOCKS is launched plainly.
Each step below reads what the step before it wrote, so a kernel that read
its inputs before its predecessor finished would change the result.  The
chain mixes every kernel family (ring, tree, LL, the capped kernels, the
pipelined kernel above 8 ranks, reduce-scatter then all-gather) with PyTorch
kernels between them, which do not signal early, and is checked element by
element against the oracle applied step by step on the host.

"NCCL and NVSHMEM -- two GPU communication models, side by side" (the host
code: collectives are enqueued on a stream and complete in stream order).
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import assert_equal_every_element, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def run_chain(comm, xs, host, count, dtype, steps, dev):
    """Issues `steps` on the device with no synchronization between them and
    applies the same steps to the host arrays with the oracle."""
    P = len(xs)
    for kind, arg in steps:
        if kind == "ar":
            algo, cap, scale = arg
            ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, cap)
            ar.ar_allreduce(comm, xs, xs, count, dtype, ar.AR_SUM, algo, scale)
            oalgo = oracle.TREE if algo == ar.AR_ALGO_TREE else oracle.RING
            host = oracle.allreduce(host, dtype, oracle.SUM, oalgo, scale)
        elif kind == "torch":            # a rank-dependent change made by a PyTorch kernel
            for r in range(P):
                xs[r].mul_(float(r + 1) if dtype != ar.AR_INT32 else r + 1)
            host = [(h * np.array(r + 1, dtype=h.dtype)).astype(h.dtype) for r, h in enumerate(host)]
        elif kind == "rs_ag":            # reduce-scatter into shards, then all-gather them back
            cap = arg
            ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, cap)
            rc = count // P
            shards = [torch.empty(rc, dtype=xs[0].dtype, device=dev) for _ in range(P)]
            ar.ar_reduce_scatter(comm, xs, shards, rc, dtype, ar.AR_SUM, 1.0)
            ar.ar_all_gather(comm, shards, xs, rc, dtype)
            host = oracle.all_gather(oracle.reduce_scatter(host, dtype, oracle.SUM, 1.0), dtype)
    torch.cuda.synchronize()
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    return host


@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_INT32])
@pytest.mark.parametrize("count", [1000 * 8, 16384 + 8 * 3, 262144 * 8])
def test_dependent_calls_back_to_back(dtype, count, dev):
    P = 8
    rng = np.random.default_rng(3300 + count + dtype)
    sends = pins.random_inputs(rng, P, count, dtype)
    if dtype == ar.AR_FLOAT32:                   # keep repeated sums finite
        sends = [(s * np.float32(2.0 ** -20)).astype(np.float32) for s in sends]
    xs = [to_device(s, dtype, dev) for s in sends]
    scale = 0.125 if dtype == ar.AR_FLOAT32 else 1.0
    small = count * 4 <= 64 * 1024
    steps = [("ar", (ar.AR_ALGO_RING, 0, scale)), ("torch", None), ("ar", (ar.AR_ALGO_TREE, 0, 1.0)),
             ("torch", None), ("ar", (ar.AR_ALGO_LL if small else ar.AR_ALGO_AUTO, 0, scale)),
             ("ar", (ar.AR_ALGO_RING, 16, 1.0)),       # capped: a plain launch after a programmatic one
             ("ar", (ar.AR_ALGO_TREE, 0, scale)),      # and a programmatic one after a plain one
             ("rs_ag", 0), ("torch", None), ("rs_ag", 16), ("ar", (ar.AR_ALGO_RING, 0, 1.0))]
    comm = ar.ar_init(P)
    try:
        for rep in range(3):
            host = run_chain(comm, xs, [s.copy() for s in sends] if rep == 0 else host, count, dtype,
                             steps, dev)
            for r in range(P):
                assert_equal_every_element(xs[r], host[r], f"repetition {rep} rank {r}")
    finally:
        ar.ar_destroy(comm)


def test_dependent_calls_above_eight_ranks(dev):
    """The pipelined kernel (72 ranks), uncapped and capped, chained the same way."""
    P, dtype, count = 72, ar.AR_INT32, 72 * 4096 + 72 * 3
    rng = np.random.default_rng(3400)
    sends = pins.random_inputs(rng, P, count, dtype)
    xs = [to_device(s, dtype, dev) for s in sends]
    steps = [("ar", (ar.AR_ALGO_RING, 0, 1.0)), ("torch", None), ("ar", (ar.AR_ALGO_TREE, 0, 1.0)),
             ("ar", (ar.AR_ALGO_RING, 16, 1.0)), ("ar", (ar.AR_ALGO_TREE, 0, 1.0)), ("rs_ag", 0),
             ("torch", None), ("rs_ag", 16)]
    comm = ar.ar_init(P)
    try:
        host = run_chain(comm, xs, [s.copy() for s in sends], count, dtype, steps, dev)
        for r in range(P):
            assert_equal_every_element(xs[r], host[r], f"rank {r}")
    finally:
        ar.ar_destroy(comm)


def test_dependent_calls_replayed_from_a_graph(dev):
    """The same kind of chain captured once in a CUDA graph and replayed three
    times: each replay starts from the previous replay's results."""
    P, dtype, count = 8, ar.AR_FLOAT32, 16384 - 8      # LL-sized: at most 64 KiB per rank
    rng = np.random.default_rng(3500)
    sends = [(s * np.float32(2.0 ** -20)).astype(np.float32) for s in pins.random_inputs(rng, P, count, dtype)]
    xs = [to_device(s, dtype, dev) for s in sends]
    comm = ar.ar_init(P)
    try:
        # first call on each path outside the capture (per-device set-up)
        for algo in (ar.AR_ALGO_RING, ar.AR_ALGO_TREE, ar.AR_ALGO_LL):
            ar.ar_allreduce(comm, [x.clone() for x in xs], [torch.empty_like(x) for x in xs], count, dtype,
                            ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        host = [s.copy() for s in sends]
        stream = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                ar.ar_allreduce(comm, xs, xs, count, dtype, ar.AR_SUM, ar.AR_ALGO_LL, 0.125, stream)
                for r in range(P):
                    xs[r].mul_(float(r + 1))
                ar.ar_allreduce(comm, xs, xs, count, dtype, ar.AR_SUM, ar.AR_ALGO_TREE, 0.125, stream)
                ar.ar_allreduce(comm, xs, xs, count, dtype, ar.AR_SUM, ar.AR_ALGO_RING, 1.0, stream)
        for _ in range(3):
            g.replay()
            host = oracle.allreduce(host, dtype, oracle.SUM, oracle.RING, 0.125)
            host = [(h * np.float32(r + 1)).astype(np.float32) for r, h in enumerate(host)]
            host = oracle.allreduce(host, dtype, oracle.SUM, oracle.TREE, 0.125)
            host = oracle.allreduce(host, dtype, oracle.SUM, oracle.RING, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        for r in range(P):
            assert_equal_every_element(xs[r], host[r], f"rank {r}")
    finally:
        ar.ar_destroy(comm)
