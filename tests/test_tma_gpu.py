"""Collectives capped to fewer SMs than the GPU has, against the oracle, bit
for bit: the all-reduce and reduce-scatter (P <= 8) in both capped kernels --
the wide load/store shape (1024-thread blocks, the default) and the TMA
bulk-copy pipeline (AR_CAPPED_KERNEL=tma) -- and the TMA all-gather (any P).

"NCCL, NIXL, and Distributed GPU Communication" (the overlap checklist): the
all-reduce runs beside computation, so AR_OPT_MAX_BLOCKS gives it a few SMs.
Same orders as the uncapped kernel, so the results agree element for element;
ragged counts exercise partial tiles and the trailing partial vector; the TMA
pipeline's bounded mbarrier waits are made to run out with the producer-skip
test hook.
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import (VEC, Guarded, assert_equal_every_element, device_inputs, host_inputs, init_comm,
                      oracle_full, to_device, to_host)

pytestmark = pytest.mark.gpu

OPS = (ar.AR_SUM, ar.AR_MIN, ar.AR_MAX)
BLOCKS = 16
KINDS = ("wide", "tma")   # AR_CAPPED_KERNEL: the capped all-reduce / reduce-scatter kernel


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def tma_counts(dtype):
    V, tile = VEC[dtype], 4096 // (2 if dtype == ar.AR_BFLOAT16 else 4)
    return [BLOCKS * tile, BLOCKS * tile + 3 * V + 1, 37 * tile + V - 1, 200_003]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_calls_match_the_oracle(P, dtype, kind, dev, capfd):
    rng = np.random.default_rng(800 + 10 * P + dtype)
    comm = init_comm(P, kind)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_DEBUG, 1)
        for count in tma_counts(dtype):
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for op in OPS:
                for algo, oalgo in ((ar.AR_ALGO_RING, oracle.RING), (ar.AR_ALGO_TREE, oracle.TREE)):
                    scale = 0.125 if (op == ar.AR_SUM and dtype != ar.AR_INT32) else 1.0
                    outs = [Guarded(count, dtype, dev) for _ in range(P)]
                    ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, algo, scale)
                    torch.cuda.synchronize()
                    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                    want = oracle.allreduce(sends, dtype, op, oalgo, scale)
                    for r in range(P):
                        assert outs[r].guards_intact()
                        pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                            f"P={P} dtype={dtype} count={count} op={op} algo={algo} rank={r}")
        log = capfd.readouterr().err
        assert f"kernel={kind}_ring" in log and f"kernel={kind}_tree" in log
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("kind", KINDS)
def test_full_size_equals_the_uncapped_kernel(kind, dev):
    """8 x 64 MiB fp32, ring, scale 1/8 on 64 SMs: every element against the
    oracle, and element for element the uncapped kernel's result, in place
    and out of place."""
    P, count = 8, 16 * 1024 * 1024
    comm = init_comm(P, kind)
    try:
        sends = device_inputs("normal", 0, P, count, dev, 1e-3)
        ref = [torch.empty_like(s) for s in sends]
        got = [torch.empty_like(s) for s in sends]
        ar.ar_allreduce(comm, sends, ref, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 64)
        ar.ar_allreduce(comm, sends, got, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
        torch.cuda.synchronize()
        want = oracle_full(host_inputs(sends, "normal", 0, 1e-3), ar.AR_FLOAT32, oracle.SUM, oracle.RING, 0.125)
        assert_equal_every_element(got[0], want, "64 SMs rank 0")
        for r in range(P):
            assert torch.equal(got[r].view(torch.int32), ref[r].view(torch.int32)), f"rank {r}"
        inplace = [s.clone() for s in sends]
        ar.ar_allreduce(comm, inplace, inplace, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        for r in range(P):
            assert torch.equal(inplace[r].view(torch.int32), ref[r].view(torch.int32)), f"in place, rank {r}"
    finally:
        ar.ar_destroy(comm)


def test_bounded_waits_report_a_timeout_and_recover(dev):
    """The TMA pipeline's mbarrier waits (the wide kernel has none)."""
    P, count = 8, 1 << 20
    comm = init_comm(P, "tma")
    try:
        rng = np.random.default_rng(12)
        sends = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.zeros_like(x) for x in xs]
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 32)
        # no tile is ever loaded: every consumer wait, then the producer's, runs out
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 2000)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 1)
        ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 0)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 1 << 22)
        ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING)
        pins.assert_bitwise(to_host(ys[6]), want[6], "TMA call after a timed-out one")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("P", [1, 2, 3, 8])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_reduce_scatter_matches_the_oracle(P, dtype, kind, dev, capfd):
    """Reduce-scatter on 16 SMs: shard s folded in ring chunk s's order, stored
    to its owner only; shards of whole 4 KiB tiles and shards whose edges fall
    inside a tile (the TMA pipeline stores those segment by segment)."""
    rng = np.random.default_rng(900 + 10 * P + dtype)
    comm = init_comm(P, kind)
    used = False
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_DEBUG, 1)
        for rc in (16384, 20000, 50000):
            sends = pins.random_inputs(rng, P, P * rc, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for op in OPS:
                scale = 0.125 if (op == ar.AR_SUM and dtype != ar.AR_INT32) else 1.0
                outs = [Guarded(rc, dtype, dev) for _ in range(P)]
                ar.ar_reduce_scatter(comm, xs, [o.tensor for o in outs], rc, dtype, op, scale)
                torch.cuda.synchronize()
                assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                want = oracle.reduce_scatter(sends, dtype, op, scale)
                for r in range(P):
                    assert outs[r].guards_intact()
                    pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                        f"RS P={P} dtype={dtype} rc={rc} op={op} rank={r}")
        used = f"kernel={kind}_reduce_scatter" in capfd.readouterr().err
    finally:
        ar.ar_destroy(comm)
    assert used


@pytest.mark.parametrize("kind", KINDS)
def test_capped_reduce_scatter_in_place(kind, dev):
    P, rc = 8, 20000
    comm = init_comm(P, kind)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        rng = np.random.default_rng(31)
        sends = pins.random_inputs(rng, P, P * rc, ar.AR_FLOAT32)
        want = oracle.reduce_scatter(sends, ar.AR_FLOAT32, ar.AR_SUM, 0.125)
        big = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ar.ar_reduce_scatter(comm, big, [big[r][r * rc:(r + 1) * rc] for r in range(P)], rc,
                             ar.AR_FLOAT32, ar.AR_SUM, 0.125)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        for r in range(P):
            pins.assert_bitwise(to_host(big[r][r * rc:(r + 1) * rc]), want[r], f"in place rank {r}")
    finally:
        ar.ar_destroy(comm)


def ag_counts(P, dtype):
    """Shard lengths giving at least BLOCKS tiles of 32 KiB in all: whole tiles
    and a ragged last tile (still whole 16-byte vectors)."""
    es, V = (2, 8) if dtype == ar.AR_BFLOAT16 else (4, 4)
    base = -(-BLOCKS * 32768 // (P * es) // V) * V
    return [base, base + 3 * V, 4 * base + V]


@pytest.mark.parametrize("P", [1, 2, 3, 8, 13, 72])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_all_gather_matches_the_oracle(P, dtype, dev, capfd):
    rng = np.random.default_rng(950 + 10 * P + dtype)
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_DEBUG, 1)
        for sc in ag_counts(P, dtype):
            pieces = pins.random_inputs(rng, P, sc, dtype)
            xs = [to_device(a, dtype, dev) for a in pieces]
            outs = [Guarded(P * sc, dtype, dev) for _ in range(P)]
            ar.ar_all_gather(comm, xs, [o.tensor for o in outs], sc, dtype)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            want = oracle.all_gather(pieces, dtype)
            for r in (0, P // 2, P - 1):
                assert outs[r].guards_intact()
                pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"AG P={P} dtype={dtype} sc={sc} rank={r}")
        assert "kernel=tma_all_gather" in capfd.readouterr().err
    finally:
        ar.ar_destroy(comm)


def test_capped_all_gather_in_place_and_timeout(dev):
    P, sc = 8, 100_004
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        rng = np.random.default_rng(41)
        pieces = pins.random_inputs(rng, P, sc, ar.AR_FLOAT32)
        full = [torch.zeros(P * sc, device=dev) for _ in range(P)]
        for r in range(P):
            full[r][r * sc:(r + 1) * sc] = torch.from_numpy(pieces[r]).to(dev)
        ar.ar_all_gather(comm, [full[r][r * sc:(r + 1) * sc] for r in range(P)], full, sc, ar.AR_FLOAT32)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        want = oracle.all_gather(pieces, ar.AR_FLOAT32)
        for r in range(P):
            pins.assert_bitwise(to_host(full[r]), want[r], f"in place rank {r}")
        # no tile is ever loaded: the bounded waits run out and report
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 2000)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 1)
        outs = [torch.zeros(P * sc, device=dev) for _ in range(P)]
        srcs = [to_device(a, ar.AR_FLOAT32, dev) for a in pieces]
        ar.ar_all_gather(comm, srcs, outs, sc, ar.AR_FLOAT32)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 0)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 1 << 22)
        ar.ar_all_gather(comm, srcs, outs, sc, ar.AR_FLOAT32)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        pins.assert_bitwise(to_host(outs[5]), want[5], "after a timed-out call")
    finally:
        ar.ar_destroy(comm)


FIRST_CALL_CAPTURED = r"""
import sys
import numpy as np, torch
sys.path.insert(0, {root!r})
import allreduce_reduction_emulated_gb300 as ar
torch.cuda.set_device(0)
dev = torch.device("cuda:0")
P, n = 8, 1 << 20
xs = [torch.full((n,), float(r + 1), device=dev) for r in range(P)]
ys = [torch.zeros(n, device=dev) for _ in range(P)]
comm = ar.ar_init(P)
ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 16)
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    with torch.cuda.graph(g, stream=s):          # the process's first capped call
        ar.ar_allreduce(comm, xs, ys, n, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125, s)
g.replay()
torch.cuda.synchronize()
assert ar.ar_get_status(comm) == ar.AR_SUCCESS
assert bool((ys[3] == 4.5).all())                # (1 + ... + 8) / 8
ar.ar_destroy(comm)
print("ok")
"""


def test_first_capped_call_inside_a_graph_capture(dev):
    """The TMA kernel's shared-memory opt-in happens on a device's first capped
    call; here that call is being captured (in a fresh process)."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", FIRST_CALL_CAPTURED.format(root=root)],
                         capture_output=True, text=True, timeout=300,
                         env={**os.environ, "AR_CAPPED_KERNEL": "tma"})
    assert out.returncode == 0 and "ok" in out.stdout, out.stderr[-2000:]


@pytest.mark.parametrize("kind", KINDS)
def test_full_size_reduce_scatter_and_all_gather_on_64_sms(kind, dev):
    """P=8, 8 MiB shards / pieces (the bench's sizes): the capped kernels
    equal the uncapped kernels element for element, and every reduce-scatter
    output element equals the oracle's."""
    P, rc = 8, 2 * 1024 * 1024
    comm = init_comm(P, kind)
    try:
        sends = device_inputs("normal", 0, P, P * rc, dev, 1e-3)
        ref = [torch.empty(rc, device=dev) for _ in range(P)]
        got = [torch.empty(rc, device=dev) for _ in range(P)]
        ar.ar_reduce_scatter(comm, sends, ref, rc, ar.AR_FLOAT32, ar.AR_SUM, 0.125)
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 64)
        ar.ar_reduce_scatter(comm, sends, got, rc, ar.AR_FLOAT32, ar.AR_SUM, 0.125)
        gathered = [torch.empty(P * rc, device=dev) for _ in range(P)]
        ar.ar_all_gather(comm, got, gathered, rc, ar.AR_FLOAT32)
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 0)
        gathered_ref = [torch.empty(P * rc, device=dev) for _ in range(P)]
        ar.ar_all_gather(comm, ref, gathered_ref, rc, ar.AR_FLOAT32)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        for r in range(P):
            assert torch.equal(got[r].view(torch.int32), ref[r].view(torch.int32)), f"RS rank {r}"
            assert torch.equal(gathered[r].view(torch.int32), gathered_ref[r].view(torch.int32)), f"AG rank {r}"
        want = oracle.reduce_scatter(host_inputs(sends, "normal", 0, 1e-3), ar.AR_FLOAT32, oracle.SUM, 0.125)
        for s in range(P):
            assert_equal_every_element(got[s], want[s], f"capped reduce-scatter shard {s}")
        assert_equal_every_element(gathered[0], np.concatenate(want), "all-gather of the shards, rank 0")
    finally:
        ar.ar_destroy(comm)


def test_capped_kernel_option(dev, capfd):
    """AR_OPT_CAPPED_KERNEL switches the capped kernel at run time; other
    values are refused; uncapped calls are unaffected."""
    P, count = 8, 1 << 18
    comm = ar.ar_init(P)
    try:
        rng = np.random.default_rng(61)
        sends = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING)
        with pytest.raises(ar.ArError) as e:
            ar.ar_set_option(comm, ar.AR_OPT_CAPPED_KERNEL, 2)
        assert e.value.status == ar.AR_ERR_INVALID_ARG
        ar.ar_set_option(comm, ar.AR_OPT_DEBUG, 1)
        for blocks, kind, kernel in ((16, ar.AR_CAPPED_TMA, "tma_ring"), (16, ar.AR_CAPPED_WIDE, "wide_ring"),
                                     (0, ar.AR_CAPPED_TMA, "static_ring")):
            ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, blocks)
            ar.ar_set_option(comm, ar.AR_OPT_CAPPED_KERNEL, kind)
            ys = [torch.empty_like(x) for x in xs]
            ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
            torch.cuda.synchronize()
            assert f"kernel={kernel} " in capfd.readouterr().err
            pins.assert_bitwise(to_host(ys[2]), want[2], f"{kernel}")
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("P", [1, 3, 8])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_small_messages(P, dtype, kind, dev):
    """Capped calls on messages too small to give every block a tile: the
    wide kernel takes them (one partial block and the trailing partial
    vector), or with AR_CAPPED_TMA the 256-thread kernel does; every output
    element against the oracle."""
    rng = np.random.default_rng(1700 + 10 * P + dtype)
    comm = init_comm(P, kind)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        V = VEC[dtype]
        for count in (1, 2, V - 1, V + 1, 33, 1000, 4099, 1024 * V + 5):
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for op in OPS:
                for algo, oalgo in ((ar.AR_ALGO_RING, oracle.RING), (ar.AR_ALGO_TREE, oracle.TREE)):
                    scale = 0.125 if (op == ar.AR_SUM and dtype != ar.AR_INT32) else 1.0
                    outs = [Guarded(count, dtype, dev) for _ in range(P)]
                    ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, algo, scale)
                    torch.cuda.synchronize()
                    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                    want = oracle.allreduce(sends, dtype, op, oalgo, scale)
                    for r in range(P):
                        assert outs[r].guards_intact()
                        pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                            f"{kind} P={P} dtype={dtype} count={count} op={op} algo={algo} rank={r}")
        for rc in (V, 3 * V, 100 * V, 1025 * V):              # whole-vector shards: the capped kernels
            sends = pins.random_inputs(rng, P, P * rc, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            outs = [Guarded(rc, dtype, dev) for _ in range(P)]
            ar.ar_reduce_scatter(comm, xs, [o.tensor for o in outs], rc, dtype, ar.AR_MAX, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            want = oracle.reduce_scatter(sends, dtype, oracle.MAX, 1.0)
            for r in range(P):
                assert outs[r].guards_intact()
                pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"{kind} RS P={P} dtype={dtype} rc={rc} rank={r}")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("P,Q", [(9, 3), (13, 13), (72, 8)])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_many_ranks(P, Q, dtype, dev, capfd):
    """More than 8 ranks on 16 SMs: the pipelined kernel in 768-thread blocks
    (one per SM, grid-stride) for the ring, tree and hierarchical orders and
    the reduce-scatter; every output element against the oracle."""
    rng = np.random.default_rng(1900 + P + dtype)
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        ar.ar_set_option(comm, ar.AR_OPT_DEBUG, 1)
        V = VEC[dtype]
        for count in (1, V + 3, 1000, BLOCKS * 768 * V + 2 * V + 1, 3 * BLOCKS * 768 * V - 5):
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for op in (ar.AR_SUM, ar.AR_MAX):
                for algo in (ar.AR_ALGO_RING, ar.AR_ALGO_TREE, ar.AR_ALGO_HIER):
                    outs = [Guarded(count, dtype, dev) for _ in range(P)]
                    ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, algo, 1.0)
                    torch.cuda.synchronize()
                    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                    if algo == ar.AR_ALGO_HIER:
                        want = oracle.allreduce_hier(sends, Q, dtype, op)
                    else:
                        want = oracle.allreduce(sends, dtype, op, oracle.TREE if algo == ar.AR_ALGO_TREE else oracle.RING)
                    for r in range(P):
                        assert outs[r].guards_intact()
                        pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                            f"P={P} dtype={dtype} count={count} op={op} algo={algo} rank={r}")
        for rc in (V, 200 * V, BLOCKS * 768 * V // P + V):
            sends = pins.random_inputs(rng, P, P * rc, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            outs = [Guarded(rc, dtype, dev) for _ in range(P)]
            ar.ar_reduce_scatter(comm, xs, [o.tensor for o in outs], rc, dtype, ar.AR_SUM, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            want = oracle.reduce_scatter(sends, dtype, oracle.SUM, 1.0)
            for r in range(P):
                assert outs[r].guards_intact()
                pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"RS P={P} dtype={dtype} rc={rc} rank={r}")
        log = capfd.readouterr().err
        for k in ("wide_pipelined_ring", "wide_pipelined_tree", "wide_pipelined_hier", "wide_pipelined_reduce_scatter"):
            assert f"kernel={k} " in log, k
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("dtype", [ar.AR_BFLOAT16, ar.AR_INT32])
def test_capped_many_ranks_long_grid_stride(dtype, dev):
    """72 ranks on 16 SMs with about 21 column groups per block: the results
    leave through the store warp's two alternating shared-memory buffers many
    times over.  Every element of every rank against the oracle (every order,
    the hierarchical one with groups of 8), out of place and in place."""
    P, Q = 72, 8
    V = VEC[dtype]
    count = 21 * BLOCKS * 768 * V + 5 * V + 3
    kind = "int" if dtype == ar.AR_INT32 else "normal_bf16"
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        sends = device_inputs(kind, 5, P, count, dev, 1e-3)
        host = host_inputs(sends, kind, 5, 1e-3)
        for algo, oalgo, group in ((ar.AR_ALGO_RING, oracle.RING, None), (ar.AR_ALGO_TREE, oracle.TREE, None),
                                   (ar.AR_ALGO_HIER, None, Q)):
            op = ar.AR_MAX if algo == ar.AR_ALGO_TREE else ar.AR_SUM
            want = oracle_full(host, dtype, op, oalgo, 1.0, group=group)
            outs = [torch.empty_like(s) for s in sends]
            ar.ar_allreduce(comm, sends, outs, count, dtype, op, algo, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            for r in range(P):
                assert_equal_every_element(outs[r], want, f"algo={algo} rank {r}")
            inplace = [s.clone() for s in sends]
            ar.ar_allreduce(comm, inplace, inplace, count, dtype, op, algo, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            for r in range(P):
                assert torch.equal(inplace[r], outs[r]), f"in place, algo={algo} rank {r}"
    finally:
        ar.ar_destroy(comm)


def test_capped_at_the_rank_limit(dev):
    """AR_MAX_RANKS ranks on 16 SMs (the 768-thread pipelined kernel at its
    largest rank count): ring, tree, hierarchical (groups of 16) and the
    reduce-scatter, every element of every rank against the oracle."""
    P, Q, dtype = ar.AR_MAX_RANKS, 16, ar.AR_INT32
    V = VEC[dtype]
    count = 2 * BLOCKS * 768 * V + 3 * V + 2
    rng = np.random.default_rng(4100)
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, BLOCKS)
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        sends = pins.random_inputs(rng, P, count, dtype)
        xs = [to_device(a, dtype, dev) for a in sends]
        for algo, op in ((ar.AR_ALGO_RING, ar.AR_SUM), (ar.AR_ALGO_TREE, ar.AR_SUM), (ar.AR_ALGO_HIER, ar.AR_MIN)):
            outs = [Guarded(count, dtype, dev) for _ in range(P)]
            ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, algo, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            if algo == ar.AR_ALGO_HIER:
                want = oracle.allreduce_hier(sends, Q, dtype, op)
            else:
                want = oracle.allreduce(sends, dtype, op, oracle.TREE if algo == ar.AR_ALGO_TREE else oracle.RING)
            for r in range(P):
                assert outs[r].guards_intact()
                pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"P={P} algo={algo} rank={r}")
        rc = 64 * V + V
        sends = pins.random_inputs(rng, P, P * rc, dtype)
        xs = [to_device(a, dtype, dev) for a in sends]
        outs = [Guarded(rc, dtype, dev) for _ in range(P)]
        ar.ar_reduce_scatter(comm, xs, [o.tensor for o in outs], rc, dtype, ar.AR_SUM, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        want = oracle.reduce_scatter(sends, dtype, oracle.SUM, 1.0)
        for r in range(P):
            assert outs[r].guards_intact()
            pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"RS P={P} rank={r}")
    finally:
        ar.ar_destroy(comm)
