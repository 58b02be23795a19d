"""Ring-chunk edges and the tree split on the GPU, made visible by the data.

Ranks c, c+1, c+2, c+3 (mod P) hold 2^24, 1, 1, -2^24 (exact in fp32 and
bf16) and every other rank holds 0.  A fold that meets 2^24 before the two 1s
absorbs them and ends at 0; a fold that meets a 1 first ends at 2.  In the
ring order chunk k starts at rank k, so chunks c+1, c+2 and c+3 reduce to 2
and every other chunk to 0: the edges c|c+1 and c+3|c+4 are 0|2 steps.  The
pattern runs from every start rank c, so every chunk edge (and every
reduce-scatter shard edge) is such a step at least once, and an edge off by
even one 16-byte vector changes whole elements -- which random data, whose
fp32 sums are mostly exact, rarely shows.  Every element is compared with the
oracle, whose own edges are pinned by hand-worked boundaries.  The ring
chunks and the split
follow "NCCL, NIXL, and Distributed GPU Communication" (section
"Reduce-scatter") and "NCCL and NVSHMEM -- two GPU communication models,
side by side" (the double binary tree).
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import init_comm, oracle_full, to_device, to_host

pytestmark = pytest.mark.gpu

COUNTS = (7, 9, 17, 40, 100, 1000, 4099, 65536 + 13)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def crafted(P, count, dtype, c=0):
    """2^24, 1, 1, -2^24 on ranks c .. c+3 (mod P), 0 elsewhere."""
    base = [2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)] + [0.0] * (P - 4)
    vals = [base[(r - c) % P] for r in range(P)]
    sends = [np.full(count, v, dtype=np.float32) for v in vals]
    if dtype == ar.AR_BFLOAT16:
        sends = [pins.bf16_bits_torch(x) for x in sends]
    return sends


def check(comm, sends, count, dtype, algo, dev, want, tag):
    P = len(sends)
    xs = [to_device(s, dtype, dev) for s in sends]
    outs = [torch.empty_like(x) for x in xs]
    ar.ar_allreduce(comm, xs, outs, count, dtype, ar.AR_SUM, algo, 1.0)
    torch.cuda.synchronize()
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    for r in (0, P - 1):
        w = want if isinstance(want, np.ndarray) else want[r]
        pins.assert_bitwise(to_host(outs[r]), w, f"{tag} rank {r}")


def start_ranks(P, count=None):
    """Every start rank; at 72 ranks only for the two counts whose chunks span
    several vectors (the others leave most chunks empty or one vector long)."""
    if P > 12 and count is not None and count < 4096:
        return [0]
    return list(range(P))


@pytest.mark.parametrize("P,Q", [(4, 2), (5, 0), (8, 4), (12, 4), (72, 8)])
def test_edges_every_algorithm(P, Q, dev):
    comm = ar.ar_init(P)
    try:
        if Q:
            ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        for dtype in (ar.AR_FLOAT32, ar.AR_BFLOAT16):
            esize = 2 if dtype == ar.AR_BFLOAT16 else 4
            for count in COUNTS:
                for c in start_ranks(P, count):
                    sends = crafted(P, count, dtype, c)
                    ring = oracle_full(sends, dtype, oracle.SUM, oracle.RING)
                    tree = oracle_full(sends, dtype, oracle.SUM, oracle.TREE)
                    algos = [(ar.AR_ALGO_RING, ring), (ar.AR_ALGO_TREE, tree)]
                    if count * esize <= 65536:
                        algos.append((ar.AR_ALGO_LL, ring))
                    if count * esize <= 1 << 20:
                        algos.append((ar.AR_ALGO_LL128, ring))
                    if Q:
                        algos.append((ar.AR_ALGO_HIER, oracle_full(sends, dtype, oracle.SUM, None, group=Q)))
                    for algo, want in algos:
                        check(comm, sends, count, dtype, algo, dev, want,
                              f"P={P} c={c} dtype={dtype} count={count} algo={algo}")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("kind", ["wide", "tma"])
@pytest.mark.parametrize("P", [4, 8])
def test_edges_on_a_few_sms(P, kind, dev):
    """Capped to 8 SMs: the wide kernel, and the TMA pipeline, whose tiles are
    loaded rotated per ring chunk, so a chunk edge inside a tile takes the
    per-element path."""
    comm = init_comm(P, kind)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 8)
        for dtype in (ar.AR_FLOAT32, ar.AR_BFLOAT16):
            for count in (65536 + 13, (1 << 20) + 5, 3 * (1 << 20) + 1000):
                for c in start_ranks(P):
                    sends = crafted(P, count, dtype, c)
                    for algo, oalgo in ((ar.AR_ALGO_RING, oracle.RING), (ar.AR_ALGO_TREE, oracle.TREE)):
                        if algo == ar.AR_ALGO_TREE and c % 2:
                            continue                       # the split: every other start rank suffices
                        want = oracle_full(sends, dtype, oracle.SUM, oalgo)
                        check(comm, sends, count, dtype, algo, dev, want,
                              f"TMA P={P} c={c} dtype={dtype} count={count} algo={algo}")
    finally:
        ar.ar_destroy(comm)


def interleaved(P, Q, count, dtype):
    """Group g's first rank holds the g-th of 2^24, 1, 1, -2^24 (0 from the
    fifth group on); every other rank holds 0.  Each group's partial is then
    that value, and the fold across groups shows its start group: the
    hierarchical sub-chunk edges become visible."""
    vals = [2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)]
    sends = [np.zeros(count, dtype=np.float32) for _ in range(P)]
    for g in range(min(4, P // Q)):
        sends[g * Q][:] = vals[g]
    if dtype == ar.AR_BFLOAT16:
        sends = [pins.bf16_bits_torch(x) for x in sends]
    return sends


@pytest.mark.parametrize("P,Q", [(8, 2), (12, 3), (16, 4), (72, 8)])
def test_hierarchical_subchunk_edges(P, Q, dev):
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        for dtype in (ar.AR_FLOAT32, ar.AR_BFLOAT16):
            for count in COUNTS:
                sends = interleaved(P, Q, count, dtype)
                want = oracle.allreduce_hier(sends, Q, dtype, oracle.SUM)
                check(comm, sends, count, dtype, ar.AR_ALGO_HIER, dev, want,
                      f"hier sub-chunks P={P} Q={Q} dtype={dtype} count={count}")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("kind", ["wide", "tma"])
@pytest.mark.parametrize("P", [4, 8, 12])
def test_reduce_scatter_shard_edges(P, kind, dev):
    """Shard s is ring chunk s, folded from rank s: with the crafted data
    started at rank c, shards c+1..c+3 reduce to 2 and the others to 0, so a
    tile that crosses a shard edge and keeps the wrong order shows; every start
    rank runs, so every shard edge is a 0|2 step once.  Element-wise shards
    (not whole vectors), whole-vector shards, and 8 SMs (P <= 8: the wide
    kernel or the TMA pipeline)."""
    comm = init_comm(P, kind)
    try:
        for dtype in (ar.AR_FLOAT32, ar.AR_BFLOAT16):
            for rc, blocks in ((5, 0), (1003, 0), (1024, 0), (65536 + 8, 0), (65536 + 8, 8), (3 * 4096 + 8, 8)):
                if blocks and P > 8:
                    continue
                for c in start_ranks(P):
                    sends = crafted(P, P * rc, dtype, c)
                    want = oracle.reduce_scatter(sends, dtype, oracle.SUM, 1.0)
                    xs = [to_device(s, dtype, dev) for s in sends]
                    shards = [torch.empty(rc, dtype=xs[0].dtype, device=dev) for _ in range(P)]
                    ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, blocks)
                    ar.ar_reduce_scatter(comm, xs, shards, rc, dtype, ar.AR_SUM, 1.0)
                    torch.cuda.synchronize()
                    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                    for s in range(P):
                        pins.assert_bitwise(to_host(shards[s]), want[s],
                                            f"RS shard {s} P={P} c={c} dtype={dtype} rc={rc} blocks={blocks}")
    finally:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 0)
        ar.ar_destroy(comm)
