"""Element counts past 2^31 (and past 2^32 for bf16): the kernels' 64-bit
index, chunk, split and tail arithmetic, against the oracle on sampled
outputs (every ring-chunk edge, the tree split, the tail, random indices).

The ring's chunk length, the tree split and the hierarchical sub-chunks follow
"NCCL, NIXL, and Distributed GPU Communication" (ring all-reduce = reduce-scatter
+ all-gather over P chunks) and "NCCL and NVSHMEM -- two GPU communication
models, side by side" (the double binary tree).  Inputs are made on the
device in pieces of 2^27 elements (bounded scratch memory); each test holds
at most about 90 GB and releases it before the next.
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
import synthetic
from gpu_util import TORCH, all_ranks_identical, check_sampled, host_columns, sample_indices, to_host

pytestmark = pytest.mark.gpu

PIECE = 1 << 27


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def release_memory():
    yield
    if torch.cuda.is_available():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def make_inputs(kind, seed, P, count, dtype, dev, sigma=1.0):
    out = []
    for r in range(P):
        t = torch.empty(count, dtype=TORCH[dtype], device=dev)
        for s in range(0, count, PIECE):
            n = min(PIECE, count - s)
            t[s:s + n] = synthetic.values_torch(kind, seed, r, s, n, dev, sigma)
        out.append(t)
    return out


def run(comm, sends, recvs, count, dtype, algo, scale=1.0, max_blocks=0):
    ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, max_blocks)
    ar.ar_allreduce(comm, sends, recvs, count, dtype, ar.AR_SUM, algo, scale)
    torch.cuda.synchronize()
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS


def test_p3_fp32_count_past_2_31(dev):
    """P=3 (rank-specialised kernel and, capped to 64 SMs, the TMA pipeline),
    2^31 + 2^20 + 3 fp32 per rank (8.6 GB): ring and tree, ragged tail."""
    P, count = 3, 2 ** 31 + 2 ** 20 + 3
    comm = ar.ar_init(P)
    try:
        sends = make_inputs("uniform", 21, P, count, ar.AR_FLOAT32, dev)
        recvs = [torch.empty_like(s) for s in sends]
        for algo, blocks, scale in ((ar.AR_ALGO_RING, 0, 1.0), (ar.AR_ALGO_TREE, 0, 0.5),
                                    (ar.AR_ALGO_RING, 64, 0.25), (ar.AR_ALGO_TREE, 64, 1.0)):
            for r in recvs:
                r.fill_(float("nan"))
            run(comm, sends, recvs, count, ar.AR_FLOAT32, algo, scale, blocks)
            check_sampled(recvs, sends, "uniform", 21, count, ar.AR_FLOAT32, ar.AR_SUM, algo, scale,
                          n_random=2048)
            assert all_ranks_identical(recvs), f"algo={algo} blocks={blocks}"
    finally:
        ar.ar_destroy(comm)


def test_p2_bf16_count_past_2_32(dev):
    """P=2, 2^32 + 13 bf16 per rank (8.6 GB): element indices beyond 32 bits,
    ring and tree, full grid and the TMA pipeline on 64 SMs."""
    P, count = 2, 2 ** 32 + 13
    comm = ar.ar_init(P)
    try:
        sends = make_inputs("uniform_bf16", 22, P, count, ar.AR_BFLOAT16, dev)
        recvs = [torch.empty_like(s) for s in sends]
        for algo, blocks in ((ar.AR_ALGO_RING, 0), (ar.AR_ALGO_TREE, 0), (ar.AR_ALGO_RING, 64),
                             (ar.AR_ALGO_TREE, 64)):
            for r in recvs:
                r.fill_(float("nan"))
            run(comm, sends, recvs, count, ar.AR_BFLOAT16, algo, 1.0, blocks)
            check_sampled(recvs, sends, "uniform_bf16", 22, count, ar.AR_BFLOAT16, ar.AR_SUM, algo, 1.0,
                          n_random=2048)
            assert all_ranks_identical(recvs), f"algo={algo} blocks={blocks}"
    finally:
        ar.ar_destroy(comm)


def test_p9_bf16_count_past_2_31_generic_kernel(dev):
    """P=9 (the kernel for any rank count), 2^31 + 9 bf16 per rank (4.3 GB):
    ring, tree and the hierarchical order in 3 groups of 3."""
    P, Q, count = 9, 3, 2 ** 31 + 9
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        sends = make_inputs("uniform_bf16", 23, P, count, ar.AR_BFLOAT16, dev)
        recvs = [torch.empty_like(s) for s in sends]
        for algo in (ar.AR_ALGO_RING, ar.AR_ALGO_TREE):
            run(comm, sends, recvs, count, ar.AR_BFLOAT16, algo)
            check_sampled(recvs, sends, "uniform_bf16", 23, count, ar.AR_BFLOAT16, ar.AR_SUM, algo, 1.0,
                          n_random=1024)
        run(comm, sends, recvs, count, ar.AR_BFLOAT16, ar.AR_ALGO_HIER)
        idx = sample_indices(count, Q, ar.AR_BFLOAT16, n_random=1024, seed=24)
        V, G = 8, P // Q
        L1 = -(-(-(-count // Q)) // V) * V            # intra-group chunk length
        edges = []
        for c1 in range(Q):
            len1 = max(0, min(L1, count - c1 * L1))
            L2 = -(-(-(-len1 // G)) // V) * V          # sub-chunk length inside chunk c1
            edges += [c1 * L1 + c2 * L2 + d for c2 in range(1, G) for d in (-1, 0, 1)]
        idx = np.union1d(idx, np.array([e for e in edges if 0 <= e < count], dtype=np.int64))
        cols = host_columns("uniform_bf16", 23, P, idx)
        want = oracle.allreduce_hier_sampled(cols, idx, count, Q, ar.AR_BFLOAT16, oracle.SUM, 1.0)
        it = torch.from_numpy(idx).to(dev)
        for r in (0, 4, 8):
            pins.assert_bitwise(to_host(recvs[r].index_select(0, it)), want, f"hier rank {r}")
        assert all_ranks_identical(recvs)
    finally:
        ar.ar_destroy(comm)


def test_p2_reduce_scatter_and_all_gather_past_2_31(dev):
    """P=2, shards of 2^31 + 4 fp32 (8.6 GB): reduce-scatter (full grid and on
    64 SMs) against the oracle's ring all-reduce of the whole input (shard c =
    ring chunk c), then all-gather of the shards (bit copies)."""
    P, rc = 2, 2 ** 31 + 4
    comm = ar.ar_init(P)
    try:
        sends = make_inputs("uniform", 25, P, P * rc, ar.AR_FLOAT32, dev)
        shards = [torch.empty(rc, device=dev) for _ in range(P)]
        rng = np.random.default_rng(26)
        idx = np.unique(np.concatenate([rng.integers(0, P * rc, 1024),
                                        [0, 1, rc - 1, rc, rc + 1, P * rc - 1, 2 ** 31, 2 ** 32]]))
        cols = host_columns("uniform", 25, P, idx)
        want = oracle.allreduce_sampled(cols, idx, P * rc, ar.AR_FLOAT32, oracle.SUM, oracle.RING, 0.5)
        it = torch.from_numpy(idx).to(dev)
        for blocks in (0, 64):
            for s in shards:
                s.fill_(float("nan"))
            ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, blocks)
            ar.ar_reduce_scatter(comm, sends, shards, rc, ar.AR_FLOAT32, ar.AR_SUM, 0.5)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            got = np.empty(len(idx), dtype=np.float32)
            for c in range(P):
                sel = (idx >= c * rc) & (idx < (c + 1) * rc)
                local = torch.from_numpy(idx[sel] - c * rc).to(dev)
                got[sel] = to_host(shards[c].index_select(0, local))
            pins.assert_bitwise(got, want, f"reduce-scatter blocks={blocks}")
        del sends
        torch.cuda.empty_cache()
        gathered = [torch.empty(P * rc, device=dev) for _ in range(P)]
        for blocks in (0, 64):
            for g in gathered:
                g.fill_(float("nan"))
            ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, blocks)
            ar.ar_all_gather(comm, shards, gathered, rc, ar.AR_FLOAT32)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            for r in range(P):
                pins.assert_bitwise(to_host(gathered[r].index_select(0, it)), want,
                                    f"all-gather blocks={blocks} rank {r}")
                for c in range(P):
                    assert torch.equal(gathered[r][c * rc:(c + 1) * rc].view(torch.int32),
                                       shards[c].view(torch.int32)), f"all-gather rank {r} piece {c}"
    finally:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, 0)
        ar.ar_destroy(comm)
