"""Tree and ring order (and the LL protocols) above eight ranks, over the tree
shapes the rank count produces ("NCCL and NVSHMEM -- two GPU communication models, side by side",
the double binary tree).

The kernel for P > 8 walks the in-order lowbit tree's right spine and folds
every complete subtree in blocks of seven inputs, with the nodes above them
on a small stack.  These rank counts cover whole trees (P = 2^k - 1), a root
without a right child (P = 2^k), spines of several steps, and complete
subtrees of lowbit 8 ... 128 (up to five stacked levels).  fp32 sums make any
change of association visible; int32 max checks the orders' shared result.
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import Guarded, to_device, to_host

pytestmark = pytest.mark.gpu

RANKS = [15, 16, 17, 31, 33, 63, 64, 65, 100, 127, 128, 129, 200, 255, 256]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("P", RANKS)
def test_tree_and_ring_orders_for_many_ranks(P, dev):
    rng = np.random.default_rng(500 + P)
    comm = ar.ar_init(P)
    try:
        for dtype, op, count in ((ar.AR_FLOAT32, ar.AR_SUM, 1001), (ar.AR_FLOAT32, ar.AR_SUM, 3),
                                 (ar.AR_INT32, ar.AR_MAX, 517), (ar.AR_BFLOAT16, ar.AR_SUM, 333)):
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for algo, oalgo in ((ar.AR_ALGO_TREE, oracle.TREE), (ar.AR_ALGO_RING, oracle.RING)):
                outs = [Guarded(count, dtype, dev) for _ in range(P)]
                ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, algo, 1.0)
                torch.cuda.synchronize()
                assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                want = oracle.allreduce(sends, dtype, op, oalgo, 1.0)
                for r in (0, P // 2, P - 1):
                    assert outs[r].guards_intact()
                    pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                        f"P={P} dtype={dtype} op={op} count={count} algo={algo} rank={r}")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("P", [17, 129, 256])
def test_ll_protocols_at_many_ranks(P, dev):
    """LL and LL128 with up to AR_MAX_RANKS ranks (the widest parameter block;
    LL stages several words per thread above 8 ranks, LL128 keeps every
    rank's block group resident at once), against the oracle's ring."""
    rng = np.random.default_rng(700 + P)
    comm = ar.ar_init(P)
    try:
        for algo in (ar.AR_ALGO_LL, ar.AR_ALGO_LL128):
            for count in (5, 1001, 16384):
                sends = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
                xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
                outs = [Guarded(count, ar.AR_FLOAT32, dev) for _ in range(P)]
                ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
                torch.cuda.synchronize()
                assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING, 1.0)
                for r in (0, P - 1):
                    assert outs[r].guards_intact()
                    pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"P={P} algo={algo} count={count} rank={r}")
    finally:
        ar.ar_destroy(comm)
