"""Hierarchical all-reduce order on the GPU against the CPU oracle, bit for bit.

lecture_068 page, section 06: reduce-scatter inside each node, ring
all-reduce between nodes, all-gather inside each node; here P = G groups of
Q consecutive emulated ranks (72 = 9 x 8 is one NVL72 rack of 8-GPU boards).
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import (Guarded, all_ranks_identical, assert_equal_every_element, device_inputs, host_inputs,
                      oracle_full, to_device, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("P,Q", [(2, 1), (4, 2), (6, 3), (8, 4), (8, 8), (9, 3), (12, 4), (16, 8),
                                 (72, 8), (72, 9), (72, 1), (128, 8), (256, 16), (256, 256)])
def test_hier_small(P, Q, dev):
    rng = np.random.default_rng(900 + P * 7 + Q)
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        for dtype in (ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32):
            V = 8 if dtype == ar.AR_BFLOAT16 else 4
            for count in sorted({1, V + 1, P * V - 1, 1000, 4099, 3 * 128 * V + 7}):
                sends = pins.random_inputs(rng, P, count, dtype)
                xs = [to_device(a, dtype, dev) for a in sends]
                for op in (ar.AR_SUM, ar.AR_MIN, ar.AR_MAX):
                    scale = 0.125 if (op == ar.AR_SUM and dtype != ar.AR_INT32) else 1.0
                    outs = [Guarded(count, dtype, dev) for _ in range(P)]
                    ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, ar.AR_ALGO_HIER, scale)
                    torch.cuda.synchronize()
                    want = oracle.allreduce_hier(sends, Q, dtype, op, scale)
                    for r in (0, P // 2, P - 1):
                        assert outs[r].guards_intact()
                        pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                            f"hier P={P} Q={Q} dtype={dtype} count={count} op={op}")
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)


def test_hier_full_size_p72(dev):
    """P=72 in 9 groups of 8, 4,194,304 elements per rank (16 MiB): fp32 every
    element against the oracle; int32 exact, and equal to the ring (integers)."""
    P, Q, count = 72, 8, 4 * 1024 * 1024
    comm = ar.ar_init(P)
    try:
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, Q)
        sends = device_inputs("normal", 3, P, count, dev, 1e-3)
        recvs = [torch.empty_like(s) for s in sends]
        ar.ar_allreduce(comm, sends, recvs, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_HIER, 1.0 / 72)
        torch.cuda.synchronize()
        host = host_inputs(sends, "normal", 3, 1e-3)
        want = oracle_full(host, ar.AR_FLOAT32, oracle.SUM, None, 1.0 / 72, group=Q)
        assert_equal_every_element(recvs[0], want, "P=72 hier fp32 rank 0")
        assert all_ranks_identical(recvs)
        del sends, recvs
        ints = device_inputs("int", 0, P, count, dev)
        a = [torch.empty_like(s) for s in ints]
        b = [torch.empty_like(s) for s in ints]
        ar.ar_allreduce(comm, ints, a, count, ar.AR_INT32, ar.AR_SUM, ar.AR_ALGO_HIER, 1.0)
        ar.ar_allreduce(comm, ints, b, count, ar.AR_INT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
        torch.cuda.synchronize()
        exact = torch.zeros(count, dtype=torch.int64, device=dev)
        for s in ints:
            exact += s.long()
        assert torch.equal(a[0], b[0]) and torch.equal(a[0], exact.to(torch.int32))
        assert all_ranks_identical(a)
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)


def test_hier_group_option(dev):
    comm = ar.ar_init(12)
    try:
        with pytest.raises(ar.ArError):
            ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, 5)        # does not divide 12
        x = [torch.zeros(64, device=dev) for _ in range(12)]
        with pytest.raises(ar.ArError) as e:                      # default group 8 does not divide 12
            ar.ar_allreduce(comm, x, x, 64, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_HIER, 1.0)
        assert e.value.status == ar.AR_ERR_UNSUPPORTED
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, 4)
        ar.ar_allreduce(comm, x, x, 64, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_HIER, 1.0)
        assert ar.ar_select_algo(comm, 64, ar.AR_FLOAT32, ar.AR_ALGO_HIER) == ar.AR_ALGO_HIER
        assert ar.ar_select_algo(comm, 64, ar.AR_FLOAT32, ar.AR_ALGO_AUTO) != ar.AR_ALGO_HIER
    finally:
        ar.ar_destroy(comm)
