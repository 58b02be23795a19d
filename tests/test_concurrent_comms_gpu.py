"""Two communicators used at the same time from two streams.

Each communicator owns its LL / LL128 staging areas and its device epoch, so
calls on different communicators may run concurrently ("NCCL and NVSHMEM --
two GPU communication models, side by side": one communicator per group of
ranks, collectives on the caller's stream).  The LL kernels' waits stay
inside one block, so two such kernels never wait on each other.  Each
stream runs a chain of dependent in-place calls (LL, LL128, ring, tree) with
no host wait between them; every element of every rank is compared with the
oracle applied step by step.
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


ALGOS = (ar.AR_ALGO_LL, ar.AR_ALGO_RING, ar.AR_ALGO_LL128, ar.AR_ALGO_TREE)


def test_two_communicators_on_two_streams(dev):
    setups = [(8, 16384 - 4), (5, 1000 * 4 + 3)]          # (ranks, elements per rank): both LL-sized
    rng = np.random.default_rng(5100)
    comms, streams, xs, hosts = [], [], [], []
    try:
        for P, count in setups:
            comms.append(ar.ar_init(P))
            streams.append(torch.cuda.Stream())
            sends = [(s * np.float32(2.0 ** -20)).astype(np.float32)
                     for s in pins.random_inputs(rng, P, count, ar.AR_FLOAT32)]
            xs.append([to_device(s, ar.AR_FLOAT32, dev) for s in sends])
            hosts.append([s.copy() for s in sends])
        torch.cuda.synchronize()
        for rnd in range(6):
            for i, (P, count) in enumerate(setups):
                algo = ALGOS[(rnd + i) % len(ALGOS)]
                scale = 0.125 if rnd % 2 == 0 else 1.0
                with torch.cuda.stream(streams[i]):
                    ar.ar_allreduce(comms[i], xs[i], xs[i], count, ar.AR_FLOAT32, ar.AR_SUM, algo, scale,
                                    streams[i])
                oalgo = oracle.TREE if algo == ar.AR_ALGO_TREE else oracle.RING
                hosts[i] = oracle.allreduce(hosts[i], ar.AR_FLOAT32, oracle.SUM, oalgo, scale)
        torch.cuda.synchronize()
        for i, (P, count) in enumerate(setups):
            assert ar.ar_get_status(comms[i]) == ar.AR_SUCCESS
            for r in range(P):
                assert_equal_every_element(xs[i][r], hosts[i][r], f"communicator {i} rank {r}")
    finally:
        for c in comms:
            ar.ar_destroy(c)
