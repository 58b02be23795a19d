"""Reduce-scatter and all-gather on the GPU against the CPU oracle, bit for bit.

"NCCL, NIXL, and Distributed GPU Communication", sections "Reduce-scatter"
and "All-gather".  Small cases run every rank count, data type and op, over
shard lengths that are and are not whole 16-byte vectors (the vector and the
element-wise kernels); the full-size case checks that reduce-scatter followed
by all-gather equals the ring all-reduce, element for element.
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import (VEC, Guarded, all_ranks_identical, assert_equal_every_element, device_inputs, host_inputs,
                      to_device, to_host)

pytestmark = pytest.mark.gpu

OPS = (ar.AR_SUM, ar.AR_MIN, ar.AR_MAX)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def comms(dev):
    made = {}

    def get(P):
        if P not in made:
            made[P] = ar.ar_init(P)
        return made[P]

    yield get
    torch.cuda.synchronize()
    for c in made.values():
        ar.ar_destroy(c)


def shard_counts(dtype):
    V = VEC[dtype]
    return sorted({1, 3, V - 1, V, 2 * V, 5 * V + 3, 1000, 4096, 3 * 128 * V + V})


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 9, 13, 72])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_reduce_scatter_small(P, dtype, dev, comms):
    rng = np.random.default_rng(200 + P * 3 + dtype)
    comm = comms(P)
    for rc in shard_counts(dtype):
        if P * rc > 200_000:
            continue
        sends = pins.random_inputs(rng, P, P * rc, dtype)
        xs = [to_device(a, dtype, dev) for a in sends]
        for op in OPS:
            scales = (1.0, 0.125) if (op == ar.AR_SUM and dtype != ar.AR_INT32) else (1.0,)
            for scale in scales:
                outs = [Guarded(rc, dtype, dev) for _ in range(P)]
                ar.ar_reduce_scatter(comm, xs, [o.tensor for o in outs], rc, dtype, op, scale)
                torch.cuda.synchronize()
                want = oracle.reduce_scatter(sends, dtype, op, scale)
                for r in range(P):
                    assert outs[r].guards_intact()
                    pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                        f"RS P={P} dtype={dtype} rc={rc} op={op} scale={scale} rank={r}")


@pytest.mark.parametrize("P", [1, 2, 3, 8, 13, 72])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_all_gather_small(P, dtype, dev, comms):
    rng = np.random.default_rng(300 + P * 3 + dtype)
    comm = comms(P)
    for sc in shard_counts(dtype):
        if P * sc > 200_000:
            continue
        sends = pins.random_inputs(rng, P, sc, dtype)
        xs = [to_device(a, dtype, dev) for a in sends]
        outs = [Guarded(P * sc, dtype, dev) for _ in range(P)]
        ar.ar_all_gather(comm, xs, [o.tensor for o in outs], sc, dtype)
        torch.cuda.synchronize()
        want = oracle.all_gather(sends, dtype)
        for r in range(P):
            assert outs[r].guards_intact()
            pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"AG P={P} dtype={dtype} sc={sc} rank={r}")


def test_in_place_layouts(dev, comms):
    """recvbuf at rank r's own shard inside its sendbuf (reduce-scatter), and
    sendbuf at rank r's own slot inside its recvbuf (all-gather)."""
    rng = np.random.default_rng(17)
    for P, rc in ((8, 1024), (8, 1001), (13, 64)):
        comm = comms(P)
        sends = pins.random_inputs(rng, P, P * rc, ar.AR_FLOAT32)
        want = oracle.reduce_scatter(sends, ar.AR_FLOAT32, ar.AR_SUM)
        big = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ar.ar_reduce_scatter(comm, big, [big[r][r * rc:(r + 1) * rc] for r in range(P)], rc,
                             ar.AR_FLOAT32, ar.AR_SUM)
        torch.cuda.synchronize()
        for r in range(P):
            pins.assert_bitwise(to_host(big[r][r * rc:(r + 1) * rc]), want[r], f"RS in place P={P} rank={r}")
        pieces = pins.random_inputs(rng, P, rc, ar.AR_FLOAT32)
        full = [torch.zeros(P * rc, device=dev) for _ in range(P)]
        for r in range(P):
            full[r][r * rc:(r + 1) * rc] = torch.from_numpy(pieces[r]).to(dev)
        ar.ar_all_gather(comm, [full[r][r * rc:(r + 1) * rc] for r in range(P)], full, rc, ar.AR_FLOAT32)
        torch.cuda.synchronize()
        want_ag = oracle.all_gather(pieces, ar.AR_FLOAT32)
        for r in range(P):
            pins.assert_bitwise(to_host(full[r]), want_ag[r], f"AG in place P={P} rank={r}")


def test_layout_errors(dev, comms):
    comm = comms(4)
    big = [torch.zeros(4 * 256, device=dev) for _ in range(4)]
    small = [torch.zeros(256, device=dev) for _ in range(4)]
    with pytest.raises(ar.ArError) as e:   # rank 1's shard placed at rank 0's offset
        ar.ar_reduce_scatter(comm, big, [small[0], big[1][:256], small[2], small[3]], 256, ar.AR_FLOAT32)
    assert e.value.status == ar.AR_ERR_INVALID_ARG
    with pytest.raises(ar.ArError) as e:   # not even element-aligned
        raw = torch.zeros(4096, dtype=torch.uint8, device=dev)
        ar.ar_all_gather(comm, [raw[2:].data_ptr(), small[1],
                                small[2], small[3]], big, 100, ar.AR_FLOAT32)
    assert e.value.status == ar.AR_ERR_INVALID_ARG
    # element-aligned but not 16-byte aligned: accepted (element-wise kernel)
    ar.ar_all_gather(comm, [small[0][1:], small[1][1:], small[2][1:], small[3][1:]], big, 100, ar.AR_FLOAT32)
    with pytest.raises(ar.ArError) as e:
        ar.ar_reduce_scatter(comm, big, small, 256, ar.AR_INT32, ar.AR_SUM, 0.5)
    assert e.value.status == ar.AR_ERR_UNSUPPORTED
    ar.ar_reduce_scatter(comm, big, small, 0, ar.AR_FLOAT32)  # no-op
    ar.ar_all_gather(comm, small, big, 0, ar.AR_FLOAT32)


def test_reduce_scatter_then_all_gather_is_the_ring_allreduce(dev, comms):
    """P=8, 2,097,152 fp32 per shard (64 MiB per rank), scale 1/8: RS + AG on
    the GPU equals the GPU ring all-reduce for every element, and every
    reduce-scatter output element equals the oracle's."""
    P, rc, sigma = 8, 2 * 1024 * 1024, 1e-3
    comm = comms(P)
    sends = device_inputs("normal", 0, P, P * rc, dev, sigma)
    shards = [torch.empty(rc, device=dev) for _ in range(P)]
    gathered = [torch.empty(P * rc, device=dev) for _ in range(P)]
    ref = [torch.empty(P * rc, device=dev) for _ in range(P)]
    ar.ar_reduce_scatter(comm, sends, shards, rc, ar.AR_FLOAT32, ar.AR_SUM, 0.125)
    ar.ar_all_gather(comm, shards, gathered, rc, ar.AR_FLOAT32)
    ar.ar_allreduce(comm, sends, ref, P * rc, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
    torch.cuda.synchronize()
    for r in range(P):
        assert torch.equal(gathered[r].view(torch.int32), ref[r].view(torch.int32)), f"rank {r}"
    assert all_ranks_identical(gathered)
    host = host_inputs(sends, "normal", 0, sigma)
    want = oracle.reduce_scatter(host, ar.AR_FLOAT32, oracle.SUM, 0.125)
    for s in range(P):
        assert_equal_every_element(shards[s], want[s], f"reduce-scatter shard {s}")
    assert_equal_every_element(gathered[0], np.concatenate(want), "all-gather of the shards, rank 0")
