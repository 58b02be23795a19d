"""LL128 (128-byte lines: 120 payload bytes + a release-published flag word)
against the oracle's ring order, bit for bit ("Demystifying NVSHMEM", the
collectives paragraph: LL / LL128 pack data and arrival flag together)."""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import Guarded, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def line_counts(dtype):
    """Counts around whole 120-byte lines and up to the 1 MiB limit."""
    per_line = 60 if dtype == ar.AR_BFLOAT16 else 30
    top = (1 << 20) // (2 if dtype == ar.AR_BFLOAT16 else 4)
    return sorted({1, per_line - 1, per_line, per_line + 1, 2 * per_line + 1, 1000, 12345, top - 1, top})


@pytest.mark.parametrize("P", [1, 2, 8, 13])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_ll128_line_boundaries_and_limit(P, dtype, dev):
    rng = np.random.default_rng(70 + P + 10 * dtype)
    comm = ar.ar_init(P)
    try:
        for count in line_counts(dtype):
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            for op in (ar.AR_SUM, ar.AR_MAX):
                scale = 0.125 if (op == ar.AR_SUM and dtype != ar.AR_INT32) else 1.0
                outs = [Guarded(count, dtype, dev) for _ in range(P)]
                ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, op, ar.AR_ALGO_LL128, scale)
                torch.cuda.synchronize()
                assert ar.ar_get_status(comm) == ar.AR_SUCCESS
                want = oracle.allreduce(sends, dtype, op, oracle.RING, scale)
                for r in range(P):
                    assert outs[r].guards_intact()
                    pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                        f"LL128 P={P} dtype={dtype} count={count} op={op} rank={r}")
    finally:
        ar.ar_destroy(comm)


def test_ll_ll128_ring_interleaved(dev):
    """LL, LL128 and ring calls interleaved on one communicator stay exact."""
    rng = np.random.default_rng(9)
    comm = ar.ar_init(8)
    try:
        for i in range(40):
            algo = (ar.AR_ALGO_LL, ar.AR_ALGO_LL128, ar.AR_ALGO_RING)[i % 3]
            limit = 16384 if algo == ar.AR_ALGO_LL else 262144
            count = int(rng.integers(1, limit + 1))
            sends = pins.random_inputs(rng, 8, count, ar.AR_FLOAT32)
            xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
            ys = [torch.empty_like(x) for x in xs]
            ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
            torch.cuda.synchronize()
            want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING)
            pins.assert_bitwise(to_host(ys[i % 8]), want[i % 8], f"call {i} algo={algo} count={count}")
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)


def test_ll128_bounded_wait_limit_and_capture(dev):
    comm = ar.ar_init(8)
    try:
        rng = np.random.default_rng(4)
        sends = pins.random_inputs(rng, 8, 5000, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.zeros_like(x) for x in xs]
        # no line is ever published: every flag wait runs out and reports
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 2000)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 1)
        ar.ar_allreduce(comm, xs, ys, 5000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL128, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 0)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 1 << 22)
        ar.ar_allreduce(comm, xs, ys, 5000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL128, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        pins.assert_bitwise(to_host(ys[2]), oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING)[2],
                            "LL128 after a timed-out call")
        # above the limit, and a lowered limit
        big = [torch.zeros(262145, device=dev) for _ in range(8)]
        with pytest.raises(ar.ArError) as e:
            ar.ar_allreduce(comm, big, big, 262145, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL128, 1.0)
        assert e.value.status == ar.AR_ERR_UNSUPPORTED
        ar.ar_set_option(comm, ar.AR_OPT_LL128_MAX_BYTES, 4096)
        with pytest.raises(ar.ArError):
            ar.ar_allreduce(comm, xs, ys, 5000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL128, 1.0)
        # captured under the lowered limit and replayed twice
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                ar.ar_allreduce(comm, xs, ys, 500, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL128, 1.0)
        for _ in range(2):
            ys[1].zero_()
            g.replay()
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            pins.assert_bitwise(to_host(ys[1])[:500],
                                oracle.allreduce([a[:500] for a in sends], ar.AR_FLOAT32, oracle.SUM,
                                                 oracle.RING)[1],
                                "LL128 call replayed from the capture")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("P", [2, 8, 13])
def test_ll_at_its_largest_limit(P, dev):
    """LL with its limit raised to the 1 MiB maximum (AR_LL_MAX_BYTES at
    ar_init): past about 32 words per block per resident wave the slices
    widen beyond one word per thread, so threads stage and receive several
    words each.  Every element against the oracle's ring order, the epoch
    wrap included."""
    import os

    old = os.environ.get("AR_LL_MAX_BYTES")
    os.environ["AR_LL_MAX_BYTES"] = str(1 << 20)
    try:
        comm = ar.ar_init(P)
    finally:
        if old is None:
            os.environ.pop("AR_LL_MAX_BYTES", None)
        else:
            os.environ["AR_LL_MAX_BYTES"] = old
    try:
        rng = np.random.default_rng(1300 + P)
        cases = [(ar.AR_FLOAT32, 262144, 0.125), (ar.AR_FLOAT32, 200_003, 1.0), (ar.AR_BFLOAT16, 524287, 1.0),
                 (ar.AR_INT32, 150_001, 1.0)]
        for dtype, count, scale in cases:
            sends = pins.random_inputs(rng, P, count, dtype)
            xs = [to_device(a, dtype, dev) for a in sends]
            outs = [Guarded(count, dtype, dev) for _ in range(P)]
            ar.ar_allreduce(comm, xs, [o.tensor for o in outs], count, dtype, ar.AR_SUM, ar.AR_ALGO_LL, scale)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            want = oracle.allreduce(sends, dtype, oracle.SUM, oracle.LL, scale)
            for r in (0, P - 1):
                assert outs[r].guards_intact()
                pins.assert_bitwise(to_host(outs[r].tensor), want[r], f"LL 1 MiB P={P} dtype={dtype} count={count} rank={r}")
        ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, 2**32 - 3)       # across the wrap at this size
        for i in range(4):
            sends = pins.random_inputs(rng, P, 262144, ar.AR_FLOAT32)
            xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
            ys = [torch.empty_like(x) for x in xs]
            ar.ar_allreduce(comm, xs, ys, 262144, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.LL)
            pins.assert_bitwise(to_host(ys[1 % P]), want[1 % P], f"LL 1 MiB wrap call {i}")
    finally:
        ar.ar_destroy(comm)
