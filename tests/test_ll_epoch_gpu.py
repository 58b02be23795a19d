"""The LL / LL128 epoch on the device: CUDA-graph replay and the 32-bit wrap.

"Demystifying NVSHMEM" (the collectives paragraph): LL and LL128 carry each
payload with its arrival flag, so a reader must never accept a flag written
by an earlier call.  Each call's flag is a fresh epoch that the kernel takes
from device memory, so a captured call replayed many times still uses a new
value each time.  After 2^32 - 1 the kernel clears the staging area and
numbering restarts at 1; the wrap test plants words under epoch 1 first and
checks that the restarted epoch 1 does not accept them: with the producer
skipped, a call that accepted them would report success, while after the
clear every wait runs out (bounded, AR_ERR_TIMEOUT).
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu

LIMITS = {ar.AR_ALGO_LL: 65536, ar.AR_ALGO_LL128: 1 << 20}   # default per-rank limits, bytes


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def ring_want(sends, scale=1.0):
    return oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, oracle.RING, scale)


@pytest.mark.parametrize("algo", [ar.AR_ALGO_LL, ar.AR_ALGO_LL128])
def test_calls_across_the_wrap_stay_exact(algo, dev):
    P = 8
    comm = ar.ar_init(P)
    try:
        rng = np.random.default_rng(90 + algo)
        ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, 0xFFFFFFFD)
        for i in range(5):        # epochs 2^32-2, 2^32-1 (then cleared), 1, 2, 3
            count = int(rng.integers(1, LIMITS[algo] // 4 + 1))
            sends = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
            xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
            ys = [torch.full_like(x, float("nan")) for x in xs]
            ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 0.125)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS, f"call {i}"
            want = ring_want(sends, 0.125)
            for r in (0, P - 1):
                pins.assert_bitwise(to_host(ys[r]), want[r], f"call {i} count={count} rank={r}")
    finally:
        ar.ar_destroy(comm)


@pytest.mark.parametrize("algo", [ar.AR_ALGO_LL, ar.AR_ALGO_LL128])
def test_wrap_clears_words_of_the_old_epoch_one(algo, dev):
    P = 8
    comm = ar.ar_init(P)
    try:
        rng = np.random.default_rng(7 + algo)
        full = LIMITS[algo] // 4
        sends = pins.random_inputs(rng, P, full, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.empty_like(x) for x in xs]
        # 1: a full-size call under epoch 1 leaves epoch-1 words in every slot
        ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, 0)
        ar.ar_allreduce(comm, xs, ys, full, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        # 2: a call under the last epoch value that stages nothing (its waits
        # run out); it must still clear the staging area at its end
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 2000)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 1)
        ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, 0xFFFFFFFE)
        ar.ar_allreduce(comm, xs, ys, 4, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        # 3: epoch 1 again, nothing staged: had the old epoch-1 words survived,
        # every wait would accept them and the call would report success
        ar.ar_allreduce(comm, xs, ys, full, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        # 4: and the protocol works again afterwards
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 0)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 1 << 22)
        ar.ar_allreduce(comm, xs, ys, full, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        pins.assert_bitwise(to_host(ys[3]), ring_want(sends)[3], "after the wrap")
    finally:
        ar.ar_destroy(comm)


def test_ll_and_ll128_replayed_from_one_graph(dev):
    """One capture holding LL, LL128 and ring calls, replayed on new data."""
    P = 8
    comm = ar.ar_init(P)
    try:
        sizes = {ar.AR_ALGO_LL: 3001, ar.AR_ALGO_LL128: 70001, ar.AR_ALGO_RING: 4096}
        sends = {a: [torch.empty(n, device=dev) for _ in range(P)] for a, n in sizes.items()}
        recvs = {a: [torch.empty(n, device=dev) for _ in range(P)] for a, n in sizes.items()}

        def run_all():
            for a, n in sizes.items():
                ar.ar_allreduce(comm, sends[a], recvs[a], n, ar.AR_FLOAT32, ar.AR_SUM, a, 0.125)

        run_all()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                run_all()
        rng = np.random.default_rng(23)
        for replay in range(5):
            host = {a: pins.random_inputs(rng, P, n, ar.AR_FLOAT32) for a, n in sizes.items()}
            for a in sizes:
                for r in range(P):
                    sends[a][r].copy_(torch.from_numpy(host[a][r]))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            for a in sizes:
                want = ring_want(host[a], 0.125)
                for r in (0, 5):
                    pins.assert_bitwise(to_host(recvs[a][r]), want[r], f"replay {replay} algo {a} rank {r}")
    finally:
        ar.ar_destroy(comm)


def test_epoch_option_arguments(dev):
    comm = ar.ar_init(2)
    try:
        # the last value 2^32 - 1 is never "last used" when a call starts: the
        # call that uses it resets the state to 0
        for bad in (-1, 0xFFFFFFFF, 1 << 32):
            with pytest.raises(ar.ArError) as e:
                ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, bad)
            assert e.value.status == ar.AR_ERR_INVALID_ARG
        ar.ar_set_option(comm, ar.AR_OPT_LL_EPOCH, 0xFFFFFFFE)
    finally:
        ar.ar_destroy(comm)


def test_many_back_to_back_calls(dev):
    """20,000 LL / LL128 calls in a row on one stream, sizes changing: in each
    call the block that completes the count publishes the epoch the next call
    starts from.  Checked
    against the ring every few hundred calls and for the device status."""
    P = 8
    comm = ar.ar_init(P)
    try:
        rng = np.random.default_rng(2024)
        top = 16384
        sends = pins.random_inputs(rng, P, top, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.empty_like(x) for x in xs]
        ref = [torch.empty_like(x) for x in xs]
        counts = rng.integers(1, top + 1, size=20000)
        for i, n in enumerate(counts):
            algo = ar.AR_ALGO_LL if i % 2 == 0 else ar.AR_ALGO_LL128
            ar.ar_allreduce(comm, xs, ys, int(n), ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
            if i % 997 == 0:
                ar.ar_allreduce(comm, xs, ref, int(n), ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
                torch.cuda.synchronize()
                assert torch.equal(ys[i % P][:n].view(torch.int32), ref[i % P][:n].view(torch.int32)), f"call {i}"
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)
