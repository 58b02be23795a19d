"""The all-reduce entry point that allocates no device memory.

Some callers of this library cannot allocate device memory: their device
memory belongs to a framework's pool, they run in a latency-critical loop
where cudaMalloc / cudaFree may synchronize the device, or they may not
allocate after start-up.  ar_allreduce_ll_noalloc serves them from one
fixed array compiled into the library.  These tests call it through the C
ABI and check its results against the CPU oracle in the ring order (which
the LL protocol follows) for 1, 3 and 8 ranks, every data type and op, and
counts from one element to the array's 64 KiB limit, and, twice in a row,
against the communicator-based ar_allreduce (LL) on the same inputs -- bit
for bit, the tolerance of every fp32 test here.  They then check that
requests beyond the array's limits are rejected.  The file is collected last
and passes alone in a fresh process as well as after the other tests (the
array keeps the last call's contents; each call must still give its own
result).
"""
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


# (dtype, op, scale): fp32 sum with the DDP mean, bf16 sum (odd counts end in a
# 2-byte half of the last staged word), int32 min and max
CASES = [(ar.AR_FLOAT32, ar.AR_SUM, 0.125), (ar.AR_BFLOAT16, ar.AR_SUM, 1.0),
         (ar.AR_INT32, ar.AR_MIN, 1.0), (ar.AR_INT32, ar.AR_MAX, 1.0)]


@pytest.mark.parametrize("P", [1, 3, 8])
def test_matches_the_oracle(P, dev):
    """Every element of every rank against the oracle's ring order; fewer
    ranks than the array's 8 slots, counts 1 and 7 and the 64 KiB maximum."""
    rng = np.random.default_rng(500 + P)
    for dtype, op, scale in CASES:
        esize = 2 if dtype == ar.AR_BFLOAT16 else 4
        for count in (1, 7, ar.AR_NOALLOC_MAX_BYTES // esize - (1 if dtype == ar.AR_BFLOAT16 else 0),
                      ar.AR_NOALLOC_MAX_BYTES // esize):
            sends_np = pins.random_inputs(rng, P, count, dtype)
            sends = [to_device(a, dtype, dev) for a in sends_np]
            outs = [Guarded(count, dtype, dev) for _ in range(P)]
            status = ar.ar_allreduce_ll_noalloc(sends, [o.tensor for o in outs], count, dtype, op,
                                                scale, wait_status=True)
            assert status == ar.AR_SUCCESS
            want = oracle.allreduce(sends_np, dtype, op, oracle.RING, scale)
            for r in range(P):
                assert outs[r].guards_intact(), f"write outside rank {r}'s receive buffer"
                pins.assert_bitwise(to_host(outs[r].tensor), want[r],
                                    f"P={P} dtype={dtype} op={op} count={count} rank={r}")


def test_two_calls_match_the_communicator_entry_point(dev):
    P = 8
    comm = ar.ar_init(P)
    try:
        rng = np.random.default_rng(77)
        # call 1: 5000 fp32 per rank with the DDP scale; call 2: the full 64 KiB per rank
        for count, scale in ((5000, 0.125), (ar.AR_NOALLOC_MAX_BYTES // 4, 1.0)):
            sends_np = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
            sends = [to_device(a, ar.AR_FLOAT32, dev) for a in sends_np]
            want = [torch.empty_like(s) for s in sends]
            got = [torch.full_like(s, float("nan")) for s in sends]
            ar.ar_allreduce(comm, sends, want, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL, scale)
            status = ar.ar_allreduce_ll_noalloc(sends, got, count, ar.AR_FLOAT32, ar.AR_SUM, scale,
                                                wait_status=True)
            torch.cuda.synchronize()
            assert status == ar.AR_SUCCESS
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            for r in range(P):
                pins.assert_bitwise(to_host(got[r]), to_host(want[r]), f"count={count} rank={r}")
    finally:
        ar.ar_destroy(comm)


def test_requests_beyond_the_array_are_rejected(dev):
    too_many = [torch.zeros(16, device=dev) for _ in range(ar.AR_NOALLOC_MAX_RANKS + 1)]
    outs = [torch.zeros(16, device=dev) for _ in too_many]
    with pytest.raises(ar.ArError) as e:
        ar.ar_allreduce_ll_noalloc(too_many, outs, 16, ar.AR_FLOAT32)
    assert e.value.status == ar.AR_ERR_UNSUPPORTED
    n = ar.AR_NOALLOC_MAX_BYTES // 4 + 1
    big = [torch.zeros(n, device=dev) for _ in range(2)]
    big_out = [torch.zeros(n, device=dev) for _ in range(2)]
    with pytest.raises(ar.ArError) as e:
        ar.ar_allreduce_ll_noalloc(big, big_out, n, ar.AR_FLOAT32)
    assert e.value.status == ar.AR_ERR_UNSUPPORTED
