"""GPU path (through the C ABI) against the CPU oracle, bit for bit.

Small cases run every rank count, data type, op and algorithm over ragged
sizes and compare all P outputs element by element with the oracle; the
full-size cases run the workloads at their real sizes, in the launch
configuration the benchmark uses, and compare every element of rank 0's
output with the oracle run on host copies of the same inputs, plus every
rank against rank 0 on the device (all ranks identical) and properties that
hold at any size (integer results equal to the exact sum, fp32 error bounds).

Tolerance: fp32 and int32 must match the oracle's combination order exactly;
for bf16 the contract allows 1 bf16 ulp (fp32 accumulation), but the kernels
perform the same operations in the same order, so the tests require 0.
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import (TORCH, VEC, Guarded, all_ranks_identical, assert_equal_every_element, device_inputs,
                      host_inputs, oracle_full, to_device, to_host)

pytestmark = pytest.mark.gpu

OPS = (ar.AR_SUM, ar.AR_MIN, ar.AR_MAX)
ALGOS = (ar.AR_ALGO_RING, ar.AR_ALGO_TREE, ar.AR_ALGO_LL, ar.AR_ALGO_LL128)
# LL and LL128 are transports: they fold in the ring order
ORACLE_ALGO = {ar.AR_ALGO_RING: oracle.RING, ar.AR_ALGO_TREE: oracle.TREE, ar.AR_ALGO_LL: oracle.LL,
               ar.AR_ALGO_LL128: oracle.RING}


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
        assert ar.ar_get_status(c) == ar.AR_SUCCESS
        ar.ar_destroy(c)


def small_counts(P, dtype):
    V = VEC[dtype]
    tiles = 3 * 256 * 2 * V + 5        # several tiles of the rank-specialised kernel + ragged tail
    return sorted({1, 2, 3, V - 1, V, V + 1, P * V - 1, P * V, P * V + 1, 1000, 4096 + 3, tiles})


def run_guarded(comm, sends_np, dtype, op, algo, scale, dev, stream=None):
    P = len(sends_np)
    count = len(sends_np[0])
    sends = [to_device(s, dtype, dev) for s in sends_np]
    outs = [Guarded(count, dtype, dev) for _ in range(P)]
    ar.ar_allreduce(comm, sends, [o.tensor for o in outs], count, dtype, op, algo, scale, stream)
    torch.cuda.synchronize()
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    for o in outs:
        assert o.guards_intact(), "write outside the receive buffer"
    return [to_host(o.tensor) for o in outs]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 72])
@pytest.mark.parametrize("dtype", [ar.AR_FLOAT32, ar.AR_BFLOAT16, ar.AR_INT32])
def test_small_exhaustive(P, dtype, dev, comms):
    rng = np.random.default_rng(1000 * P + dtype)
    comm = comms(P)
    for count in small_counts(P, dtype):
        sends = pins.random_inputs(rng, P, count, dtype)
        for op in OPS:
            for algo in ALGOS:
                scales = (1.0, 0.125) if (op == ar.AR_SUM and dtype != ar.AR_INT32) else (1.0,)
                for scale in scales:
                    got = run_guarded(comm, sends, dtype, op, algo, scale, dev)
                    want = oracle.allreduce(sends, dtype, op, ORACLE_ALGO[algo], scale)
                    for r in range(P):
                        pins.assert_bitwise(got[r], want[r], f"P={P} dtype={dtype} count={count} "
                                                             f"op={op} algo={algo} scale={scale} rank={r}")


def test_worked_example_on_gpu(dev, comms):
    """g0 + g1 + g2 + g3 on every rank ("NCCL, NIXL, ...", section "All-reduce")."""
    rng = np.random.default_rng(3)
    g = [rng.integers(-1000, 1001, size=4096).astype(np.float32) for _ in range(4)]
    exact = sum(x.astype(np.int64) for x in g).astype(np.float32)
    for algo in ALGOS:
        got = run_guarded(comms(4), g, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0, dev)
        for r in range(4):
            pins.assert_bitwise(got[r], exact, f"worked example algo={algo} rank={r}")


def test_signed_zero_ties_on_gpu(dev, comms):
    pz, nz = np.float32(0.0), np.float32(-0.0)
    p2 = [np.full(8, pz, np.float32), np.full(8, nz, np.float32)]
    want_ring = np.array([pz] * 4 + [nz] * 4)
    want_tree = np.array([nz] * 4 + [pz] * 4)
    for op in (ar.AR_MIN, ar.AR_MAX):
        for algo, want in ((ar.AR_ALGO_RING, want_ring), (ar.AR_ALGO_LL, want_ring),
                           (ar.AR_ALGO_TREE, want_tree)):
            got = run_guarded(comms(2), p2, ar.AR_FLOAT32, op, algo, 1.0, dev)
            pins.assert_bitwise(got[0], want, f"signed zero op={op} algo={algo}")


def test_in_place_and_aliasing(dev, comms):
    rng = np.random.default_rng(5)
    for P, algo in ((8, ar.AR_ALGO_RING), (8, ar.AR_ALGO_TREE), (8, ar.AR_ALGO_LL),
                    (13, ar.AR_ALGO_RING), (13, ar.AR_ALGO_TREE), (13, ar.AR_ALGO_LL)):
        count = 5000
        sends = pins.random_inputs(rng, P, count, ar.AR_FLOAT32)
        want = oracle.allreduce(sends, ar.AR_FLOAT32, ar.AR_SUM, ORACLE_ALGO[algo])
        bufs = [to_device(s, ar.AR_FLOAT32, dev) for s in sends]
        ar.ar_allreduce(comms(P), bufs, bufs, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        for r in range(P):
            pins.assert_bitwise(to_host(bufs[r]), want[r], f"in place P={P} algo={algo}")
        # one input buffer shared by two ranks (exact aliasing is allowed)
        shared = to_device(sends[0], ar.AR_FLOAT32, dev)
        srcs = [shared, shared] + [to_device(s, ar.AR_FLOAT32, dev) for s in sends[2:]]
        dsts = [torch.empty(count, device=dev) for _ in range(P)]
        ar.ar_allreduce(comms(P), srcs, dsts, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
        torch.cuda.synchronize()
        want2 = oracle.allreduce([sends[0], sends[0]] + sends[2:], ar.AR_FLOAT32, ar.AR_SUM,
                                 ORACLE_ALGO[algo])
        pins.assert_bitwise(to_host(dsts[P - 1]), want2[0], f"aliased inputs P={P} algo={algo}")


def test_argument_errors(dev, comms):
    comm = comms(4)
    x = [torch.zeros(1024, device=dev) for _ in range(4)]
    y = [torch.zeros(1024, device=dev) for _ in range(4)]

    def status(sends, recvs, count=1024, dtype=ar.AR_FLOAT32, op=ar.AR_SUM, algo=ar.AR_ALGO_RING,
               scale=1.0):
        try:
            ar.ar_allreduce(comm, sends, recvs, count, dtype, op, algo, scale)
        except ar.ArError as e:
            return e.status
        return ar.AR_SUCCESS

    base = torch.zeros(2048, device=dev)
    assert status([base[1:1025]] + x[1:], y) == ar.AR_ERR_INVALID_ARG            # misaligned
    assert status(x, [x[0][4:]] + y[1:], count=1000) == ar.AR_ERR_INVALID_ARG    # partial overlap
    assert status(x, y, scale=0.5, dtype=ar.AR_INT32) == ar.AR_ERR_UNSUPPORTED
    assert status(x, y, scale=0.5, op=ar.AR_MAX) == ar.AR_ERR_UNSUPPORTED
    big = [torch.zeros(1 << 15, device=dev) for _ in range(4)]
    big2 = [torch.zeros(1 << 15, device=dev) for _ in range(4)]
    assert status(big, big2, count=1 << 15, algo=ar.AR_ALGO_LL) == ar.AR_ERR_UNSUPPORTED
    assert status(x, y, dtype=7) == ar.AR_ERR_INVALID_ARG
    assert status(x, y, algo=9) == ar.AR_ERR_INVALID_ARG
    # count 0 is a no-op that leaves the outputs alone
    y[0].fill_(7.0)
    assert status(x, y, count=0) == ar.AR_SUCCESS
    torch.cuda.synchronize()
    assert bool((y[0] == 7.0).all())
    # auto selection: LL up to 64 KiB per rank, ring above
    assert ar.ar_select_algo(comm, 16384, ar.AR_FLOAT32) == ar.AR_ALGO_LL
    assert ar.ar_select_algo(comm, 16385, ar.AR_FLOAT32) == ar.AR_ALGO_RING
    assert ar.ar_select_algo(comm, 32768, ar.AR_BFLOAT16) == ar.AR_ALGO_LL
    assert ar.ar_select_algo(comm, 16385, ar.AR_FLOAT32, ar.AR_ALGO_TREE) == ar.AR_ALGO_TREE
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS


def test_non_default_stream(dev, comms):
    rng = np.random.default_rng(9)
    sends = pins.random_inputs(rng, 8, 100000, ar.AR_FLOAT32)
    want = oracle.allreduce(sends, ar.AR_FLOAT32, ar.AR_SUM, oracle.RING, 0.125)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.empty_like(a) for a in xs]
        ar.ar_allreduce(comms(8), xs, ys, 100000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
    s.synchronize()
    pins.assert_bitwise(to_host(ys[5]), want[5], "non-default stream")


def test_ll_bounded_wait_reports_timeout_and_recovers(dev):
    """The only device-side wait (LL flags) ends at its limit with a status.

    The test hook skips the staging phase, so no flag ever carries the
    call's epoch; each waiting thread gives up after the spin limit, records
    AR_ERR_TIMEOUT and exits.  The context stays usable: the next call on the
    same communicator is correct.
    """
    comm = ar.ar_init(8)
    try:
        rng = np.random.default_rng(21)
        sends = pins.random_inputs(rng, 8, 2000, ar.AR_FLOAT32)
        xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
        ys = [torch.zeros_like(a) for a in xs]
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 2000)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 1)
        ar.ar_allreduce(comm, xs, ys, 2000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_ERR_TIMEOUT
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS          # reading clears it
        ar.ar_set_option(comm, ar.AR_OPT_LL_SKIP_PRODUCER, 0)
        ar.ar_set_option(comm, ar.AR_OPT_LL_SPIN_LIMIT, 1 << 22)
        ar.ar_allreduce(comm, xs, ys, 2000, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL, 1.0)
        torch.cuda.synchronize()
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
        want = oracle.allreduce(sends, ar.AR_FLOAT32, ar.AR_SUM, oracle.LL)
        pins.assert_bitwise(to_host(ys[3]), want[3], "LL after a timed-out call")
    finally:
        ar.ar_destroy(comm)


def test_ll_many_calls_epochs(dev, comms):
    """Back-to-back LL calls reuse the staging area via fresh epochs."""
    rng = np.random.default_rng(31)
    comm = comms(8)
    for i in range(50):
        count = int(rng.integers(1, 16385))
        sends = pins.random_inputs(rng, 8, count, ar.AR_FLOAT32)
        got = run_guarded(comm, sends, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_LL, 1.0, dev)
        want = oracle.allreduce(sends, ar.AR_FLOAT32, ar.AR_SUM, oracle.LL)
        pins.assert_bitwise(got[i % 8], want[i % 8], f"LL call {i} count={count}")


# ------------------------------------------------------------- full sizes

def full_call(comm, sends, dtype, op, algo, scale):
    recvs = [torch.empty_like(s) for s in sends]
    ar.ar_allreduce(comm, sends, recvs, sends[0].numel(), dtype, op, algo, scale)
    torch.cuda.synchronize()
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    return recvs


def test_p4_4096_fp32_ring_full(dev, comms):
    """P=4, 4096 fp32 uniform[-1,1] from seed 0, ring, no scale: every element."""
    sends = device_inputs("uniform", 0, 4, 4096, dev)
    recvs = full_call(comms(4), sends, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 1.0)
    want = oracle.allreduce([to_host(s) for s in sends], ar.AR_FLOAT32, oracle.SUM, oracle.RING)
    for r in range(4):
        pins.assert_bitwise(to_host(recvs[r]), want[r], f"rank {r}")


def test_p8_64MiB_fp32_ring_ddp_mean(dev, comms):
    """P=8, 16,777,216 fp32 N(0, 1e-3) per rank, ring, fused scale 1/8:
    every element against the oracle."""
    count, sigma = 16 * 1024 * 1024, 1e-3
    sends = device_inputs("normal", 0, 8, count, dev, sigma)
    recvs = full_call(comms(8), sends, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
    host = host_inputs(sends, "normal", 0, sigma)
    want = oracle_full(host, ar.AR_FLOAT32, oracle.SUM, oracle.RING, 0.125)
    assert_equal_every_element(recvs[0], want, "P=8 64 MiB fp32 ring rank 0")
    assert all_ranks_identical(recvs)
    exact = torch.zeros(count, dtype=torch.float64, device=dev)
    mag = torch.zeros_like(exact)
    for s in sends:
        exact += s.double()
        mag += s.double().abs()
    err = (recvs[0].double() - 0.125 * exact).abs()
    bound = 0.125 * 7 * 2.0 ** -24 * mag * (1 + 1e-6) + 2.0 ** -24 * recvs[0].double().abs()
    assert bool((err <= bound).all())


def test_p8_256MiB_bf16_tree(dev, comms):
    """P=8, 134,217,728 bf16 N(0, 1e-2) per rank, double-binary-tree order:
    every element against the oracle (the contract allows 1 bf16 ulp; the
    kernel performs the oracle's operations in its order, so 0 is required)."""
    count, sigma = 128 * 1024 * 1024, 1e-2
    sends = device_inputs("normal_bf16", 0, 8, count, dev, sigma)
    recvs = full_call(comms(8), sends, ar.AR_BFLOAT16, ar.AR_SUM, ar.AR_ALGO_TREE, 1.0)
    host = host_inputs(sends, "normal_bf16", 0, sigma)
    want = oracle_full(host, ar.AR_BFLOAT16, oracle.SUM, oracle.TREE)
    assert_equal_every_element(recvs[0], want, "P=8 256 MiB bf16 tree rank 0")
    assert all_ranks_identical(recvs)


def test_size_sweep_auto_and_forced(dev, comms):
    """P=8 fp32 uniform[-1,1]: 8 B .. 1 GiB per rank (x2), AUTO and each forced
    algorithm, every element of every point against the oracle."""
    comm = comms(8)
    top = 1 << 28                                     # 1 GiB of fp32 per rank
    sends_full = device_inputs("uniform", 0, 8, top, dev)
    recvs_full = [torch.empty_like(s) for s in sends_full]
    host_full = host_inputs(sends_full, "uniform", 0)
    count = 2
    while count <= top:
        sends = [s[:count] for s in sends_full]
        recvs = [r[:count] for r in recvs_full]
        host = [h[:count] for h in host_full]
        want = {oracle.RING: oracle_full(host, ar.AR_FLOAT32, oracle.SUM, oracle.RING),
                oracle.TREE: oracle_full(host, ar.AR_FLOAT32, oracle.SUM, oracle.TREE)}
        algos = [ar.AR_ALGO_AUTO, ar.AR_ALGO_RING, ar.AR_ALGO_TREE]
        if count * 4 <= 65536:
            algos.append(ar.AR_ALGO_LL)
        for algo in algos:
            recvs[0].fill_(float("nan"))
            ar.ar_allreduce(comm, sends, recvs, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0)
            torch.cuda.synchronize()
            assert ar.ar_get_status(comm) == ar.AR_SUCCESS
            eff = ar.ar_select_algo(comm, count, ar.AR_FLOAT32, algo)
            o = oracle.TREE if eff == ar.AR_ALGO_TREE else oracle.RING
            assert_equal_every_element(recvs[0], want[o], f"sweep count={count} algo={algo}")
            assert all_ranks_identical(recvs)
        count *= 2


def test_ddp_buckets_25MiB(dev, comms):
    """1,207,959,552 fp32 gradients N(0, 1e-3) in 25 MiB buckets, scale 1/8.

    All 185 buckets (the last holds the 2,097,152-element remainder), each
    its own all-reduce call, every element against the oracle.
    """
    total, bucket, sigma = 1_207_959_552, 6_553_600, 1e-3
    nb = -(-total // bucket)
    assert nb == 185
    comm = comms(8)
    for b in range(nb):
        start = b * bucket
        n = min(bucket, total - start)
        sends = device_inputs("normal", 5, 8, n, dev, sigma, start=start)
        recvs = full_call(comm, sends, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)
        host = host_inputs(sends, "normal", 5, sigma, start=start, n_check=32)
        want = oracle_full(host, ar.AR_FLOAT32, oracle.SUM, oracle.RING, 0.125)
        assert_equal_every_element(recvs[0], want, f"bucket {b} rank 0")
        assert all_ranks_identical(recvs)


def test_p72_int32_sum_max_min(dev, comms):
    """P=72 int32 uniform[-2^20, 2^20], 4,194,304 per rank, sum / max / min,
    ring and tree: every element against the oracle in each order, and ring
    == tree == the exact result."""
    P, count = 72, 4 * 1024 * 1024
    comm = comms(P)
    sends = device_inputs("int", 0, P, count, dev)
    host = host_inputs(sends, "int", 0)
    exact_sum = torch.zeros(count, dtype=torch.int64, device=dev)
    exact_min = sends[0].clone()
    exact_max = sends[0].clone()
    for s in sends:
        exact_sum += s.long()
        torch.minimum(exact_min, s, out=exact_min)
        torch.maximum(exact_max, s, out=exact_max)
    exact = {ar.AR_SUM: exact_sum.to(torch.int32), ar.AR_MIN: exact_min, ar.AR_MAX: exact_max}
    for op in OPS:
        outs = {}
        for algo, oalgo in ((ar.AR_ALGO_RING, oracle.RING), (ar.AR_ALGO_TREE, oracle.TREE)):
            recvs = full_call(comm, sends, ar.AR_INT32, op, algo, 1.0)
            want = oracle_full(host, ar.AR_INT32, op, oalgo)
            assert_equal_every_element(recvs[0], want, f"P=72 int32 op={op} algo={algo} rank 0")
            assert all_ranks_identical(recvs)
            outs[algo] = recvs[0]
        assert torch.equal(outs[ar.AR_ALGO_RING], outs[ar.AR_ALGO_TREE])
        assert torch.equal(outs[ar.AR_ALGO_RING], exact[op])


def test_bucket_loop_captured_in_a_cuda_graph(dev, comms):
    """A DDP-style bucket loop recorded once into a CUDA graph and replayed.

    Ring, tree, AUTO (LL for the small bucket) and a forced LL128 call replay
    correctly on new data written into the same buffers: the LL protocols
    take their epoch from device memory, so replays never reuse one.
    """
    comm = comms(8)
    sizes = [1 << 20, 3 * (1 << 18) + 5, 1000, 40000]   # two large buckets and two small ones
    algos = [ar.AR_ALGO_RING, ar.AR_ALGO_TREE, ar.AR_ALGO_AUTO, ar.AR_ALGO_LL128]
    assert ar.ar_select_algo(comm, 1000, ar.AR_FLOAT32, ar.AR_ALGO_AUTO) == ar.AR_ALGO_LL
    sends = [[torch.empty(n, device=dev) for _ in range(8)] for n in sizes]
    recvs = [[torch.empty(n, device=dev) for _ in range(8)] for n in sizes]

    def run_all():
        for b, n in enumerate(sizes):
            ar.ar_allreduce(comm, sends[b], recvs[b], n, ar.AR_FLOAT32, ar.AR_SUM, algos[b], 0.125)

    run_all()                                            # warm-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run_all()
    rng = np.random.default_rng(41)
    for replay in range(3):
        host = [pins.random_inputs(rng, 8, n, ar.AR_FLOAT32) for n in sizes]
        for b in range(len(sizes)):
            for r in range(8):
                sends[b][r].copy_(torch.from_numpy(host[b][r]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for b, n in enumerate(sizes):
            oalgo = oracle.TREE if algos[b] == ar.AR_ALGO_TREE else oracle.RING
            want = oracle.allreduce(host[b], ar.AR_FLOAT32, oracle.SUM, oalgo, 0.125)
            for r in (0, 7):
                pins.assert_bitwise(to_host(recvs[b][r]), want[r], f"replay {replay} bucket {b} rank {r}")
    assert ar.ar_get_status(comm) == ar.AR_SUCCESS
