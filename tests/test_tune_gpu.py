"""ar_tune: AUTO picks the algorithm measured fastest per size on this device
("NCCL and NVSHMEM ...", exercise 6: find the ring / tree crossover by
forcing each; "Demystifying NVSHMEM": selection is a measured rule table)."""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu

VALID = {ar.AR_ALGO_RING, ar.AR_ALGO_TREE, ar.AR_ALGO_LL, ar.AR_ALGO_LL128}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def test_tune_drives_auto_and_results_stay_exact(dev):
    comm = ar.ar_init(8)
    try:
        with pytest.raises(ar.ArError):                       # nothing measured yet
            ar.ar_set_option(comm, ar.AR_OPT_AUTO_TUNED, 1)
        table = ar.ar_tune(comm)
        assert len(table) == ar.AR_TUNE_BUCKETS and set(table) <= VALID
        # LL is only ever chosen within its limit
        for b, a in enumerate(table):
            if a == ar.AR_ALGO_LL:
                assert (8 << b) <= 65536
        rng = np.random.default_rng(12)
        for nbytes in (8, 100, 4096, 65536, 70000, 1 << 20, 5 << 20):
            count = nbytes // 4
            b = max(0, int(np.ceil(np.log2(max(nbytes, 8)))) - 3)
            chosen = ar.ar_select_algo(comm, count, ar.AR_FLOAT32, ar.AR_ALGO_AUTO)
            assert chosen == table[min(b, ar.AR_TUNE_BUCKETS - 1)]
            sends = pins.random_inputs(rng, 8, count, ar.AR_FLOAT32)
            xs = [to_device(a, ar.AR_FLOAT32, dev) for a in sends]
            ys = [torch.empty_like(x) for x in xs]
            ar.ar_allreduce(comm, xs, ys, count, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_AUTO, 1.0)
            torch.cuda.synchronize()
            order = oracle.TREE if chosen == ar.AR_ALGO_TREE else oracle.RING
            want = oracle.allreduce(sends, ar.AR_FLOAT32, oracle.SUM, order)
            pins.assert_bitwise(to_host(ys[5]), want[5], f"AUTO after tuning, {nbytes} B, algo {chosen}")
        # back to the fixed rule, and to the table again
        ar.ar_set_option(comm, ar.AR_OPT_AUTO_TUNED, 0)
        assert ar.ar_select_algo(comm, 4096, ar.AR_FLOAT32) == ar.AR_ALGO_LL
        ar.ar_set_option(comm, ar.AR_OPT_AUTO_TUNED, 1)
        assert ar.ar_select_algo(comm, 1024, ar.AR_FLOAT32) == table[9]
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)
