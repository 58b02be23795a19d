"""Bucketed all-reduce overlapped with a synthetic backward pass.

The overlapped schedule (each bucket's all-reduce on a second stream as soon
as an event says its gradients are written) must give exactly the result of
the serial schedule, and each bucket must equal the oracle's all-reduce of
the gradients the backward produced -- so the events order every bucket
after its writes ("NCCL, NIXL, ...", DDP overlap).
"""
import numpy as np
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
import oracle
import pins
from allreduce_reduction_emulated_gb300.buckets import BucketReducer
from gpu_util import to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("max_blocks,capped", [(None, None), (16, None), ("auto", None), (16, ar.AR_CAPPED_WIDE)],
                         ids=["uncapped", "16", "auto", "16-wide"])
def test_overlapped_buckets_match_serial_and_oracle(dev, max_blocks, capped, gdt):
    """max_blocks=16 or "auto" (48 of 152 SMs): the bucket all-reduces run on a
    few SMs (the TMA pipeline, BucketReducer's default beside computation, or
    the wide load/store kernel).
    bf16: bf16 GEMMs write bf16 gradients, reduced with fp32 accumulation."""
    P, T, bucket = 4, 96, 300_000
    shapes = [(512, 1024), (1024, 512), (512, 768)] * 2          # 6 "parameters", backward order
    total = sum(m * n for m, n in shapes)
    gen = torch.Generator(device=dev).manual_seed(3)
    acts = {d: [torch.randn(T, d, device=dev, generator=gen).to(gdt) for _ in range(P)] for d in (512, 768, 1024)}
    comm = ar.ar_init(P)
    results = {}
    try:
        for overlap in (False, True):
            grads = [torch.zeros(total, dtype=gdt, device=dev) for _ in range(P)]
            outs = [torch.full((total,), float("nan"), dtype=gdt, device=dev) for _ in range(P)]
            compute = torch.cuda.Stream()
            kw = {} if capped is None else {"capped_kernel": capped}
            red = BucketReducer(comm, grads, bucket, scale=0.25, out=outs, max_blocks=max_blocks, **kw)
            torch.cuda.synchronize()              # buffers initialised on the default stream
            with torch.cuda.stream(compute):
                off = 0
                for m, n in shapes:
                    for r in range(P):
                        torch.mm(acts[m][r].t(), acts[n][r], out=grads[r][off:off + m * n].view(m, n))
                    off += m * n
                    if overlap:
                        ev = torch.cuda.Event()
                        ev.record(compute)
                        red.ready(off, ev)
                if not overlap:
                    ev = torch.cuda.Event()
                    ev.record(compute)
                    red.ready(total, ev)
                compute.wait_event(red.finish())
            torch.cuda.synchronize()
            results[overlap] = ([to_host(g) for g in grads], [to_host(o) for o in outs])
        assert ar.ar_get_status(comm) == ar.AR_SUCCESS
    finally:
        ar.ar_destroy(comm)
    g_serial, o_serial = results[False]
    g_over, o_over = results[True]
    for r in range(P):
        pins.assert_bitwise(o_over[r], o_serial[r], f"overlapped vs serial rank {r}")
    for s in range(0, total, bucket):
        e = min(s + bucket, total)
        odt = oracle.BF16 if gdt == torch.bfloat16 else oracle.F32
        want = oracle.allreduce([g[s:e] for g in g_over], odt, oracle.SUM, oracle.RING, 0.25)
        pins.assert_bitwise(o_over[P - 1][s:e], want[P - 1], f"bucket at {s}")
