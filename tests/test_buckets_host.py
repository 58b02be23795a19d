"""BucketReducer's host logic on CPU (no GPU): which buckets a progress report
releases, in what order, after which event, and with which block cap.

DDP ("NCCL, NIXL, and Distributed GPU Communication", the DDP paragraph and
the overlap checklist): a bucket is all-reduced as soon as all of its
gradients are written; the library call itself is replaced by a recorder.
"""
import pytest
import torch

import allreduce_reduction_emulated_gb300 as ar
from allreduce_reduction_emulated_gb300 import buckets as B


class FakeStream:
    def __init__(self):
        self.waited = []

    def wait_event(self, ev):
        self.waited.append(ev)


@pytest.fixture
def recorder(monkeypatch):
    log = []
    monkeypatch.setattr(B, "ar_allreduce",
                        lambda comm, s, r, n, dt, op, algo, scale, stream:
                        log.append(("allreduce", s[0].data_ptr(), r[0].data_ptr(), n, scale)))
    monkeypatch.setattr(B, "ar_set_option", lambda comm, opt, val: log.append(("option", opt, val)))
    return log


def make(total=1000, bucket=300, **kw):
    grads = [torch.arange(total, dtype=torch.float32) for _ in range(2)]
    stream = FakeStream()
    red = B.BucketReducer(comm=1, grads=grads, bucket=bucket, scale=0.5, stream=stream, **kw)
    return red, grads, stream


def test_buckets_released_in_order_once_wholly_written(recorder):
    red, grads, stream = make()
    assert red.starts == [0, 300, 600, 900]                 # the last bucket is 100 long
    assert red.ready(299, "e0") == 0 and recorder == []     # bucket 0 not complete yet
    assert red.ready(650, "e1") == 2                        # buckets [0, 300) and [300, 600)
    assert stream.waited == ["e1"]                          # one wait, before the first call
    es = grads[0].element_size()
    assert [(c[1] - grads[0].data_ptr()) // es for c in recorder] == [0, 300]
    assert [c[3] for c in recorder] == [300, 300] and all(c[4] == 0.5 for c in recorder)
    assert red.ready(1000, "e2") == 2                       # [600, 900) and the short [900, 1000)
    assert [c[3] for c in recorder] == [300, 300, 300, 100]
    assert stream.waited == ["e1", "e2"]
    assert red.ready(1000, "e3") == 0                       # nothing left


def test_finish_requires_every_bucket(recorder):
    red, _, _ = make()
    red.ready(600, "e")
    with pytest.raises(RuntimeError):
        red.finish()
    red.reset()
    assert red.next_bucket == 0


def test_block_cap_set_before_each_bucket(recorder):
    """The cap and the capped kernel (the TMA pipeline by default: measured
    faster beside the gradient GEMMs) are set before every bucket."""
    red, _, _ = make(max_blocks=48)
    red.ready(1000, "e")
    kinds = [c[0] for c in recorder]
    assert kinds == ["option", "option", "allreduce"] * 4
    opts = [c for c in recorder if c[0] == "option"]
    assert opts[0::2] == [("option", ar.AR_OPT_MAX_BLOCKS, 48)] * 4
    assert opts[1::2] == [("option", ar.AR_OPT_CAPPED_KERNEL, ar.AR_CAPPED_TMA)] * 4
    recorder.clear()
    red, _, _ = make(max_blocks=48, capped_kernel=ar.AR_CAPPED_WIDE)
    red.ready(1000, "e")
    assert [c for c in recorder if c[0] == "option"][1] == ("option", ar.AR_OPT_CAPPED_KERNEL, ar.AR_CAPPED_WIDE)


def test_no_cap_leaves_the_option_alone(recorder):
    red, _, _ = make()
    red.ready(1000, "e")
    assert all(c[0] == "allreduce" for c in recorder)


def test_out_buffers_receive_the_results(recorder):
    grads = [torch.zeros(10) for _ in range(2)]
    outs = [torch.zeros(10) for _ in range(2)]
    red = B.BucketReducer(comm=1, grads=grads, bucket=4, out=outs, stream=FakeStream())
    red.ready(10, "e")
    assert [c[2] - outs[0].data_ptr() for c in recorder] == [0, 16, 32]


def test_auto_cap_is_the_measured_share_of_the_sms(recorder, monkeypatch):
    class Props:
        multi_processor_count = 152

    monkeypatch.setattr(B.torch.cuda, "get_device_properties", lambda device: Props)
    red, _, _ = make(max_blocks="auto")
    assert red.max_blocks == 48
    red.ready(1000, "e")
    assert all(c[2] == 48 for c in recorder if c[0] == "option" and c[1] == ar.AR_OPT_MAX_BLOCKS)
    Props.multi_processor_count = 132
    assert B.auto_max_blocks("cuda:0") == 42
    Props.multi_processor_count = 1
    assert B.auto_max_blocks("cuda:0") == 1


def test_bad_cap_rejected():
    with pytest.raises(ValueError):
        make(max_blocks="most")
