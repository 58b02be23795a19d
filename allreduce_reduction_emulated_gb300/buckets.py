"""Bucketed gradient all-reduce overlapped with the backward pass.

DDP's pattern ("NCCL, NIXL, and Distributed GPU Communication", the DDP
paragraph under "All-reduce" and the "Performance engineer checklist"): as
soon as a bucket's gradients are ready, its all-reduce is enqueued on a
separate communication stream, so later layers' backward compute overlaps
earlier buckets' communication; total time ~ max(compute, comm) + a tail.

Here every emulated rank's gradients live in one flat buffer (parameters in
the order the backward produces them), cut into fixed-size buckets.  The
producer reports how far the flat gradient is complete (an element offset
and an event recorded after the writes); every bucket wholly below that
offset is all-reduced on the communication stream after waiting on the
event.  Plumbing only: the reduction is ar_allreduce.
"""
from __future__ import annotations

import torch

from . import (AR_ALGO_RING, AR_CAPPED_TMA, AR_OPT_CAPPED_KERNEL, AR_OPT_MAX_BLOCKS, AR_SUM, ar_allreduce,
               ar_set_option, dtype_of)

# Share of the SMs that max_blocks="auto" gives the all-reduces.  Measured on
# GB300 (152 SMs) with the bucket all-reduces of a 1.2B-parameter backward
# (8 emulated ranks, 25 MiB buckets) beside the gradient GEMMs: 48 SMs gave
# the shortest step with fp32 and with bf16 gradients (64 within 1% with bf16;
# 32, 40, 80 and 96 slower), and the uncapped grid was no faster than running
# the two serially.
AUTO_SM_FRACTION = 48 / 152


def auto_max_blocks(device=None) -> int:
    """The block cap max_blocks="auto" uses on `device` (default: current)."""
    if device is None:
        device = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return max(1, round(sms * AUTO_SM_FRACTION))


class BucketReducer:
    """All-reduces fixed-size buckets of P flat gradient buffers as they fill.

    grads     P contiguous CUDA tensors of the same length (one per rank)
    bucket    elements per bucket (the last one may be shorter)
    comm      an ar_init communicator for P ranks
    out       optional P result tensors (default: reduce in place)
    max_blocks    if given, AR_OPT_MAX_BLOCKS is set to it on the communicator
                  before each bucket's all-reduce: the all-reduces then run on a
                  few SMs beside the backward pass; "auto" takes
                  AUTO_SM_FRACTION of the gradients' GPU's SMs
    capped_kernel AR_OPT_CAPPED_KERNEL set with max_blocks (default: the TMA
                  pipeline -- beside the gradient GEMMs it gave 25.1 ms per step
                  on 48 SMs against 27.7 ms for the wide load/store kernel,
                  which is the faster of the two when nothing else runs)
    """

    def __init__(self, comm: int, grads, bucket: int, scale: float = 1.0, algo: int = AR_ALGO_RING,
                 out=None, stream: torch.cuda.Stream | None = None, max_blocks: int | str | None = None,
                 capped_kernel: int = AR_CAPPED_TMA):
        self.comm = comm
        self.grads = list(grads)
        self.out = list(out) if out is not None else self.grads
        self.total = self.grads[0].numel()
        self.bucket = bucket
        self.scale = scale
        self.algo = algo
        self.dtype = dtype_of(self.grads[0])
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.starts = list(range(0, self.total, bucket))
        self.next_bucket = 0
        if max_blocks == "auto":
            max_blocks = auto_max_blocks(self.grads[0].device)
        elif max_blocks is not None and not isinstance(max_blocks, int):
            raise ValueError(f"max_blocks must be an int, 'auto' or None, not {max_blocks!r}")
        self.max_blocks = max_blocks
        self.capped_kernel = capped_kernel

    def reset(self):
        self.next_bucket = 0

    def ready(self, upto: int, event: torch.cuda.Event) -> int:
        """Elements [0, upto) are written once `event` completes: enqueue every
        bucket that now lies wholly below upto.  Returns how many it enqueued."""
        n = 0
        while self.next_bucket < len(self.starts):
            s = self.starts[self.next_bucket]
            e = min(s + self.bucket, self.total)
            if e > upto:
                break
            if n == 0:
                self.stream.wait_event(event)
            if self.max_blocks is not None:
                ar_set_option(self.comm, AR_OPT_MAX_BLOCKS, self.max_blocks)
                ar_set_option(self.comm, AR_OPT_CAPPED_KERNEL, self.capped_kernel)
            ar_allreduce(self.comm, [g[s:e] for g in self.grads], [o[s:e] for o in self.out], e - s,
                         self.dtype, AR_SUM, self.algo, self.scale, self.stream)
            self.next_bucket += 1
            n += 1
        return n

    def finish(self) -> torch.cuda.Event:
        """An event on the communication stream after the last bucket."""
        if self.next_bucket != len(self.starts):
            raise RuntimeError("BucketReducer.finish: not every bucket was reported ready")
        ev = torch.cuda.Event()
        ev.record(self.stream)
        return ev
