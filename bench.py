#!/usr/bin/env python3
"""Throughput of the emulated all-reduce on GB300.

One step = one all-reduce call over the workload (P emulated ranks' buffers
resident in HBM).  Default workload: P = 8 ranks x 16,777,216 fp32 (64 MiB per
rank) of N(0, 1e-3) gradients from seed 0, sum in ring order with the fused
1/8 DDP-mean scale.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  value = algbw (bytes per rank / time, summed over the N
replicas); busbw = algbw * 2(P-1)/P; roofline.frac = (2 * P * count * size / t)
/ measured HBM copy bandwidth.  With N > 1 (torchrun) every rank runs an
independent replica on its own GPU (the emulated all-reduce never talks
between GPUs); timing takes the max over ranks.  --impl reference times the
CPU oracle on host cores on a bounded slice of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "allreduce algbw/busbw GB/s (P emulated ranks, 1 GB300) and % of HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
_CSRC = "allreduce_reduction_emulated_gb300/csrc/"
_STATIC = [_CSRC + "ar_device.cuh", _CSRC + "ar_static.cuh"]
_GENERIC = [_CSRC + "ar_device.cuh", _CSRC + "ar_generic.cuh", _CSRC + "ar_generic.cu"]
_GENERIC_WIDE = [_CSRC + "ar_device.cuh", _CSRC + "ar_generic.cuh", _CSRC + "ar_generic_wide.cu"]
# per workload: (ncu summary under profiles/, kernel sources it was taken on,
#                launches of the profiled case per launch of this workload)
PROFILES = {
    "p8_64MiB_fp32_ring_ddp_mean": ("static_ring_p8_64MiB_fp32.ncu.txt", _STATIC + [_CSRC + "ar_static_f32.cu"], 1.0),
    "p8_64MiB_bf16_tree": ("static_tree_p8_64MiB_bf16.ncu.txt", _STATIC + [_CSRC + "ar_static_bf16.cu"], 1.0),
    "p8_256MiB_bf16_tree": ("static_tree_p8_64MiB_bf16.ncu.txt", _STATIC + [_CSRC + "ar_static_bf16.cu"], 4.0),
    "p72_4MiB_int32_sum_ring": ("pipelined_ring_p72_4MiB_int32.ncu.txt", _GENERIC, 1.0),
    "p72_16MiB_int32_sum_ring": ("pipelined_ring_p72_4MiB_int32.ncu.txt", _GENERIC, 4.0),
    "p72_4MiB_int32_max_tree": ("pipelined_tree_p72_4MiB_int32.ncu.txt", _GENERIC, 1.0),
    "p72_16MiB_int32_max_tree": ("pipelined_tree_p72_4MiB_int32.ncu.txt", _GENERIC, 4.0),
    "p8_4KiB_fp32_ll": ("ll_p8_4KiB_fp32.ncu.txt", [_CSRC + "ar_device.cuh", _CSRC + "ar_ll_epoch.cuh", _CSRC + "ar_ll.cu"], 1.0),
    "p8_64KiB_fp32_ll": ("ll_p8_64KiB_fp32.ncu.txt", [_CSRC + "ar_device.cuh", _CSRC + "ar_ll_epoch.cuh", _CSRC + "ar_ll.cu"], 1.0),
    "p8_4KiB_fp32_ring": ("static_ring_p8_4KiB_fp32.ncu.txt", _STATIC + [_CSRC + "ar_static_f32.cu"], 1.0),
    "p8_64KiB_fp32_ring": ("static_ring_p8_64KiB_fp32.ncu.txt", _STATIC + [_CSRC + "ar_static_f32.cu"], 1.0),
    "p72_4MiB_fp32_sum_hier": ("pipelined_hier_p72_4MiB_fp32.ncu.txt", _GENERIC, 1.0),
    "p72_4MiB_int32_sum_hier": ("pipelined_hier_p72_4MiB_int32.ncu.txt", _GENERIC, 1.0),
    "p72_16MiB_int32_sum_hier": ("pipelined_hier_p72_4MiB_int32.ncu.txt", _GENERIC, 4.0),
    "p72_16MiB_fp32_sum_hier": ("pipelined_hier_p72_4MiB_fp32.ncu.txt", _GENERIC, 4.0),
    "p8_512KiB_fp32_ll128": ("ll128_p8_512KiB_fp32.ncu.txt", [_CSRC + "ar_device.cuh", _CSRC + "ar_ll_epoch.cuh", _CSRC + "ar_ll128.cu"], 1.0),
    "p8_rs_8MiB_shards_fp32": ("static_reduce_scatter_p8_8MiB_fp32.ncu.txt", _STATIC + [_CSRC + "ar_static_f32.cu"], 1.0),
    "p72_rs_256KiB_shards_fp32": ("pipelined_reduce_scatter_p72_256KiB_fp32.ncu.txt", _GENERIC, 1.0),
    "p72_16MiB_int32_sum_ring_64sm": ("wide_pipelined_ring_p72_16MiB_int32_64sm.ncu.txt", _GENERIC_WIDE, 1.0),
    "p8_64MiB_fp32_ring_ddp_mean_64sm": ("wide_ring_p8_64MiB_fp32_64sm.ncu.txt", _STATIC + [_CSRC + "ar_wide_f32.cu"], 1.0),
    "p8_rs_8MiB_shards_fp32_64sm": ("wide_reduce_scatter_p8_8MiB_fp32_64sm.ncu.txt", _STATIC + [_CSRC + "ar_wide_f32.cu"], 1.0),
    "p8_ag_8MiB_shards_fp32_64sm": ("tma_all_gather_p8_8MiB_fp32_64sm.ncu.txt", _STATIC + [_CSRC + "ar_tma.cuh", _CSRC + "ar_tma_gather.cu"], 1.0),
    "p8_ag_8MiB_shards_fp32": ("all_gather_p8_8MiB_fp32.ncu.txt", [_CSRC + "ar_device.cuh", _CSRC + "ar_collectives.cu"], 1.0),
}

HEADLINE = "p8_64MiB_fp32_ring_ddp_mean"

WORKLOADS = {
    # the headline: 8 ranks x 64 MiB fp32, ring order, DDP mean
    "p8_64MiB_fp32_ring_ddp_mean": dict(P=8, count=16 * 1024 * 1024, kind="normal", sigma=1e-3,
                                        dtype="f32", op="sum", algo="ring", scale=0.125, seed=0),
    # other sizes for exploration (parity cases, not the headline line)
    "p8_256MiB_bf16_tree": dict(P=8, count=128 * 1024 * 1024, kind="normal_bf16", sigma=1e-2,
                                dtype="bf16", op="sum", algo="tree", scale=1.0, seed=0),
    "p72_16MiB_int32_sum_ring": dict(P=72, count=4 * 1024 * 1024, kind="int", sigma=1.0,
                                     dtype="i32", op="sum", algo="ring", scale=1.0, seed=0),
    "p72_16MiB_int32_max_tree": dict(P=72, count=4 * 1024 * 1024, kind="int", sigma=1.0,
                                     dtype="i32", op="max", algo="tree", scale=1.0, seed=0),
    "p72_16MiB_int32_sum_hier": dict(P=72, count=4 * 1024 * 1024, kind="int", sigma=1.0,
                                     dtype="i32", op="sum", algo="hier", scale=1.0, seed=0, group=8),
    "p72_16MiB_fp32_sum_hier": dict(P=72, count=4 * 1024 * 1024, kind="normal", sigma=1e-3,
                                    dtype="f32", op="sum", algo="hier", scale=1.0 / 72, seed=3, group=8),
    # smaller cases of the same kernels, sized for profiler captures (inputs still exceed L2)
    "p8_64MiB_bf16_tree": dict(P=8, count=32 * 1024 * 1024, kind="normal_bf16", sigma=1e-2,
                               dtype="bf16", op="sum", algo="tree", scale=1.0, seed=0),
    "p72_4MiB_int32_sum_ring": dict(P=72, count=1024 * 1024, kind="int", sigma=1.0,
                                    dtype="i32", op="sum", algo="ring", scale=1.0, seed=0),
    "p72_4MiB_int32_max_tree": dict(P=72, count=1024 * 1024, kind="int", sigma=1.0,
                                    dtype="i32", op="max", algo="tree", scale=1.0, seed=0),
    "p72_4MiB_int32_sum_hier": dict(P=72, count=1024 * 1024, kind="int", sigma=1.0,
                                    dtype="i32", op="sum", algo="hier", scale=1.0, seed=0, group=8),
    "p72_4MiB_fp32_sum_hier": dict(P=72, count=1024 * 1024, kind="normal", sigma=1e-3,
                                   dtype="f32", op="sum", algo="hier", scale=1.0 / 72, seed=3, group=8),
    "p8_512KiB_fp32_ll128": dict(P=8, count=128 * 1024, kind="uniform", sigma=1.0, dtype="f32", op="sum",
                                 algo="ll128", scale=1.0, seed=0),
    "p8_4KiB_fp32_ll": dict(P=8, count=1024, kind="uniform", sigma=1.0, dtype="f32", op="sum",
                            algo="ll", scale=1.0, seed=0),
    # small messages for per-launch kernel times (ncu's gpu__time_duration resolves what the
    # ~2 us launch cadence of back-to-back small kernels hides): LL against the ring
    "p8_4KiB_fp32_ring": dict(P=8, count=1024, kind="uniform", sigma=1.0, dtype="f32", op="sum",
                              algo="ring", scale=1.0, seed=0),
    "p8_64KiB_fp32_ll": dict(P=8, count=16384, kind="uniform", sigma=1.0, dtype="f32", op="sum",
                             algo="ll", scale=1.0, seed=0),
    "p8_64KiB_fp32_ring": dict(P=8, count=16384, kind="uniform", sigma=1.0, dtype="f32", op="sum",
                               algo="ring", scale=1.0, seed=0),
    # the ring's two halves as standalone collectives: count = elements per shard
    "p8_rs_8MiB_shards_fp32": dict(P=8, count=2 * 1024 * 1024, kind="normal", sigma=1e-3, dtype="f32",
                                   op="sum", algo="ring", scale=0.125, seed=0, coll="reduce_scatter"),
    "p8_ag_8MiB_shards_fp32": dict(P=8, count=2 * 1024 * 1024, kind="normal", sigma=1e-3, dtype="f32",
                                   op="sum", algo="ring", scale=1.0, seed=0, coll="all_gather"),
    # the headline on 64 of the 152 SMs (AR_OPT_MAX_BLOCKS): the wide kernel (1024-thread
    # blocks, one per SM), for an all-reduce that shares the GPU with computation
    "p8_64MiB_fp32_ring_ddp_mean_64sm": dict(P=8, count=16 * 1024 * 1024, kind="normal", sigma=1e-3,
                                             dtype="f32", op="sum", algo="ring", scale=0.125, seed=0,
                                             max_blocks=64),
    # the reduce-scatter on 64 SMs (the wide kernel): gradient shards beside computation
    "p8_rs_8MiB_shards_fp32_64sm": dict(P=8, count=2 * 1024 * 1024, kind="normal", sigma=1e-3, dtype="f32",
                                        op="sum", algo="ring", scale=0.125, seed=0, coll="reduce_scatter",
                                        max_blocks=64),
    # the all-gather on 64 SMs (TMA pipeline)
    "p8_ag_8MiB_shards_fp32_64sm": dict(P=8, count=2 * 1024 * 1024, kind="normal", sigma=1e-3, dtype="f32",
                                        op="sum", algo="ring", scale=1.0, seed=0, coll="all_gather",
                                        max_blocks=64),
    # config 5b's ring on 64 of the 152 SMs: the pipelined kernel in 768-thread blocks
    "p72_16MiB_int32_sum_ring_64sm": dict(P=72, count=4 * 1024 * 1024, kind="int", sigma=1.0,
                                          dtype="i32", op="sum", algo="ring", scale=1.0, seed=0, max_blocks=64),
    # reduce-scatter above the rank-specialised limit: 72 shards of 256 KiB (18 MiB per rank)
    "p72_rs_256KiB_shards_fp32": dict(P=72, count=64 * 1024, kind="normal", sigma=1e-3, dtype="f32",
                                      op="sum", algo="ring", scale=1.0 / 72, seed=0, coll="reduce_scatter"),
}


def sizes_of(w: dict):
    """(elements per input buffer, per output buffer, nccl-tests size in bytes,
    busbw factor, HBM bytes per call) of a workload."""
    P, n, es = w["P"], w["count"], ESIZE[w["dtype"]]
    coll = w.get("coll", "allreduce")
    if coll == "reduce_scatter":
        return P * n, n, P * n * es, (P - 1) / P, P * P * n * es + P * n * es
    if coll == "all_gather":
        return n, P * n, P * n * es, (P - 1) / P, P * n * es + P * P * n * es
    return n, n, n * es, 2 * (P - 1) / P, 2 * P * n * es
ESIZE = {"f32": 4, "bf16": 2, "i32": 4}

# DDP-style bucketed run: 24 layers of [2048x8192], [8192x2048], [2048x6144],
# [2048x2048] fp32 gradients (1,207,959,552 per rank), flattened and cut into
# 25 MiB buckets (184 x 6,553,600 + 1 x 2,097,152), one all-reduce per bucket.
DDP_PARAMS = 24 * (2048 * 8192 + 8192 * 2048 + 2048 * 6144 + 2048 * 2048)
DDP_BUCKET = 25 * 1024 * 1024 // 4


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 6000; 200 with --ddp-buckets, 30 with --ddp-overlap)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ddp-buckets", action="store_true",
                    help="DDP-style run: P=8 x 1,207,959,552 fp32 gradients in 185 x 25 MiB buckets per step")
    ap.add_argument("--ddp-overlap", action="store_true",
                    help="DDP backward (synthetic per-rank weight-gradient GEMMs) overlapped with the "
                         "bucketed all-reduce: compute, comm, serial and overlapped step times")
    ap.add_argument("--tokens", type=int, default=512,
                    help="tokens per rank for --ddp-overlap's gradient GEMMs")
    ap.add_argument("--comm-blocks", type=lambda v: v if v == "auto" else int(v), default=0,
                    help="--ddp-overlap: cap the all-reduce kernels at this many thread blocks (0 = none); "
                         "below the SM count they run the TMA pipeline, one block per SM (48 measured best; "
                         "'auto' = that share of this GPU's SMs)")
    ap.add_argument("--gemm-carveout", type=int, default=0,
                    help="--ddp-overlap: leave this many SMs out of the gradient GEMMs (PyTorch's "
                         "experimental cuBLAS SM carve-out; 0 = none)")
    ap.add_argument("--grad-dtype", choices=("fp32", "bf16"), default="fp32",
                    help="--ddp-overlap: gradient dtype (bf16: bf16 GEMMs and bf16 bucket all-reduces)")
    ap.add_argument("--comm-priority", action="store_true",
                    help="--ddp-overlap: run the communication stream at the highest priority")
    ap.add_argument("--no-more-configs", action="store_true",
                    help="time only the chosen workload (skip the other large configs after it)")
    ap.add_argument("--sweep", action="store_true",
                    help="message-size sweep (P=8 fp32, 8 B .. 1 GiB per rank) with an alpha-beta fit")
    return ap.parse_args()


def config_of(name: str, w: dict, n: int) -> dict:
    return {"workload": name, "collective": w.get("coll", "allreduce"), "P": w["P"],
            "count_per_rank": w["count"], "dtype": w["dtype"],
            "op": w["op"], "algo": w["algo"], "scale": w["scale"],
            "values": f"{w['kind']} sigma={w['sigma']} seed={w['seed']}",
            "l2": "inputs larger than L2 (no flush)" if 2 * w["P"] * w["count"] * ESIZE[w["dtype"]] > 2 * 129e6
                  else "L2 not flushed (small message: latency-bound)",
            "parallelism": f"replicas x{n}",
            **({"max_blocks": w["max_blocks"]} if "max_blocks" in w else {})}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu            # nvidia-smi --id: the GPU's UUID ("GPU-...") or its index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [f.strip() for f in line.split(",")]))

    def wait_fresh_row(self, limit_s: float = 0.25):
        """Returns right after nvidia-smi has printed a row (or after limit_s).
        A timed region started then ends long before nvidia-smi's next query
        (every 50 ms), so the in-process NVML reads are not held up behind it."""
        if self.proc is None:
            return
        n = len(self.rows)
        t_end = time.time() + limit_s
        while len(self.rows) == n and time.time() < t_end:
            time.sleep(0.0002)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        rows = inside or [r for _, r in self.rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "samples_in_timed_region": len(inside)}


def gpu_uuid(torch, dev) -> str | None:
    """The device's NVML / nvidia-smi UUID ("GPU-..."), which names the same GPU
    whatever CUDA_VISIBLE_DEVICES does to the indices; None if unknown."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


class NvmlClocks:
    """Query-only NVML reads (SM clock, its maximum, the active clock-event
    reasons) taken by the host while the timed region runs on the GPU: the
    timed region of a short run is far shorter than nvidia-smi's sampling
    period.  Changes no setting.  Every method is a no-op if NVML is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str | None, index: int):
        import ctypes

        self.c = ctypes
        self.h = None
        self.samples = []           # (inside the timed region, sm_mhz, reasons bitmask)
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = (L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) if uuid
                  else L.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)))
            if rc != 0:
                return
            self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                L.nvmlDeviceGetCurrentClocksThrottleReasons
            self.L, self.h = L, h
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
        except (OSError, AttributeError):
            self.h = None

    def sample(self, inside: bool):
        if self.h is None:
            return
        c = self.c
        mhz, bits = c.c_uint(), c.c_ulonglong()
        if self.L.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) != 0:   # NVML_CLOCK_SM
            return
        if self.reasons_fn(self.h, c.byref(bits)) != 0:
            bits.value = 0
        self.samples.append((inside, float(mhz.value), int(bits.value)))

    def poll(self, start_ev, end_ev, limit_s: float = 600.0):
        """Samples until end_ev has completed; a sample counts as inside the
        timed region when start_ev had completed before it was taken."""
        t_end = time.time() + limit_s
        while not end_ev.query() and time.time() < t_end:
            inside = start_ev.query()
            self.sample(inside)
            if self.h is None:
                time.sleep(0.001)

    def summary(self) -> dict:
        inside = [x for x in self.samples if x[0]]
        names = sorted({n for _, _, b in inside for bit, n in self.REASONS.items() if b & bit})
        return {"samples_in_timed_region": len(inside),
                "sm_mhz": statistics.median([m for _, m, _ in inside]) if inside else None,
                "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": names}


def merged_clocks(smi: dict, nvml: dict) -> dict:
    """nvidia-smi's samples around the run and NVML's inside the timed region:
    the timed region's own figures win where it has any."""
    out = dict(smi)
    out["nvidia_smi_samples_in_timed_region"] = smi.get("samples_in_timed_region", 0)
    if nvml.get("samples_in_timed_region"):
        out["sm_mhz"] = nvml["sm_mhz"]
        out["sm_max_mhz"] = nvml["sm_max_mhz"] or smi.get("sm_max_mhz")
        out["reasons"] = sorted(set(smi.get("reasons", [])) | set(nvml["reasons"]))
        out["samples_in_timed_region"] = smi.get("samples_in_timed_region", 0) + nvml["samples_in_timed_region"]
        out["nvml_samples_in_timed_region"] = nvml["samples_in_timed_region"]
        out["sm_mhz_source"] = "NVML reads while the timed region ran"
    return out


# The timed region starts with a spin kernel queued ahead of the start event:
# it holds the GPU while the host enqueues the K steps, so the region times the
# steps themselves -- not the host's issue of the first call (~23 us through
# ctypes) or the GPU waking from the idle pause before it (a first step of
# 190-280 us instead of 160 us was measured without it).
HIDE_CYCLES = 4_000_000   # ~2 ms at 2 GHz


def timed_steps(torch, step, steps: int, stream, nvml: "NvmlClocks | None" = None,
                range_name: str = "timed", clocks: "ClockSampler | None" = None) -> float:
    """ms for `steps` calls of step(), timed by CUDA events on `stream`."""
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.wait_fresh_row()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HIDE_CYCLES)
    torch.cuda.nvtx.range_push(range_name)   # lets a profiler select exactly this region
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.nvtx.range_pop()
    if nvml is not None:
        nvml.poll(ev0, ev1)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


# ---------------------------------------------------------------- roofline

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources) -> str:
    h = hashlib.sha256()
    for p in sources:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this workload's
    kernel (scaled by units processed when a smaller case was captured), or
    None when there is none or the kernel sources changed since the capture."""
    if workload not in PROFILES:
        return None
    name, sources, scale = PROFILES[workload]
    try:
        fields = {}
        with open(os.path.join(ROOT, "profiles", name)) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != kernel_source_hash(sources):
            return None
        return float(fields["dram_bytes_per_launch"]) * scale
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------ aggregation

def sm_time_bound_ms(compute_ms: float, comm_ms: float, comm_sms: int, sms: int):
    """Lower bound on an overlapped step when both sides are SM-bound: the
    GEMMs need compute_ms on all `sms` SMs, the all-reduces comm_ms on
    `comm_sms` of them, and the step can be no shorter than their SM-time
    spread over the whole GPU (nor than either side alone).  None when the
    all-reduces are not capped (they then take whole SMs from the GEMMs in
    turns, and the split is not known)."""
    if not comm_sms or comm_sms >= sms:
        return None
    return max((compute_ms * sms + comm_ms * comm_sms) / sms, compute_ms, comm_ms)


PG_TIMEOUT_S = 600  # rank 0 builds the library while the other ranks wait at the first barrier


def init_replicas(world: int, rank: int, timeout_s: float = PG_TIMEOUT_S):
    """The gloo process group of N independent replicas (it carries only the
    host-side barriers and the max over ranks of the timings).  A rank that
    exits makes its peers' next barrier fail at once; one that never arrives
    makes it fail after timeout_s, instead of blocking them."""
    import datetime

    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def max_over_ranks(x: float, dist=None) -> float:
    """The slowest rank's time (every rank gets it)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_replica_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every replica's bytes over the slowest replica's time."""
    return world * bytes_per_replica_step / (ms_per_step * 1e-3) / 1e9


# -------------------------------------------------------------- CPU oracle

HOST_CORES = os.cpu_count() or 1


class OneCore:
    """Pins the calling thread to one host core while the (single-threaded)
    oracle is timed, then restores its affinity."""

    def __enter__(self):
        self.saved = None
        if hasattr(os, "sched_getaffinity"):
            try:
                self.saved = os.sched_getaffinity(0)
                os.sched_setaffinity(0, {max(self.saved)})
            except OSError:
                self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


def oracle_throughput(w: dict, host_sends, seconds: float):
    """The oracle as it stands, one host core, over whole-workload passes."""
    import numpy as np

    import oracle

    P, count = w["P"], w["count"]
    coll = w.get("coll", "allreduce")
    dt = {"f32": oracle.F32, "bf16": oracle.BF16, "i32": oracle.I32}[w["dtype"]]
    op = {"sum": oracle.SUM, "min": oracle.MIN, "max": oracle.MAX}[w["op"]]
    algo = {"ring": oracle.RING, "tree": oracle.TREE, "ll": oracle.LL, "ll128": oracle.RING,
            "hier": None}[w["algo"]]
    nccl_bytes = sizes_of(w)[2]
    if coll == "allreduce" and algo is not None:
        recvs = [np.zeros(count, dtype=oracle.NP_DTYPE[dt]) for _ in range(P)]
        oracle.allreduce(host_sends, dt, op, algo, w["scale"], 0, min(count, 65536), recvs)  # warm
    with OneCore():
        done, t0 = 0, time.perf_counter()
        while True:
            if coll == "reduce_scatter":
                oracle.reduce_scatter(host_sends, dt, op, w["scale"])
            elif coll == "all_gather":
                oracle.all_gather(host_sends, dt)
            elif algo is None:
                oracle.allreduce_hier(host_sends, w["group"], dt, op, w["scale"])
            else:
                oracle.allreduce(host_sends, dt, op, algo, w["scale"], 0, count, recvs)
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    return done * nccl_bytes / el / 1e9, done, el


def reference_arm(args, w, name):
    """--impl reference: the CPU oracle on a bounded slice of the workload."""
    import numpy as np

    import oracle
    import synthetic

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if w.get("coll", "allreduce") != "allreduce" or w["algo"] == "hier":
        raise SystemExit("--impl reference times the ring / tree / LL all-reduce workloads")
    P, count = w["P"], w["count"]
    dt = {"f32": oracle.F32, "bf16": oracle.BF16, "i32": oracle.I32}[w["dtype"]]
    op = {"sum": oracle.SUM, "min": oracle.MIN, "max": oracle.MAX}[w["op"]]
    algo = {"ring": oracle.RING, "tree": oracle.TREE, "ll": oracle.LL, "ll128": oracle.RING}[w["algo"]]
    # calibrate, then size the per-step slice so that warmup + steps take ~60 s
    probe = min(count, 32768)
    idx = np.arange(probe)
    sends = [np.zeros(count, dtype=oracle.NP_DTYPE[dt]) for _ in range(P)]
    for r in range(P):
        sends[r][:probe] = synthetic.values_np(w["kind"], w["seed"], r, idx, w["sigma"])
    recvs = [np.zeros(count, dtype=oracle.NP_DTYPE[dt]) for _ in range(P)]
    t0 = time.perf_counter()
    oracle.allreduce(sends, dt, op, algo, w["scale"], 0, probe, recvs)
    per_elem = max((time.perf_counter() - t0) / probe, 1e-9)
    budget = 60.0 / max(1, args.steps + args.warmup)
    S = int(min(count, max(1024, budget / per_elem)))
    S = max(1, S // 1024 * 1024) if S >= 1024 else S
    if S > probe:
        idx = np.arange(probe, S)
        for r in range(P):
            sends[r][probe:S] = synthetic.values_np(w["kind"], w["seed"], r, idx, w["sigma"])
    for _ in range(args.warmup):
        oracle.allreduce(sends, dt, op, algo, w["scale"], 0, S, recvs)
    with OneCore():
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.allreduce(sends, dt, op, algo, w["scale"], 0, S, recvs)
        el = time.perf_counter() - t0
    value = S * ESIZE[w["dtype"]] * args.steps / el / 1e9
    sample = (f"elements [0, {S}) of each of the {P} ranks' {count}-element buffers per step "
              f"(ring chunking of the full count), one host core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"],
        "data": "synthetic", "config": config_of(name, w, args.gpus),
        "busbw": value * 2 * (P - 1) / P,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": HOST_CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- our arm

def ours_arm(args, w, name):
    import numpy as np
    import torch

    import __graft_entry__
    import allreduce_reduction_emulated_gb300 as ar
    import synthetic

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = init_replicas(world, rank) if world > 1 else None
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    P, count = w["P"], w["count"]
    esize = ESIZE[w["dtype"]]
    dtype = {"f32": ar.AR_FLOAT32, "bf16": ar.AR_BFLOAT16, "i32": ar.AR_INT32}[w["dtype"]]
    op = ar.OPS[w["op"]]
    algo = ar.ALGOS[w["algo"]]
    coll = w.get("coll", "allreduce")
    n_in, n_out, nccl_bytes, bus_factor, hbm_bytes = sizes_of(w)
    sends = [synthetic.values_torch(w["kind"], w["seed"], r, 0, n_in, dev, w["sigma"]) for r in range(P)]
    recvs = [torch.empty(n_out, dtype=sends[0].dtype, device=dev) for _ in range(P)]
    comm = ar.ar_init(P)
    if "group" in w:
        ar.ar_set_option(comm, ar.AR_OPT_HIER_GROUP, w["group"])
    if "max_blocks" in w:
        ar.ar_set_option(comm, ar.AR_OPT_MAX_BLOCKS, w["max_blocks"])
    stream = torch.cuda.current_stream()

    def call(xs, ys, s):
        if coll == "reduce_scatter":
            ar.ar_reduce_scatter(comm, xs, ys, count, dtype, op, w["scale"], s)
        elif coll == "all_gather":
            ar.ar_all_gather(comm, xs, ys, count, dtype, s)
        else:
            ar.ar_allreduce(comm, xs, ys, count, dtype, op, algo, w["scale"], s)

    def step():
        call(sends, recvs, stream)

    uuid = gpu_uuid(torch, dev)
    clocks = ClockSampler(uuid or local)
    clocks.start()
    nvml = NvmlClocks(uuid, local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ar.ar_get_status(comm) != ar.AR_SUCCESS:
        raise SystemExit("device status error in warm-up")

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ms = timed_steps(torch, step, args.steps, stream, nvml, clocks=clocks)
    t1 = time.time()
    if dist:
        dist.barrier()
    time.sleep(0.2)
    clocks.stop()
    if ar.ar_get_status(comm) != ar.AR_SUCCESS:
        raise SystemExit("device status error in the timed region")
    ms_step = max_over_ranks(ms, dist) / args.steps
    algbw = job_gbs(nccl_bytes, ms_step, world)
    achieved = hbm_bytes / (ms_step * 1e-3) / 1e9           # one kernel per step
    peak, peak_kind = measured_hbm_peak()

    # end to end through the public API with host buffers: every step copies
    # its P inputs from pinned host memory, runs the call and copies all P
    # results back.  Steps are pipelined over two device buffer sets and three
    # streams (H2D of step i+1 and D2H of step i-1 overlap the call of step i).
    host_in = [s.cpu().pin_memory() for s in sends]
    host_out = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in recvs]
    sets = [(sends, recvs), ([torch.empty_like(s) for s in sends], [torch.empty_like(s) for s in recvs])]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nsteps = args.e2e_steps

    def e2e_run(n):
        done_run = [None] * n
        done_out = [None] * n
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        s_run.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            d_in, d_out = sets[i % 2]
            if i >= 2:
                s_in.wait_event(done_run[i - 2])     # step i-2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                for d, h in zip(d_in, host_in):
                    d.copy_(h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(s_in)
            s_run.wait_event(ready)
            if i >= 2:
                s_run.wait_event(done_out[i - 2])    # step i-2's results have left
            call(d_in, d_out, s_run)
            done_run[i] = torch.cuda.Event()
            done_run[i].record(s_run)
            s_out.wait_event(done_run[i])
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out, d_out):
                    h.copy_(d, non_blocking=True)
            done_out[i] = torch.cuda.Event()
            done_out[i].record(s_out)
        end.record(s_out)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    e2e_run(3)
    if dist:
        dist.barrier()
    e2e_ms = max_over_ranks(e2e_run(nsteps) / nsteps, dist)
    if ar.ar_get_status(comm) != ar.AR_SUCCESS:
        raise SystemExit("device status error in the end-to-end run")
    e2e_value = job_gbs(nccl_bytes, e2e_ms, world)

    line = None
    if rank == 0:
        cpu = None
        if world == 1:
            host_np = [h.numpy() if h.dtype != torch.bfloat16 else h.view(torch.int16).numpy().view(np.uint16)
                       for h in host_in]
            gbs, passes, el = oracle_throughput(w, host_np, args.cpu_seconds)
            cpu = {"value": gbs, "unit": UNIT, "cores": 1, "host_cores": HOST_CORES, "kind": "oracle",
                   "sample": f"{passes} full pass(es) over the workload ({P} x {n_in} input elements), "
                             f"{el:.1f} s on one host core"}
        traffic = profiled_traffic(name)
        line = {
            "metric": METRIC, "value": algbw, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
            "config": config_of(name, w, world),
            "busbw": algbw * bus_factor,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": hbm_bytes},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "steps": nsteps, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": P * n_in * esize, "d2h_bytes_per_step": P * n_out * esize,
                    "path": "pinned host -> device copies, ar_allreduce, device -> pinned host copies "
                            "of all P results; pipelined over 2 buffer sets / 3 streams"},
            "gpu_launches": args.steps,
            "clocks": merged_clocks(clocks.summary(t0, t1), nvml.summary()),
            "timing": "CUDA events on the launching stream around the K steps; a ~2 ms spin kernel "
                      "queued ahead of the start event holds the GPU while the host enqueues them",
        }
    ar.ar_destroy(comm)
    if line is not None and world == 1 and name == HEADLINE and not args.no_more_configs:
        del sends, recvs, sets
        torch.cuda.empty_cache()
        line["more_configs"] = more_configs(args, dev, stream, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------- the other large configs

MORE_CONFIGS = ("p8_256MiB_bf16_tree", "p72_16MiB_int32_sum_ring", "p72_16MiB_int32_max_tree",
                "ddp_1p2b_fp32_25MiB_buckets")


def more_configs(args, dev, stream, world: int) -> dict:
    """The other large-message workloads, each timed like the headline (warm-up,
    a spin ahead of the start event, K steps between CUDA events) in this
    process after it: 8 x 256 MiB bf16 in the double-binary-tree order, 72
    ranks x 16 MiB int32 (ring sum, tree max), and the DDP bucket loop (185
    calls of 25 MiB per step, replayed from one CUDA graph; at most 100 timed
    steps).  Only after the headline workload at N = 1."""
    import torch

    import allreduce_reduction_emulated_gb300 as ar
    import synthetic

    peak, _ = measured_hbm_peak()
    out = {}
    for name in MORE_CONFIGS:
        if name.startswith("ddp_"):
            P, total, B, sigma, seed = 8, DDP_PARAMS, DDP_BUCKET, 1e-3, 5
            buckets = [(b, min(B, total - b)) for b in range(0, total, B)]
            sends = []
            for r in range(P):
                flat = torch.empty(total, dtype=torch.float32, device=dev)
                for start, n in buckets:
                    flat[start:start + n] = synthetic.values_torch("normal", seed, r, start, n, dev, sigma)
                sends.append(flat)
            recvs = [torch.empty_like(x) for x in sends]
            comm = ar.ar_init(P)
            views = [([x[a:a + n] for x in sends], [y[a:a + n] for y in recvs], n) for a, n in buckets]
            side = torch.cuda.Stream()

            def calls(s=None):
                for sv, rv, n in views:
                    ar.ar_allreduce(comm, sv, rv, n, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125, s)

            calls(stream)                                   # warm-up outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    calls(side)
            step = g.replay
            per_rank, esize, launches = total * 4, 4, len(buckets)
            cfg = {"P": P, "params_per_rank": total, "buckets": len(buckets), "bucket_elems": B,
                   "dtype": "f32", "op": "sum", "algo": "ring", "scale": 0.125,
                   "values": f"normal sigma={sigma} seed={seed}",
                   "launch": f"{len(buckets)} calls per step replayed from one CUDA graph"}
        else:
            w = WORKLOADS[name]
            P, count = w["P"], w["count"]
            dt = {"f32": ar.AR_FLOAT32, "bf16": ar.AR_BFLOAT16, "i32": ar.AR_INT32}[w["dtype"]]
            sends = [synthetic.values_torch(w["kind"], w["seed"], r, 0, count, dev, w["sigma"]) for r in range(P)]
            recvs = [torch.empty_like(x) for x in sends]
            comm = ar.ar_init(P)

            def step(w=w, sends=sends, recvs=recvs, comm=comm, dt=dt, count=count):
                ar.ar_allreduce(comm, sends, recvs, count, dt, ar.OPS[w["op"]], ar.ALGOS[w["algo"]],
                                w["scale"], stream)

            per_rank, esize, launches = count * ESIZE[w["dtype"]], ESIZE[w["dtype"]], 1
            cfg = {k: w[k] for k in ("P", "dtype", "op", "algo", "scale")}
            cfg["count_per_rank"] = count
            cfg["values"] = f"{w['kind']} sigma={w['sigma']} seed={w['seed']}"
        k = min(args.steps, 100) if name.startswith("ddp_") else args.steps
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        ms = timed_steps(torch, step, k, stream, range_name=f"more_configs {name}") / k
        if ar.ar_get_status(comm) != ar.AR_SUCCESS:
            raise SystemExit(f"device status error in {name}")
        achieved = 2 * P * per_rank / (ms * 1e-3) / 1e9
        algbw = job_gbs(per_rank, ms, world)
        out[name] = {**cfg, "steps": k, "warmup": args.warmup, "ms_per_step": ms,
                     "algbw": algbw, "busbw": algbw * 2 * (P - 1) / P,
                     "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                  "frac": achieved / peak, "traffic": profiled_traffic(name)},
                     "gpu_launches": launches * k}
        ar.ar_destroy(comm)
        del sends, recvs, step
        if name.startswith("ddp_"):
            del g, views
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ sweep

def fit_alpha_beta(points):
    """Least-squares t = alpha + beta * n over (n bytes, t seconds) points."""
    n = len(points)
    sx = sum(p[0] for p in points)
    sy = sum(p[1] for p in points)
    sxx = sum(p[0] * p[0] for p in points)
    sxy = sum(p[0] * p[1] for p in points)
    beta = (n * sxy - sx * sy) / (n * sxx - sx * sx)
    alpha = (sy - beta * sx) / n
    return alpha, beta


SPIN_CYCLES = 200_000   # ~0.1 ms of GPU spin ahead of a timed small call


def sweep(args):
    """nccl-tests style sweep ("NCCL and NVSHMEM ...", exercise 1: 8 B .. 1 GiB,
    factor 2) for AUTO and each forced algorithm, with t = alpha + beta * n."""
    import torch

    import __graft_entry__
    import allreduce_reduction_emulated_gb300 as ar
    import synthetic

    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    P, top = 8, 1 << 28
    sends_full = [synthetic.values_torch("uniform", 0, r, 0, top, dev) for r in range(P)]
    recvs_full = [torch.empty_like(s) for s in sends_full]
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    comm = ar.ar_init(P)
    stream = torch.cuda.current_stream()
    names = {ar.AR_ALGO_AUTO: "auto", ar.AR_ALGO_RING: "ring", ar.AR_ALGO_TREE: "tree",
             ar.AR_ALGO_LL: "ll", ar.AR_ALGO_LL128: "ll128"}
    rows = []
    count = 2
    while count <= top:
        sends = [x[:count] for x in sends_full]
        recvs = [x[:count] for x in recvs_full]
        nbytes = count * 4
        small = 2 * P * nbytes < 2 * 129e6           # working set could sit in L2: flush it
        algos = [ar.AR_ALGO_AUTO, ar.AR_ALGO_RING, ar.AR_ALGO_TREE]
        if nbytes <= 65536:
            algos.append(ar.AR_ALGO_LL)
        if nbytes <= 1 << 20:
            algos.append(ar.AR_ALGO_LL128)
        for algo in algos:
            def call():
                ar.ar_allreduce(comm, sends, recvs, count, ar.AR_FLOAT32, ar.AR_SUM, algo, 1.0, stream)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            t_issue = None
            if small:
                # "us": the call's GPU time -- a spin kernel keeps the GPU busy
                # while the host enqueues the start event and the call, so the
                # host's issue time is not inside the events; "us_with_issue":
                # the events bracket the host's issue of the call as well
                times, issued = [], []
                for _ in range(100):
                    for hide, out in ((True, times), (False, issued)):
                        flush.zero_()
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        if hide:
                            torch.cuda._sleep(SPIN_CYCLES)
                        a.record(stream)
                        call()
                        b.record(stream)
                        torch.cuda.synchronize()
                        out.append(a.elapsed_time(b))
                t = statistics.median(times) * 1e-3
                t_mean = statistics.fmean(times) * 1e-3
                t_issue = statistics.median(issued) * 1e-3
            else:
                iters = max(5, min(200, int(2e9 / (2 * P * nbytes))))
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(iters):
                    call()
                b.record(stream)
                torch.cuda.synchronize()
                t = a.elapsed_time(b) * 1e-3 / iters
                t_mean = t
            if ar.ar_get_status(comm) != ar.AR_SUCCESS:
                raise SystemExit("device status error in the sweep")
            rows.append({"bytes_per_rank": nbytes, "algo": names[algo],
                         "resolved": names[ar.ar_select_algo(comm, count, ar.AR_FLOAT32, algo)],
                         "us": t * 1e6, "us_mean": t_mean * 1e6,
                         "us_with_issue": None if t_issue is None else t_issue * 1e6,
                         "algbw": nbytes / t / 1e9,
                         "busbw": nbytes / t / 1e9 * 2 * (P - 1) / P,
                         "hbm_gbs": 2 * P * nbytes / t / 1e9, "l2_flushed": small})
        count *= 2
    table = ar.ar_tune(comm)
    ar.ar_destroy(comm)
    fits = {}
    # fitted on the per-point means: the event timer steps by about 2 us, so
    # single calls (and their medians) are quantized, their means are not
    for name in ("ring", "tree", "ll", "ll128", "auto"):
        pts = [(r["bytes_per_rank"], r["us_mean"] * 1e-6) for r in rows if r["algo"] == name]
        if len(pts) >= 2:
            alpha, beta = fit_alpha_beta(pts)
            fits[name] = {"alpha_us": alpha * 1e6, "inv_beta_gbs": (1 / beta / 1e9) if beta > 0 else None,
                          "points": len(pts)}
    print(json.dumps({"sweep": "P=8 fp32 uniform[-1,1] sum, bytes per rank 8 B .. 1 GiB (x2)",
                      "unit": "us / GB/s", "rows": rows, "fit": fits,
                      "ar_tune_table": {str(8 << b): names[a] for b, a in enumerate(table)}}), flush=True)


# ------------------------------------------------------------ DDP buckets

def ddp_buckets(args):
    """One step = the 185 bucket all-reduces of the 1.2B-parameter gradients
    (sum, scale 1/8, ring), issued eagerly and replayed from a CUDA graph."""
    import numpy as np
    import torch

    import __graft_entry__
    import allreduce_reduction_emulated_gb300 as ar
    import oracle
    import synthetic

    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    P, total, B, sigma, seed = 8, DDP_PARAMS, DDP_BUCKET, 1e-3, 5
    buckets = [(b, min(B, total - b)) for b in range(0, total, B)]
    sends = []
    for r in range(P):
        flat = torch.empty(total, dtype=torch.float32, device=dev)
        for start, n in buckets:
            flat[start:start + n] = synthetic.values_torch("normal", seed, r, start, n, dev, sigma)
        sends.append(flat)
    recvs = [torch.empty_like(x) for x in sends]
    comm = ar.ar_init(P)
    stream = torch.cuda.current_stream()
    views = [([x[s:s + n] for x in sends], [y[s:s + n] for y in recvs], n) for s, n in buckets]

    def step():
        for sv, rv, n in views:
            ar.ar_allreduce(comm, sv, rv, n, ar.AR_FLOAT32, ar.AR_SUM, ar.AR_ALGO_RING, 0.125)

    uuid = gpu_uuid(torch, dev)
    clocks = ClockSampler(uuid or 0)
    clocks.start()
    nvml = NvmlClocks(uuid, 0)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    eager_ms = timed_steps(torch, step, args.steps, stream) / args.steps
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    t0 = time.time()
    graph_ms = timed_steps(torch, g.replay, args.steps, stream, nvml, clocks=clocks) / args.steps
    t1 = time.time()
    time.sleep(0.2)
    clocks.stop()
    if ar.ar_get_status(comm) != ar.AR_SUCCESS:
        raise SystemExit("device status error")
    ar.ar_destroy(comm)
    per_rank = total * 4
    peak, peak_kind = measured_hbm_peak()
    achieved = 2 * P * per_rank / (graph_ms * 1e-3) / 1e9
    # the oracle on a bounded sample: the first buckets, each its own all-reduce
    nb_cpu, done, t_cpu = 0, 0, 0.0
    for start, n in buckets:
        host = [x[start:start + n].cpu().numpy() for x in sends]
        with OneCore():
            c0 = time.perf_counter()
            oracle.allreduce(host, oracle.F32, oracle.SUM, oracle.RING, 0.125)
            t_cpu += time.perf_counter() - c0
        nb_cpu += 1
        done += n
        if t_cpu >= args.cpu_seconds:
            break
    line = {
        "metric": METRIC, "value": per_rank / (graph_ms * 1e-3) / 1e9, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": graph_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "ddp_1p2b_fp32_25MiB_buckets", "P": P, "params_per_rank": total,
                   "buckets": len(buckets), "bucket_elems": B, "op": "sum", "algo": "ring",
                   "scale": 0.125, "values": f"normal sigma={sigma} seed={seed}",
                   "launch": "185 calls per step replayed from one CUDA graph",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas x1"},
        "busbw": per_rank / (graph_ms * 1e-3) / 1e9 * 2 * (P - 1) / P,
        "eager_ms_per_step": eager_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "cpu_baseline": {"value": done * 4 / t_cpu / 1e9, "unit": UNIT, "cores": 1, "host_cores": HOST_CORES,
                         "kind": "oracle",
                         "sample": f"the first {nb_cpu} bucket all-reduces ({done} elements per rank)"},
        "e2e": None, "gpu_launches": len(buckets) * args.steps,
        "clocks": merged_clocks(clocks.summary(t0, t1), nvml.summary()),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ DDP overlap

DDP_LAYER_SHAPES = [(2048, 8192), (8192, 2048), (2048, 6144), (2048, 2048)]


def ddp_overlap(args):
    """The 1.2B-parameter DDP step on 8 emulated ranks: backward = per-rank
    weight-gradient GEMMs dW = X^T dY (TF32 into fp32 gradients, or bf16 with
    --grad-dtype bf16; tokens x shapes below) written straight into each rank's
    flat gradient buffer in reverse layer order; communication = 25 MiB bucket
    all-reduces (ring, scale 1/8; 185 buckets of fp32, 93 of bf16).  Four
    variants, each one CUDA graph: compute only, comm only, compute then comm,
    and overlapped (each bucket's all-reduce enqueued on a second stream as
    soon as its gradients are written)."""
    import torch

    import __graft_entry__
    import allreduce_reduction_emulated_gb300 as ar
    from allreduce_reduction_emulated_gb300.buckets import BucketReducer

    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    torch.backends.cuda.matmul.allow_tf32 = True
    gdt = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    esize = 2 if args.grad_dtype == "bf16" else 4
    P, T, total, B = 8, args.tokens, DDP_PARAMS, 25 * 1024 * 1024 // esize
    grads = [torch.zeros(total, dtype=gdt, device=dev) for _ in range(P)]
    outs = [torch.empty_like(g) for g in grads]
    order = [(layer, i) for layer in reversed(range(24)) for i in range(4)]
    views, off = [], 0
    for layer, i in order:
        m, n = DDP_LAYER_SHAPES[i]
        views.append(([g[off:off + m * n].view(m, n) for g in grads], m, n, off + m * n))
        off += m * n
    assert off == total
    gen = torch.Generator(device=dev).manual_seed(11)
    acts = {d: [(torch.randn(T, d, device=dev, generator=gen) * 0.01).to(gdt) for _ in range(P)]
            for d in (2048, 6144, 8192)}
    comm = ar.ar_init(P)
    compute = torch.cuda.Stream()
    high = torch.cuda.Stream.priority_range()[1] if args.comm_priority else 0
    reducer = BucketReducer(comm, grads, B, scale=0.125, out=outs, stream=torch.cuda.Stream(priority=high),
                            max_blocks=args.comm_blocks)
    comm_blocks = reducer.max_blocks
    torch.cuda.synchronize()                    # inputs made on the default stream
    if args.gemm_carveout:
        if not hasattr(torch._C, "_set_sm_carveout_experimental"):
            raise SystemExit("--gemm-carveout: this PyTorch has no SM carve-out")
        torch._C._set_sm_carveout_experimental(args.gemm_carveout)

    def backward(overlap):
        for vs, m, n, end in views:
            for r in range(P):
                torch.mm(acts[m][r].t(), acts[n][r], out=vs[r])
            if overlap:
                ev = torch.cuda.Event()
                ev.record(compute)
                reducer.ready(end, ev)

    def variant(kind):
        reducer.reset()
        if kind in ("compute", "serial", "overlap"):
            backward(kind == "overlap")
        if kind in ("comm", "serial"):
            ev = torch.cuda.Event()
            ev.record(compute)
            reducer.ready(total, ev)
        if kind != "compute":
            compute.wait_event(reducer.finish())

    graphs = {}
    for kind in ("compute", "comm", "serial", "overlap"):
        with torch.cuda.stream(compute):
            variant(kind)                       # warm-up outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(compute):
            with torch.cuda.graph(g, stream=compute):
                variant(kind)
        graphs[kind] = g
    times = {}
    for kind, g in graphs.items():
        for _ in range(max(args.warmup, 1)):
            g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        times[kind] = a.elapsed_time(b) / args.steps
    # where the overlapped step's time goes: one eager run with events at the
    # step start, after the last GEMM and after the last bucket's all-reduce;
    # a 100 ms spin holds the GPU while the host enqueues the step, so the
    # host's issue rate does not set the pace
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(compute):
        reducer.reset()
        torch.cuda._sleep(int(2e8))
        marks[0].record(compute)
        backward(True)
        marks[1].record(compute)
        compute.wait_event(reducer.finish())
        marks[2].record(compute)
    torch.cuda.synchronize()
    gemm_end, step_end = marks[0].elapsed_time(marks[1]), marks[0].elapsed_time(marks[2])
    if ar.ar_get_status(comm) != ar.AR_SUCCESS:
        raise SystemExit("device status error")
    ar.ar_destroy(comm)
    flops = P * 2.0 * total * T
    model = max(times["compute"], times["comm"])
    print(json.dumps({
        "ddp_overlap": f"P=8 x 1,207,959,552 {args.grad_dtype} gradients, "
                       f"{(total + B - 1) // B} x 25 MiB buckets, ring, scale 1/8",
        "grad_dtype": args.grad_dtype,
        "tokens_per_rank": T, "steps": args.steps, "unit": "ms",
        "comm_blocks": comm_blocks, "comm_priority": bool(args.comm_priority),
        "gemm_carveout": args.gemm_carveout,
        "compute_ms": times["compute"], "comm_ms": times["comm"], "serial_ms": times["serial"],
        "overlap_ms": times["overlap"], "exposed_comm_ms": times["overlap"] - times["compute"],
        "max_compute_comm_ms": model, "tail_ms": times["overlap"] - model,
        "sm_time_bound_ms": sm_time_bound_ms(times["compute"], times["comm"], comm_blocks or 0,
                                             torch.cuda.get_device_properties(dev).multi_processor_count),
        "hidden_fraction_of_shorter": (times["serial"] - times["overlap"]) / min(times["compute"], times["comm"]),
        "gemm_tflops": flops / (times["compute"] * 1e-3) / 1e12,
        "eager_overlap": {"last_gemm_end_ms": gemm_end, "step_end_ms": step_end,
                          "after_last_gemm_ms": step_end - gemm_end,
                          "buckets_after_last_gemm_at_comm_rate":
                              (step_end - gemm_end) / (times["comm"] / len(reducer.starts))},
        "comm_hbm_gbs": 2 * P * total * esize / (times["comm"] * 1e-3) / 1e9,
    }), flush=True)


def main():
    args = parse_args()
    if args.steps is None:
        args.steps = 30 if args.ddp_overlap else 200 if args.ddp_buckets else 6000
    if args.ddp_overlap:
        ddp_overlap(args)
        return
    if args.ddp_buckets:
        ddp_buckets(args)
        return
    if args.sweep:
        sweep(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, w, args.workload)
    else:
        ours_arm(args, w, args.workload)


if __name__ == "__main__":
    main()
