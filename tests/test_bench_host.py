"""bench.py's host logic on CPU: workload byte counts and the ncu summaries.

The roofline's `achieved` divides each workload's algorithmic bytes by the
kernel's time, and `traffic` comes from the committed ncu summary under
profiles/ only while the kernel sources still hash to the captured value.
"""
import os
import re

import pytest

import bench


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_algorithmic_bytes_follow_the_collective(name):
    w = bench.WORKLOADS[name]
    P, n, es = w["P"], w["count"], bench.ESIZE[w["dtype"]]
    n_in, n_out, nccl_bytes, bus, hbm = bench.sizes_of(w)
    coll = w.get("coll", "allreduce")
    if coll == "allreduce":
        # every rank's buffer read once, the result written to every rank
        assert (n_in, n_out) == (n, n)
        assert hbm == P * n * es + P * n * es
        assert nccl_bytes == n * es and bus == pytest.approx(2 * (P - 1) / P)
    elif coll == "reduce_scatter":
        # P inputs of P shards read, one shard written per rank
        assert (n_in, n_out) == (P * n, n)
        assert hbm == P * (P * n) * es + P * n * es
        assert nccl_bytes == P * n * es and bus == pytest.approx((P - 1) / P)
    else:
        # one shard read per rank, P shards written per rank
        assert (n_in, n_out) == (n, P * n)
        assert hbm == P * n * es + P * (P * n) * es
        assert nccl_bytes == P * n * es and bus == pytest.approx((P - 1) / P)


def test_headline_bytes_per_launch():
    w = bench.WORKLOADS["p8_64MiB_fp32_ring_ddp_mean"]
    assert bench.sizes_of(w)[4] == 2 * 8 * 16_777_216 * 4 == 1_073_741_824


def test_ddp_bucket_layout():
    # 24 x {2048x8192, 8192x2048, 2048x6144, 2048x2048} fp32 cut into 25 MiB buckets
    assert bench.DDP_PARAMS == 1_207_959_552
    assert bench.DDP_BUCKET == 6_553_600
    full, rest = divmod(bench.DDP_PARAMS, bench.DDP_BUCKET)
    assert (full, rest) == (184, 2_097_152)


@pytest.mark.parametrize("name", sorted(bench.PROFILES))
def test_profile_summary_is_complete(name):
    fname, sources, scale = bench.PROFILES[name]
    assert name in bench.WORKLOADS
    assert scale > 0
    for s in sources:
        assert os.path.isfile(os.path.join(bench.ROOT, s)), s
    path = os.path.join(bench.ROOT, "profiles", fname)
    assert os.path.isfile(path), fname
    text = open(path).read()
    assert re.search(r"^dram_bytes_per_launch: \d+$", text, re.M)
    assert re.search(r"^source_sha256: [0-9a-f]{16}$", text, re.M)
    # the commands that made it run committed files only, with the clocks left alone
    assert "python bench.py --workload" in text
    for line in text.splitlines():
        if line.strip().startswith("ncu "):
            assert "--clock-control none" in line


def test_every_workload_has_a_summary():
    # each of its own kernel instantiation (a larger workload may scale a
    # smaller capture of the same instantiation by the units it processes)
    assert set(bench.WORKLOADS) <= set(bench.PROFILES)


def test_traffic_only_while_the_sources_match(monkeypatch):
    name = "p72_16MiB_int32_sum_ring"                    # a scaled (4 MiB -> 16 MiB) summary
    fname, sources, scale = bench.PROFILES[name]
    text = open(os.path.join(bench.ROOT, "profiles", fname)).read()
    captured = re.search(r"^source_sha256: ([0-9a-f]{16})$", text, re.M).group(1)
    per_launch = int(re.search(r"^dram_bytes_per_launch: (\d+)$", text, re.M).group(1))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda s: captured)
    assert bench.profiled_traffic(name) == per_launch * scale
    monkeypatch.setattr(bench, "kernel_source_hash", lambda s: "0" * 16)
    assert bench.profiled_traffic(name) is None
    assert bench.profiled_traffic("no_such_workload") is None


def test_every_summary_matches_the_current_kernel_sources():
    """A kernel edited after its ncu capture makes bench.py report no traffic
    for it; this names such a summary, so it is re-captured with the change."""
    stale = [w for w in bench.PROFILES if bench.profiled_traffic(w) is None]
    assert stale == [], f"re-capture the ncu summaries of {stale}"


def test_oracle_timing_runs_on_one_core():
    import os

    if not hasattr(os, "sched_getaffinity"):
        pytest.skip("no affinity control on this platform")
    before = os.sched_getaffinity(0)
    with bench.OneCore():
        assert len(os.sched_getaffinity(0)) == 1
    assert os.sched_getaffinity(0) == before


def test_clock_summary_reads_nvidia_smi_rows():
    """The clocks record of a bench line: the median SM clock inside the timed
    region, the maximum, and every throttle reason seen Active there."""
    c = bench.ClockSampler(0)
    row = lambda sm, hw="Not Active", thermal="Not Active", cap="Not Active": \
        [f.strip() for f in f"0, {sm}, 2070, 900.1, 0x0, {hw}, {thermal}, Not Active, {cap}".split(",")]
    c.rows = [(0.5, row(1200)), (1.0, row(2070)), (1.5, row(2070, cap="Active")), (2.0, row(1965)),
              (2.5, row(2070)), (9.0, row(300, thermal="Active"))]
    s = c.summary(1.0, 2.5)
    assert s["samples_in_timed_region"] == 4 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]              # the thermal sample lies outside the region
    s = c.summary(8.5, 9.5)
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["sm_mhz"] == 300.0
    # no sample inside the region: fall back to every sample; malformed rows are skipped
    c.rows.append((3.0, ["0", "[N/A]"]))
    s = c.summary(100.0, 101.0)
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 7 and s["sm_mhz"] == 2017.5  # median of 6


def test_timed_region_starts_right_after_an_nvidia_smi_row():
    """The timed region waits for nvidia-smi's next row, so the region (a few
    ms) ends before nvidia-smi's following query; without nvidia-smi, or once
    the wait's limit has passed, it starts at once."""
    import threading
    import time

    c = bench.ClockSampler(0)
    c.wait_fresh_row()                                   # no nvidia-smi process: no wait
    c.proc = object()
    t0 = time.time()
    threading.Timer(0.05, lambda: c.rows.append((time.time(), ["0"]))).start()
    c.wait_fresh_row(limit_s=2.0)
    waited = time.time() - t0
    assert len(c.rows) == 1 and 0.04 <= waited < 1.0
    t0 = time.time()
    c.wait_fresh_row(limit_s=0.05)                       # no new row: gives up at the limit
    assert 0.04 <= time.time() - t0 < 1.0


def test_overlap_arguments(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--ddp-overlap", "--comm-blocks", "auto", "--gemm-carveout", "32",
                                     "--grad-dtype", "bf16", "--comm-priority"])
    a = bench.parse_args()
    assert (a.ddp_overlap, a.comm_blocks, a.gemm_carveout, a.grad_dtype, a.comm_priority) == \
        (True, "auto", 32, "bf16", True)
    monkeypatch.setattr("sys.argv", ["bench.py", "--ddp-overlap", "--comm-blocks", "48"])
    a = bench.parse_args()
    assert (a.comm_blocks, a.gemm_carveout, a.grad_dtype) == (48, 0, "fp32")
    monkeypatch.setattr("sys.argv", ["bench.py", "--comm-blocks", "most"])
    with pytest.raises(SystemExit):
        bench.parse_args()


def test_sm_time_bound():
    # 18.4 ms of GEMMs on 152 SMs + 17.0 ms of all-reduce on 48: 23.77 ms
    assert bench.sm_time_bound_ms(18.4, 17.0, 48, 152) == pytest.approx(18.4 + 17.0 * 48 / 152)
    assert bench.sm_time_bound_ms(1.0, 30.0, 8, 152) == 30.0          # never below either side
    assert bench.sm_time_bound_ms(18.4, 11.4, 0, 152) is None          # uncapped: split unknown
    assert bench.sm_time_bound_ms(18.4, 11.4, 152, 152) is None


def test_nvml_samples_inside_the_timed_region_win():
    """Clock samples taken by NVML while the timed region ran replace
    nvidia-smi's when nvidia-smi had none inside it; reasons are the union."""
    n = bench.NvmlClocks.__new__(bench.NvmlClocks)
    n.h, n.max_mhz = None, 2070.0
    n.samples = [(False, 1500.0, 0x1), (True, 2070.0, 0x0), (True, 2055.0, 0x4), (True, 2070.0, 0x0)]
    s = n.summary()
    assert s["samples_in_timed_region"] == 3 and s["sm_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    smi = {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 10, "samples_in_timed_region": 0}
    m = bench.merged_clocks(smi, s)
    assert m["sm_mhz"] == 2070.0 and m["samples_in_timed_region"] == 3
    assert m["nvml_samples_in_timed_region"] == 3 and m["reasons"] == ["sw_power_cap"]
    # no NVML samples: nvidia-smi's figures stand
    empty = {"samples_in_timed_region": 0, "sm_mhz": None, "sm_max_mhz": None, "reasons": []}
    assert bench.merged_clocks(smi, empty)["sm_mhz"] == 1980.0


def test_nvml_polling_is_a_no_op_without_the_library(monkeypatch):
    """Without libnvidia-ml the clock reader records nothing and polling ends
    when the end event completes."""
    import ctypes

    def missing(name, *a, **k):
        raise OSError(name)

    monkeypatch.setattr(ctypes, "CDLL", missing)
    n = bench.NvmlClocks(None, 0)
    assert n.h is None

    class Ev:
        def __init__(self, left):
            self.left = left

        def query(self):
            self.left -= 1
            return self.left <= 0

    n.poll(Ev(1), Ev(3))
    assert n.samples == [] and n.summary()["samples_in_timed_region"] == 0
