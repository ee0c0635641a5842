"""bench.py's host-side helpers that need no GPU: workload parsing and the oracle CPU baselines
of the extra workloads (each timed on a tiny sample here)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_parse_workload_names():
    assert bench.parse_workload("q8_0_4096x4096_m1")[:4] == ("q8_0", 4096, 4096, 1)
    assert bench.parse_workload("blk128_5120x17408_m8")[:4] == ("blk", 5120, 17408, 8)
    assert bench.parse_workload("e4m3_1024x4096_m2")[:4] == ("e4m3", 1024, 4096, 2)


@pytest.mark.parametrize("workload", ["producer_256x8", "silu_1536x4", "repack_e4m3_256x1024",
                                      "repack_blk128_300x512"])
def test_cpu_baseline_other(oracle, workload):
    cb = bench.cpu_baseline_other(workload, 0.05)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "GB/s"
    assert cb["value"] > 0 and "scaled to the whole workload" in cb["sample"]


@pytest.mark.parametrize("kernel,t,kv", [("absorb", 1, 0), ("decompress", 2, 0), ("attn", 1, 2048)])
def test_cpu_baseline_mla(oracle, kernel, t, kv):
    cb = bench.cpu_baseline_mla(kernel, t, kv, 0.05)
    assert cb["kind"] == "oracle" and cb["unit"] == "us" and cb["value"] > 0
    assert "of 64 heads" in cb["sample"]


def test_cpu_baseline_arms_legs(oracle):
    """The default workload's CPU baseline on a small shape: a single-threaded leg and an
    all-cores leg (rows split over the affinity mask), each GB/s of the three-arm step."""
    from types import SimpleNamespace
    arms = {k: SimpleNamespace(out_f=256, in_f=512, gemv_bytes=bench.gemv_bytes(k, 256, 512, 1))
            for k in bench.ARMS}
    cb = bench.cpu_baseline_arms(arms, 0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    cores = [leg["cores"] for leg in cb["legs"]]
    assert cores[0] == 1 and cores[-1] == bench.affinity_cores() == cb["cores"]
    assert all(leg["value"] > 0 and set(leg["arms"]) == set(bench.ARMS) for leg in cb["legs"])
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]


def test_default_workload_is_the_three_arm_target():
    assert bench.DEFAULT_WORKLOAD == "c3"
    assert (bench.C3_OUT_F, bench.C3_IN_F) == (17408, 5120)
    assert bench.ARMS == ("e4m3", "blk", "q8_0")
