"""bench.py's host logic, without a GPU."""
import json
import os

import numpy as np
import pytest

import bench


@pytest.mark.parametrize("esize,variant,expect", [
    (4, 0, {"fill_store": 1, "drain_load": 1}),
    (4, 1, {"fill_store": 4, "drain_load": 8}),
    (4, 2, {"fill_store": 1, "drain_load": 1}),
    (8, 0, {"fill_store": 1, "drain_load": 1}),
    (8, 1, {"fill_store": 2, "drain_load": 8}),
    (8, 2, {"fill_store": 1, "drain_load": 1}),
    (2, 0, {"fill_store": 1, "drain_ldmatrix": 1}),
    (2, 1, {"fill_store": 1, "drain_ldmatrix": 8}),
    (2, 2, {"fill_store": 1, "drain_ldmatrix": 1}),
    (2, 3, {"fill_store": 1, "drain_ldmatrix": 1}),
])
def test_staging_patterns_bank_predictions(orc, esize, variant, expect):
    """The warp accesses the bench feeds to the GPU profiler get, from the
    oracle's bank model, the predictions the transpose stagings are built for."""
    got = {}
    for access, (addrs, width) in bench.staging_patterns(esize, variant).items():
        ways, _ = orc.bank_profile(np.array([addrs], dtype=np.uint32), width)
        got[access] = int(ways[0])
    assert got == expect


def test_throughput_and_traffic_record(tmp_path, monkeypatch):
    assert bench.throughput(2, 1 << 30, 10, 1000.0) == pytest.approx(2 * (1 << 30) * 10 / 1.0 / 1e9)
    key = bench.HEADLINE_KERNEL
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f).get(key)
    current = bench.source_hash("swz_relayout.cu", "swz_common.cuh")
    got = bench.committed_traffic(key, current)
    # the committed record is used only while it matches the kernel source
    if rec is None:
        assert got is None
    else:
        assert (got == rec["dram_bytes_per_launch"]) == (rec["source_hash"] == current)
    assert bench.committed_traffic(key, "0" * 16) is None
    assert bench.committed_traffic("no such kernel", current) is None


def test_clock_sampler_keeps_only_the_timed_region():
    """Samples outside [t0, t1] are dropped; reasons are the union over the
    region; no sampler at all reports itself as unavailable."""
    cs = bench.ClockSampler(None)
    assert cs.stop(0.0, 1.0)["reasons"] == ["clock sampling unavailable"]

    class Done:
        def join(self, timeout=None):
            pass
    cs = bench.ClockSampler(None)
    cs.thread, cs.source = Done(), "test"
    cs.rows = [(0.5, 900.0, 2070.0, 100.0, {"hw_slowdown"}),      # before the region
               (1.0, 2070.0, 2070.0, 600.0, set()),
               (1.5, 2055.0, 2070.0, 900.0, {"sw_power_cap"}),
               (2.0, 2070.0, 2070.0, 700.0, set()),
               (2.5, 800.0, 2070.0, 100.0, {"sw_thermal_slowdown"})]  # after it
    got = cs.stop(1.0, 2.0)
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]
    assert got["power_w_max"] == 900.0


def test_clock_sampler_reason_bits():
    """NVML's clock-event reason bits map onto the names the JSON line uses."""
    bits = bench.ClockSampler.REASON_BITS
    assert bits[0x4] == "sw_power_cap" and bits[0x8] == "hw_slowdown"
    assert bits[0x20] == "sw_thermal_slowdown" and bits[0x40] == "hw_thermal_slowdown"
    assert 0x1 not in bits  # idle is not a slowdown


def test_cpu_baseline_single_and_all_cores():
    """The CPU baseline runs the oracle single-threaded and over every core
    (spawned workers on shared memory) on (a prefix of) the headline
    workload, and the 125-set sweep on a small sample; all report positive
    rates."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(256 * bench.ROWS * bench.COLS, seed=4)
    res = bench.cpu_baseline(host, seconds=0.01, seconds_all=0.01, sweep_el=1 << 16, sample_scale=64,
                             sample_tiles=16)
    assert res["kind"] == "oracle" and res["cores"] == 1 and res["value"] > 0
    assert res["all_cores"]["cores"] == len(os.sched_getaffinity(0)) and res["all_cores"]["value"] > 0
    sw = res["sweep125_uint16"]
    assert sw["all_cores_GB/s"] > 0 and set(sw["single_thread_GB/s"]) == {"1,4,7", "3,3,3", "5,2,5"}
    assert isinstance(res["cpu_model"], str) and res["cpu_model"]
    assert set(res["other_rows"]) == {
        "relayout_fp16_64x64_sw333_2MiB", "relayout_bf16_4096x128x64_sw343_64MiB", "transpose_fp32_8192",
        "transpose_fp16_16384", "transpose_fp64_8192"}
    assert all(v["single_thread_GB/s"] > 0 and v["all_cores_GB/s"] > 0 for v in res["other_rows"].values())


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    """A comment edit keeps a committed ncu record valid; a code edit does not."""
    csrc = tmp_path / "xor_swizzle_movement_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f.write_text("// header\n__global__ void k(int *p) {\n    p[0] = 1;  /* store */\n}\n")
    h0 = bench.source_hash("k.cu")
    f.write_text("// another header\n/* a block\n comment */\n__global__ void k(int *p) {\n    p[0] = 1;\n}\n")
    assert bench.source_hash("k.cu") == h0
    f.write_text("__global__ void k(int *p) {\n    p[0] = 2;\n}\n")
    assert bench.source_hash("k.cu") != h0


def test_relaunch_command_runs_one_rank_per_gpu():
    """--gpus N without torchrun becomes a torch.distributed.run command on
    one node with N processes, on the loopback address, with the same
    arguments."""
    cmd = bench.relaunch_command(["--gpus", "4", "--steps", "7"], 4, 29555)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nnodes=1" in cmd and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29555"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "7"] and cmd[-5].endswith("bench.py")
