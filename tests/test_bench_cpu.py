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
def test_staging_patterns_bank_verdicts(orc, esize, variant, expect):
    """The warp accesses the bench feeds to the GPU profiler get, from the
    oracle's bank model, the verdicts the transpose stagings are built for."""
    got = {}
    for access, (addrs, width) in bench.staging_patterns(esize, variant).items():
        ways, _ = orc.bank_profile(np.array([addrs], dtype=np.uint32), width)
        got[access] = int(ways[0])
    assert got == expect


def test_throughput_and_traffic_record(tmp_path, monkeypatch):
    assert bench.throughput(2, 1 << 30, 10, 1000.0) == pytest.approx(2 * (1 << 30) * 10 / 1.0 / 1e9)
    key = "relayout_vec_kernel<2,0,false> 4096x128x64 bf16 Sw<3,4,3>"
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)[key]
    current = bench.source_hash("swz_relayout.cu", "swz_common.cuh")
    got = bench.committed_traffic(key, current)
    # the committed record is used only while it matches the kernel source
    assert (got == rec["dram_bytes_per_launch"]) == (rec["source_hash"] == current)
    assert bench.committed_traffic(key, "0" * 16) is None
    assert bench.committed_traffic("no such kernel", current) is None
