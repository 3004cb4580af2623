"""bench.py's host-side bookkeeping on CPU: which recorded DRAM-traffic figure a bench
line may carry.  A figure belongs to one workload, partition size and set of kernel
sources; anything else (a changed field of the workload, another partition size)
must come out as no figure rather than a borrowed one."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_overridden_workload_carries_its_changes_in_its_name():
    base = workloads.make_workload(1)
    assert "[with" not in base.name
    same = workloads.make_workload(1, head_dim=64)  # workload 1 already has head_dim 64
    assert same.name == base.name
    changed = workloads.make_workload(1, block_size=8, head_dim=128)
    assert changed.name == base.name + " [with block_size=8, head_dim=128]"
    assert changed.block_size == 8 and changed.head_dim == 128


def test_recorded_traffic_matches_only_its_own_workload_and_partition():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)["entries"]
    e = next(x for x in entries if x["path"] == "tensor_core")
    got = bench.recorded_traffic("tensor_core", e["workload"], e["partition_tokens"])
    # a stale entry (sources edited since the capture) gives None; a current one its bytes
    assert got in (None, e["dram_bytes_per_launch"])
    assert bench.recorded_traffic("tensor_core", e["workload"], e["partition_tokens"] + 128) is None
    assert bench.recorded_traffic("tensor_core", e["workload"] + " [with block_size=64]",
                                  e["partition_tokens"]) is None
    assert bench.recorded_traffic("cuda_core", e["workload"], e["partition_tokens"]) is None


def test_f32_tensor_core_decode_is_looked_up_under_its_own_sources():
    import torch
    assert bench.traffic_path(2, torch.float32) == "tensor_core_f32"
    assert bench.traffic_path(2, torch.bfloat16) == "tensor_core"
    assert bench.traffic_path(1, torch.float32) == "cuda_core"
    assert "decode_tc32.cu" in bench.KERNEL_SOURCES["tensor_core_f32"]
