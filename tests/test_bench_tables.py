"""The bench's stored counter tables (DRAM traffic and global-store bytes of
one fused launch per workload, from ncu) on CPU: each entry is keyed to the
source hash of its kernel family, one hash per family, and the workloads that
--rows sizes carry the size their counters were taken at, so that no other
size is ever reported with them."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

B2B = {"mlp_b2b", "mlp_bottom", "attention_softmax", "attention_relu", "target_attention", "attention_long_keys"}
SIZED = {"mlp_bottom", "target_attention"}


@pytest.mark.parametrize("table", [bench.NCU_TRAFFIC, bench.NCU_STORES])
def test_one_source_hash_per_kernel_family(table):
    hashes = {}
    for name, entry in table.items():
        hashes.setdefault(name in B2B, set()).add(entry["src"])
    assert all(len(h) == 1 for h in hashes.values()), hashes


@pytest.mark.parametrize("table", [bench.NCU_TRAFFIC, bench.NCU_STORES])
def test_sized_workloads_name_their_size(table):
    for name, entry in table.items():
        if name in SIZED:
            assert isinstance(entry.get("rows"), int) and entry["rows"] > 0, name
        else:
            assert "rows" not in entry, name


def test_counters_hold_only_at_the_captured_size():
    for name in SIZED:
        entry = bench.NCU_TRAFFIC[name]
        at = bench.Workload(name, rows=entry["rows"])
        other = bench.Workload(name, rows=max(1, entry["rows"] // 8))
        assert at.size_rows == entry["rows"]
        assert other.size_rows != entry["rows"]
    assert bench.Workload("layernorm_256").size_rows is None
