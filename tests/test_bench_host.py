"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_is_reported_only_while_the_kernel_sources_are_unchanged(monkeypatch):
    digest = bench.kernel_source_digest()
    assert len(digest) == 64
    key = ("rankmixer_1b", 4096, 2, "gemm1")
    monkeypatch.setattr(bench, "TRAFFIC", {key: (2.5e9, digest)})
    assert bench.captured_traffic(*key) == 2.5e9
    assert bench.captured_traffic("rankmixer_1b", 2048, 2, "gemm1") is None      # another workload
    monkeypatch.setattr(bench, "TRAFFIC", {key: (2.5e9, "0" * 64)})              # sources changed since
    assert bench.captured_traffic(*key) is None


def test_recorded_traffic_entries_are_well_formed():
    for (config, batch, layers, kind), (nbytes, digest) in bench.TRAFFIC.items():
        assert config in ("rankmixer_1b", "rankmixer_100m", "moe_1b") and batch > 0 and layers > 0
        assert kind in ("gemm1", "gemm2", "moe_gemm1", "moe_gemm2")
        assert nbytes > 0 and len(digest) == 64


def test_warmup_below_three_is_rejected():
    import pytest
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
