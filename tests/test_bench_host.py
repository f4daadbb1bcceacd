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
        assert kind in ("gemm1", "gemm2", "pffn", "moe_gemm1", "moe_gemm2")
        assert nbytes > 0 and len(digest) == 64


def test_warmup_below_three_is_rejected():
    import pytest
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peak_choice_follows_the_timed_region():
    peaks = {"bf16_tflops": 1929.6, "bf16_tflops_sustained": 1740.4}
    # a short burst at the maximum clock: the burst peak
    p, why = bench.pick_tensor_peak(peaks, "measured", 0.12, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert p == 1929.6 and "burst" in why
    # seconds under the power cap, clock well below its maximum: the sustained peak
    p, why = bench.pick_tensor_peak(peaks, "measured", 6.0, {"sm_mhz": 1477.0, "sm_max_mhz": 2070.0})
    assert p == 1740.4 and "sustained" in why
    # a long region that still ran at the maximum clock: burst
    p, _ = bench.pick_tensor_peak(peaks, "measured", 6.0, {"sm_mhz": 2065.0, "sm_max_mhz": 2070.0})
    assert p == 1929.6
    # no clock record and a long region: sustained
    p, _ = bench.pick_tensor_peak(peaks, "fallback", 6.0, {"sm_mhz": None, "sm_max_mhz": None})
    assert p == 1740.4


def test_gpus_flag_must_match_the_launcher_world(monkeypatch):
    import pytest
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "4"])


def test_gpus_two_launches_two_ranks_end_to_end():
    """bench.py --gpus 2 run bare starts two ranks itself (torch.distributed.run, on
    127.0.0.1); the reference arm runs on rank 0 alone, which prints the one JSON line
    with n_gpus = 2, and rank 1 exits 0 without work."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "2"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--config", "rankmixer_100m", "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.2"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
