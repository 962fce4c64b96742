"""bench.py's host-side arithmetic on the CPU (no timing): the algorithmic
bytes and flops of a workload against hand counts, and one extra-workload
entry built from a fixed device time."""
import pytest

import bench


def test_workload_bytes_single_stream():
    case = bench.make_workload("single_stream", "cpu")
    kv, total = bench.workload_bytes(case)
    # 195 keys (4096 - 188 + 1 - 8 ... 4095) x 2 KV heads x K and V x 256 dims x 2 B
    assert kv == 195 * 2 * 2 * 256 * 2 == 399_360
    # + q and out (8 rows x 8 heads x 256 dims x 2 B each) + lse (8 x 8 x 4 B)
    assert total == kv + 2 * 8 * 8 * 256 * 2 + 8 * 8 * 4 == 465_152


def test_workload_flops_tiny():
    case = bench.make_workload("tiny_q8", "cpu")
    # rows at p = 32..39, W = 16, 40 keys: each row sees 16 keys; 2 query
    # heads; 4 * head_dim flops per (row, key, head)
    assert bench.workload_flops(case) == 8 * 16 * 2 * 4 * 64


def test_extra_entry_from_a_fixed_time(monkeypatch):
    from sliding_window_speculative_gb300 import build
    build.build()
    monkeypatch.setattr(bench, "time_device",
                        lambda case, steps, warmup: {"us_per_call": 10.0, "replicas": 3})
    e = bench.extra_entry("single_stream", "cpu", peak=6660.0, tpeak=1884.6, sms=152)
    assert e["us_per_call"] == 10.0 and e["replicas"] == 3
    assert e["kv_gbs"] == pytest.approx(399_360 / 10e-6 / 1e9, abs=0.01)
    assert e["achieved_gbs"] == pytest.approx(465_152 / 10e-6 / 1e9, abs=0.01)
    assert e["frac"] == pytest.approx(465_152 / 10e-6 / 1e9 / 6660.0, abs=1e-4)
    assert e["frac_nominal"] == pytest.approx(465_152 / 10e-6 / 1e9 / 7900.0, abs=1e-4)
    flops = 8 * 8 * 188 * 4 * 256      # 8 rows x 8 heads, every row sees 188 keys
    assert e["useful_tflops"] == pytest.approx(flops / 10e-6 / 1e12, abs=1e-3)
    assert e["tokens_per_s"] == 800_000
    assert e["kernel"] == "swa_tc_kernel" and e["splits"] == 1


def test_ncu_traffic_only_for_the_captured_sources(monkeypatch):
    import json
    import os
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    monkeypatch.setattr(bench, "source_digest", lambda: d["source_sha"])
    n, kernel = bench.ncu_traffic("single_stream")
    assert n == d["workloads"]["single_stream"]["dram_bytes_per_launch"]
    assert kernel == "swa_tc_kernel"
    assert bench.ncu_traffic("no_such_workload") == (None, None)
    # once the kernel sources change, the capture no longer applies
    monkeypatch.setattr(bench, "source_digest", lambda: "0" * 16)
    assert bench.ncu_traffic("single_stream") == (None, "stale")


def test_source_digest_covers_the_kernel_sources(tmp_path, monkeypatch):
    import os
    import shutil
    pkg = tmp_path / "sliding_window_speculative_gb300"
    shutil.copytree(os.path.join(bench.ROOT, "sliding_window_speculative_gb300", "csrc"),
                    pkg / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.source_digest()
    with open(pkg / "csrc" / "swa_tc.cuh", "a") as f:
        f.write("\n")
    assert bench.source_digest() != before
