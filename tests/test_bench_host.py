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
                        lambda case, steps, warmup: {"us_per_call": 10.0, "replicas": 3,
                                                     "l2_scheme": "x"})
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


@pytest.mark.parametrize("steps", [1, 20, 300, 1000, 20000])
@pytest.mark.parametrize("name", ["tiny_q1", "tiny_q8", "single_stream", "batched"])
def test_replicas_keep_timed_calls_out_of_l2(name, steps):
    """Whatever the step count: either every timed call reads its own
    replica (and L2 is flushed before the timed replay), or one cycle
    through the replicas reads at least twice L2; the replicas fit in
    16 GiB."""
    case = bench.make_workload(name, "cpu")
    _, total = bench.workload_bytes(case)
    l2 = 126 << 20
    n, _, distinct = bench.replica_count(case, total, steps, l2=l2)
    slab = case.k_cache.numel() * 4 + case.q.numel() * 4
    assert n * slab <= 16 << 30
    if distinct:
        assert n >= steps
    else:
        assert n * total >= 2 * l2


def test_replicas_not_needed_above_l2():
    case = bench.make_workload("tiny_q8", "cpu")
    assert bench.replica_count(case, 200 << 20, 20, l2=126 << 20) == (1, 126 << 20, False)


def test_cpu_baseline_reports_threads_and_host_cores():
    import os
    case = bench.make_workload("tiny_q8", "cpu")
    cb = bench.cpu_baseline(case, 0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["host_cores"] == (os.cpu_count() or 1)
    # tiny: one sequence of 2 query heads -> at most 2 threads have work
    assert cb["threads_used"] == cb["cores"] == min(2, os.cpu_count() or 1)
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
