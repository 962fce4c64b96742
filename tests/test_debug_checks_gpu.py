"""The library built with SWA_DEBUG_CHECKS (libswa_debug.so) on the GPU.

Runs tests/debug_checks_run.py in a child process (the binding loads one
library per process): on valid inputs, for every attention kernel, plain,
split, paged and fused-append calls count no out-of-range index attempt
and match the oracle; a sequence length past the cache and a block-table
page outside the pool are counted, the other sequences still match the
oracle, and neither a read nor a store reaches memory past the pool.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def results():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build(debug_checks=True)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_checks_run.py")],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert r.returncode == 0, r.stderr[-3000:]
    return {x["name"]: x for x in lines}


KERNELS = ("simt", "tc", "rows")
# the CTA-pair kernel reads contiguous caches only
VALID = [f"{k}/valid contiguous" for k in KERNELS + ("pairs",)] + \
        [f"{k}/valid paged" for k in KERNELS] + [f"{k}/valid fused append" for k in ("simt", "tc")]
INVALID = [f"{k}/seq_len past the cache" for k in KERNELS + ("pairs",)] + \
          [f"{k}/page outside the pool" for k in KERNELS] + \
          [f"{k}/fused append into a page outside the pool" for k in ("simt", "tc")]


@pytest.mark.parametrize("name", VALID)
def test_valid_inputs_count_nothing(results, name):
    r = results[name]
    assert r["ok"], r["detail"]
    assert r["count"] == 0, r


@pytest.mark.parametrize("name", INVALID)
def test_out_of_range_inputs_are_counted_and_contained(results, name):
    r = results[name]
    assert r["ok"], r["detail"]
    assert r["count"] > 0, r
