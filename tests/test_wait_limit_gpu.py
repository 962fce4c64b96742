"""Bounded waits that run out, on the GPU, without a fault.

Every wait inside the kernels (a K/V copy landing, an MMA completing, a
buffer coming free) gives up after a limit, sets bit 0 of the device fault
word and lets every warp role leave its loop, so a copy that never lands
cannot hang the GPU.  These tests make one happen on purpose through the
library's test controls: a short wait limit (10^6 SM cycles, about 0.5 ms)
and a K/V fill whose copies the first CTA's producer never issues.  Each
checks that the call returns, that swa_read_device_errors() reports bit 0,
that the CUDA context still works, and that the next normal call matches
the fp64 oracle.  Nothing here traps, faults or spins without a limit.
"""
import pytest
import torch

import sliding_window_speculative_gb300 as swa
from sliding_window_speculative_gb300 import inputs
from sliding_window_speculative_gb300._binding import KERNEL_IDS
from tests.helpers import compare, oracle_reference, run_gpu

pytestmark = pytest.mark.gpu

LIMIT = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield
    swa.swa_set_debug_options()


def _many():
    # 200 sequences x 2 KV heads = 400 work items: several per CTA, so the
    # tensor-core producer runs on one lane and the roles cross item borders
    return inputs.make_case("many", 200, 8, 2, 256, 8, 188, [300] * 200, 512, seed=4,
                            device="cuda")


@pytest.mark.parametrize("kernel,name,fill,splits", [
    ("simt", "tiny_q8", 0, 0),                # the only tile of the only CTA
    ("simt", "window_vs_full_w4096", 1, 0),   # second tile of chunk 0 (then the merge)
    ("tc", "single_stream", 1, 0),            # V of the first tile
    ("tc", "single_stream", 2, 0),            # K of the second tile
    ("tc", "many", 5, 0),                     # mid-item, several items per CTA
    ("tc", "single_stream", 0, 3),            # K of the first tile of a split plan
    ("rows", "single_stream", 0, 0),          # rows-major kernel, first K tile
    ("rows", "single_stream", 3, 0),          # rows-major kernel, last V tile
    ("pairs", "single_stream", 0, 0),         # CTA pairs: rank 0's half of the first K tile
    ("pairs", "single_stream", 3, 0),         # rank 0's half of the last V tile (rank 1 zeroes its own)
    ("pairs", "many", 5, 0),                  # mid-item, several items per pair
])
def test_withheld_copy_runs_out_and_reports(kernel, name, fill, splits):
    case = {"tiny_q8": lambda: inputs.tiny(8, device="cuda"),
            "window_vs_full_w4096": lambda: inputs.window_vs_full(4096, device="cuda"),
            "single_stream": lambda: inputs.single_stream(device="cuda"),
            "many": _many}[name]()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert swa.swa_read_device_errors() == 0
    swa.swa_set_debug_options(force_kernel=kernel)
    try:
        plan = swa.swa_plan(swa.dims_of(case.q, case.k_cache, splits), case.window, sms)
        assert plan["kernel"] == KERNEL_IDS[kernel], plan
        # the plan's own result first (it also grows any workspace outside the test)
        ref_o, ref_l = oracle_reference(case)
        out, lse = run_gpu(case, splits)
        compare(out, lse, ref_o, ref_l, f"{name} {kernel} before")
        swa.swa_set_debug_options(force_kernel=kernel, wait_limit_cycles=LIMIT,
                                  withhold_fill=fill)
        swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                            case.window, case.scale, num_splits=splits)
        torch.cuda.synchronize()                     # the call ended: nothing hung
        flags = swa.swa_read_device_errors()
        assert flags & 1, f"{name} {kernel}: no bounded wait reported running out"
        swa.swa_set_debug_options(force_kernel=kernel)
        # the context still works
        x = torch.arange(4096, device="cuda", dtype=torch.float32)
        assert float((x * 2).sum()) == 4095 * 4096
        # and the next normal call is right
        out, lse = run_gpu(case, splits)
        compare(out, lse, ref_o, ref_l, f"{name} {kernel} after")
        assert swa.swa_read_device_errors() == 0
    finally:
        swa.swa_set_debug_options()
