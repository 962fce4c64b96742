"""The allocation-free entry point swa_verify_attn_noalloc.

It exists for callers that may not allocate device memory while they serve
(an engine whose memory pool already holds the GPU, a plugin that is only
handed pointers, a path that cannot pay for cudaMalloc's synchronisation):
its split partials go to a fixed device array instead of a cudaMalloc'd
workspace.  These tests call it through the C ABI, on two calls in a row
(the second call finds the first call's data in the shared scratch), and
check that it returns exactly the bits of the allocating entry point
swa_verify_attn at the same plan, and that both meet the parity bar
against the fp64 oracle.  This file is collected last on purpose.
"""
import pytest
import torch

from sliding_window_speculative_gb300 import inputs
from tests.helpers import compare, oracle_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_speculative_gb300 import build
    build.build()
    yield


@pytest.mark.parametrize("name,splits", [("full_decode", 0), ("single_stream", 4),
                                         ("tiny_q8", 3), ("batched", 2)])
def test_noalloc_matches_allocating_entry_point(name, splits):
    import sliding_window_speculative_gb300 as swa
    case = {"full_decode": lambda: inputs.window_vs_full(4096, device="cuda"),
            "single_stream": lambda: inputs.single_stream(device="cuda"),
            "tiny_q8": lambda: inputs.tiny(8, device="cuda"),
            "batched": lambda: inputs.batched(device="cuda")}[name]()
    plan = swa.swa_plan(swa.dims_of(case.q, case.k_cache, splits), case.window,
                        torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["num_splits"] > 1  # the case really uses the scratch
    ref_out, ref_lse = swa.swa_verify_attn(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                           case.q_pos, case.window, case.scale,
                                           num_splits=splits)
    torch.cuda.synchronize()
    ora_out, ora_lse = oracle_reference(case)
    compare(ref_out, ref_lse, ora_out, ora_lse, f"{name} splits={splits}, allocating call")
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        swa.swa_verify_attn_noalloc(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                    case.q_pos, case.window, case.scale, out, lse,
                                    num_splits=splits)
        torch.cuda.synchronize()
        # the same plan and the same kernels: the same bits
        assert torch.equal(out, ref_out), f"{name} splits={splits} call {call}"
        assert torch.equal(lse, ref_lse), f"{name} splits={splits} call {call}"
        compare(out, lse, ora_out, ora_lse, f"{name} splits={splits} call {call}")


def test_noalloc_rejects_plans_above_the_fixed_scratch():
    import sliding_window_speculative_gb300 as swa
    case = inputs.make_case("big", 64, 8, 2, 256, 8, 188, [200] * 64, 256, device="cuda")
    dims = swa.dims_of(case.q, case.k_cache, 64)
    plan = swa.swa_plan(dims, case.window, 152)
    assert plan["workspace_bytes"] > 16 << 20
    out = torch.empty_like(case.q)
    with pytest.raises(swa.SwaError) as e:
        swa.swa_verify_attn_noalloc(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                    case.q_pos, case.window, case.scale, out, num_splits=64)
    assert e.value.status == swa.SWA_ERR_WORKSPACE
    assert str(16 << 20) in str(e.value)
    # one split needs no scratch at all
    swa.swa_verify_attn_noalloc(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                                case.window, case.scale, out, num_splits=1)
    torch.cuda.synchronize()


def test_noalloc_takes_no_device_memory():
    import sliding_window_speculative_gb300 as swa
    case = inputs.single_stream(device="cuda")
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
    # set-up call (resolves the scratch address once per device)
    swa.swa_verify_attn_noalloc(case.q, case.k_cache, case.v_cache, case.seq_lens, case.q_pos,
                                case.window, case.scale, out, lse, num_splits=6)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for splits in (0, 6, 11):
        swa.swa_verify_attn_noalloc(case.q, case.k_cache, case.v_cache, case.seq_lens,
                                    case.q_pos, case.window, case.scale, out, lse,
                                    num_splits=splits)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
